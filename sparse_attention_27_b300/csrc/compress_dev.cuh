// Softmax pooling of one compressed block, as device functions shared by the
// stand-alone compressor (compress.cu) and the fused decode kernel
// (decode_fused.cu), so that both write bit-identical cache rows.
//
// Source: "오픈소스 LLM의 새 이정표: DeepSeek-V4 시리즈", section
// "압축 희소 어텐션(CSA)과 극압축 어텐션(HCA)" (m consecutive KV entries merged
// into one) and "DeepSeek-V4 논문 읽기: 백만 토큰 컨텍스트를 저렴하게", section
// "Compressed Sparse Attention (CSA)" step 1.  The pooling rule (softmax over
// one logit per raw token) is the reading taken where the pages give none.
//
// The fp32 evaluation order is fixed, whatever the thread layout:
//  * weights: mu = max_i z_i; lane l of one warp sums exp(z_i - mu) over
//    i = l, l+32, ... in order, the 32 lane sums are added by an xor-shuffle
//    tree (distances 16, 8, 4, 2, 1); w_i = exp(z_i - mu) * (1 / sum);
//  * each output channel: RG = min(m, 8) partial sums, partial g over rows
//    i = g, g+RG, ... by fused multiply-adds in increasing i, then
//    ((p_0 + p_1) + p_2) + ... in order; rounded to the storage type.
#pragma once
#include "common.cuh"

namespace sa {

__host__ __device__ constexpr int pool_groups(int m) { return m < 8 ? m : 8; }

// Pooling weights of the block whose first raw position is p0 (ring rows
// (p0 + i) mod R of the logits z_b of one sequence) into w[0..m).  Called by
// all 32 lanes of one warp; w is shared memory; ends with a warp sync (the
// caller synchronises before other warps read w).
__device__ __forceinline__ void pool_weights_warp(const float* z_b, int64_t p0, int m, int R,
                                                  float* w) {
  const int lane = threadIdx.x & 31;
  float mu = -INFINITY;
  // a lane's logits are loaded four at a time (one memory round trip for
  // blocks of up to 128 rows), then kept and maxed in order
  for (int i0 = lane; i0 < m; i0 += 4 * 32) {
    float zi[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + 32 * u;
      zi[u] = i < m ? __ldg(z_b + (p0 + i) % R) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + 32 * u;
      if (i < m) {
        w[i] = zi[u];
        mu = fmaxf(mu, zi[u]);
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mu = fmaxf(mu, __shfl_xor_sync(0xffffffffu, mu, o));
  float sum = 0.f;
  for (int i = lane; i < m; i += 32) sum += expf(w[i] - mu);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  const float inv = 1.f / sum;
  for (int i = lane; i < m; i += 32) w[i] = expf(w[i] - mu) * inv;
  __syncwarp();
}

// 16 bytes of one raw row as floats (8 bf16 or 4 f32 channels).
template <int DT>
__device__ __forceinline__ void load_chunk(const char* p, float* f) {
  const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
  if constexpr (DT == SA_BF16) {
    bf16x8_to_f32(u, f);
  } else {
    f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
  }
}

// Partial g (of RG) of one 16-byte output chunk, rows i = g, g+RG, ... < m,
// with load(i, f) giving row i's chunk as floats.  kBatch rows' loads are
// issued before their multiply-adds (which stay in increasing i), so that
// many memory latencies overlap instead of adding up; the result does not
// depend on it.
template <int kVec, int kBatch, class Load>
__device__ __forceinline__ void pool_partial_by(Load load, int m, const float* w, int g, int RG,
                                                float* acc) {
#pragma unroll
  for (int e = 0; e < kVec; ++e) acc[e] = 0.f;
  for (int i0 = g; i0 < m; i0 += kBatch * RG) {
    float f[kBatch][kVec];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = i0 + u * RG;
      if (i < m) load(i, f[u]);
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = i0 + u * RG;
      if (i < m) {
#pragma unroll
        for (int e = 0; e < kVec; ++e) acc[e] = fmaf(w[i], f[u][e], acc[e]);
      }
    }
  }
}

// pool_partial_by over the raw array `base` in global memory (one sequence,
// rows of `row_bytes`, chunk at byte `off`), block start p0, ring of R rows.
template <int DT, int kBatch = 1>
__device__ __forceinline__ void pool_partial(const char* base, int64_t row_bytes, int off,
                                             int64_t p0, int m, int R, const float* w, int g,
                                             int RG, float* acc) {
  constexpr int kVec = 16 / Store<DT>::kBytes;
  pool_partial_by<kVec, kBatch>(
      [&](int i, float* f) { load_chunk<DT>(base + ((p0 + i) % R) * row_bytes + off, f); }, m, w,
      g, RG, acc);
}

// Store one pooled 16-byte chunk (fp32 values) in the storage type.
template <int DT>
__device__ __forceinline__ void store_chunk(char* out, const float* acc) {
  if constexpr (DT == SA_BF16) {
    uint32_t w4[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      __nv_bfloat162 h = __floats2bfloat162_rn(acc[2 * e], acc[2 * e + 1]);
      w4[e] = *reinterpret_cast<uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(out) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
  } else {
    *reinterpret_cast<float4*>(out) = make_float4(acc[0], acc[1], acc[2], acc[3]);
  }
}

// The whole chunk by one thread: the RG partials in order, added in order.
template <int DT>
__device__ __forceinline__ void pool_chunk(const char* base, int64_t row_bytes, int off,
                                           int64_t p0, int m, int R, const float* w,
                                           float* out) {
  constexpr int kVec = 16 / Store<DT>::kBytes;
  const int RG = pool_groups(m);
  pool_partial<DT>(base, row_bytes, off, p0, m, R, w, 0, RG, out);
  for (int g = 1; g < RG; ++g) {
    float acc[kVec];
    pool_partial<DT>(base, row_bytes, off, p0, m, R, w, g, RG, acc);
#pragma unroll
    for (int e = 0; e < kVec; ++e) out[e] += acc[e];
  }
}

}  // namespace sa
