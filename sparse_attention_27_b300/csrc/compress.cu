// Block compression (CSA with m = 4, HCA with m' = 128): softmax pooling of m
// consecutive raw rows into one cache row.
//
// Source: "오픈소스 LLM의 새 이정표: DeepSeek-V4 시리즈", section
// "압축 희소 어텐션(CSA)과 극압축 어텐션(HCA)" (m consecutive KV entries merged
// into one; HCA with m' >> m), and "DeepSeek-V4 논문 읽기: 백만 토큰 컨텍스트를
// 저렴하게", section "Compressed Sparse Attention (CSA)" step 1.  The pooling
// rule (softmax over one logit per raw token) is the reading taken where the
// pages give none.
//
// One CTA per (sequence, block).  One warp turns the block's m logits into
// weights in shared memory.  Each output row is cut into 16-byte chunks (8
// bf16 or 4 f32 channels of K, V or the indexer key); a thread owns one
// chunk and one of RG = min(m, 8) row groups, accumulates in fp32 with
// 16-byte loads, and the row groups are added in shared memory in order --
// the evaluation order compress_dev.cuh fixes, which the fused decode kernel
// follows too.  Memory-bound: each raw byte is read once, each output byte
// written once.
#include "compress_dev.cuh"
#include "kernels.cuh"

namespace sa {

constexpr int kCompressThreads = 256;

// Nearest e2m1 magnitude code for |v| (v already divided by the block
// scale), ties to the even code, saturating at 6 (OCP MX v1.0 FP4 E2M1 grid
// 0, 0.5, 1, 1.5, 2, 3, 4, 6).
__device__ __forceinline__ uint32_t e2m1_code(float av) {
  if (av <= 0.25f) return 0;
  if (av < 0.75f) return 1;
  if (av <= 1.25f) return 2;
  if (av < 1.75f) return 3;
  if (av <= 2.5f) return 4;
  if (av < 3.5f) return 5;
  if (av <= 5.0f) return 6;
  return 7;
}

// Quantise one 32-element block held one element per lane (MXFP4, OCP MX
// v1.0): scale exponent e = floor(log2(amax)) - 2 clamped to [-127, 127]
// (all-zero block: -127); element code = nearest e2m1 of x / 2^e; a negative
// element whose magnitude rounds to zero is stored as +0.  Lane 0 writes the
// scale byte, even lanes write one code byte each (low nibble = even element).
__device__ __forceinline__ void mxfp4_quantize_warp(float x, uint8_t* codes16, uint8_t* scale) {
  const int lane = threadIdx.x & 31;
  float amax = fabsf(x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  int e = (amax > 0.f) ? ilogbf(amax) - 2 : -127;
  e = max(-127, min(127, e));
  float v = ldexpf(x, -e);
  uint32_t mag = e2m1_code(fabsf(v));
  uint32_t nib = (v < 0.f && mag != 0) ? (8u | mag) : mag;
  uint32_t hi = __shfl_down_sync(0xffffffffu, nib, 1);
  if ((lane & 1) == 0) codes16[lane >> 1] = static_cast<uint8_t>(nib | (hi << 4));
  if (lane == 0) *scale = static_cast<uint8_t>(e + 127);
}

template <int DT>
__global__ void __launch_bounds__(kCompressThreads) compress_kernel(CompressArgs a) {
  using S = Store<DT>;
  constexpr int kVec = 16 / S::kBytes;               // channels per 16-byte chunk
  extern __shared__ float s_w[];                     // [m] pooling weights, then partials
  const int b = blockIdx.y;
  const int lo = __ldg(a.blk_lo + b), hi = __ldg(a.blk_hi + b);
  const int64_t j = (int64_t)lo + blockIdx.x;
  if (j >= hi) return;
  if (hi - lo > a.max_blocks || j < 0 || j >= a.N_cap) {
    if (threadIdx.x == 0) set_err(a.err, SA_ERR_BOUNDS);
    return;
  }
  const int m = a.m, R = a.R;
  const int64_t p0 = j * m;
  // ---- work split: item (chunk c, row group g) computes partial g of one
  // 16-byte output chunk (K, V or indexer key); the RG partials of a chunk are
  // then added in order (compress_dev.cuh fixes the arithmetic).
  const int ckv = a.d / kVec;                         // chunks per K or V row
  const bool ik_plain = a.ik_raw != nullptr && a.ik_dtype != SA_MXFP4;
  const int cik = ik_plain ? a.dI / kVec : 0;
  const int nchunks = 2 * ckv + cik;
  const int RG = pool_groups(m);
  const int nitems = RG * nchunks;
  float* s_part = s_w + m;                            // [RG][nchunks][kVec]
  auto chunk_of = [&](int c, const char*& src, char*& dst, int& width, int& off) {
    const void* sp;
    void* dp;
    if (c < ckv) { sp = a.k_raw; dp = a.k_c; width = a.d; off = c * kVec; }
    else if (c < 2 * ckv) { sp = a.v_raw; dp = a.v_c; width = a.d; off = (c - ckv) * kVec; }
    else { sp = a.ik_raw; dp = a.ik_c; width = a.dI; off = (c - 2 * ckv) * kVec; }
    src = static_cast<const char*>(sp) + (int64_t)b * R * width * S::kBytes;
    dst = static_cast<char*>(dp) + ((int64_t)b * a.N_cap + j) * width * S::kBytes;
  };
  // the rows of this thread's items start their trip to memory before the
  // pooling weights are known, so the two round trips overlap
  for (int it = threadIdx.x; it < nitems; it += blockDim.x) {
    const char* src; char* dst; int width, off;
    chunk_of(it % nchunks, src, dst, width, off);
    for (int i = it / nchunks; i < m; i += RG) {
      const char* pr = src + ((p0 + i) % R) * width * S::kBytes + off * S::kBytes;
      asm volatile("prefetch.global.L1 [%0];" ::"l"(pr));
    }
  }
  if (threadIdx.x < 32) pool_weights_warp(a.z + (int64_t)b * R, p0, m, R, s_w);
  __syncthreads();
  for (int it = threadIdx.x; it < nitems; it += blockDim.x) {
    const int c = it % nchunks, g = it / nchunks;
    const char* src; char* dst; int width, off;
    chunk_of(c, src, dst, width, off);
    float acc[kVec];
    pool_partial<DT, 8>(src, (int64_t)width * S::kBytes, off * S::kBytes, p0, m, R, s_w, g, RG,
                          acc);
#pragma unroll
    for (int e = 0; e < kVec; ++e) s_part[(g * nchunks + c) * kVec + e] = acc[e];
  }
  __syncthreads();
  for (int c = threadIdx.x; c < nchunks; c += blockDim.x) {
    const char* src; char* dst; int width, off;
    chunk_of(c, src, dst, width, off);
    float acc[kVec];
#pragma unroll
    for (int e = 0; e < kVec; ++e) acc[e] = s_part[c * kVec + e];
    for (int g = 1; g < RG; ++g)
#pragma unroll
      for (int e = 0; e < kVec; ++e) acc[e] += s_part[(g * nchunks + c) * kVec + e];
    store_chunk<DT>(dst + off * S::kBytes, acc);
  }

  // ---- indexer key stored as MXFP4: one warp per 32-element block
  if (a.ik_raw != nullptr && a.ik_dtype == SA_MXFP4) {
    const int nblk32 = a.dI / 32;
    for (int q = warp_id(); q < nblk32; q += blockDim.x / 32) {
      const int ch = q * 32 + lane_id();
      float acc = 0.f;
      for (int i = 0; i < m; ++i) {
        const int64_t slot = (p0 + i) % R;
        acc = fmaf(s_w[i], Store<SA_BF16>::ld(a.ik_raw, ((int64_t)b * R + slot) * a.dI + ch), acc);
      }
      const float rounded = __bfloat162float(__float2bfloat16_rn(acc));
      uint8_t* codes = static_cast<uint8_t*>(a.ik_c) + ((int64_t)b * a.N_cap + j) * (a.dI / 2) + q * 16;
      uint8_t* sc = static_cast<uint8_t*>(a.ik_c_scales) + ((int64_t)b * a.N_cap + j) * nblk32 + q;
      mxfp4_quantize_warp(rounded, codes, sc);
    }
  }
}

// Stand-alone MXFP4 quantiser for rows of bf16 values (the indexer queries
// and the indexer key cache): one warp per 32-element block.
__global__ void mxfp4_quantize_kernel(const __nv_bfloat16* x, int64_t nblk, uint8_t* codes,
                                      uint8_t* scales) {
  const int64_t blk = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (blk >= nblk) return;
  const float v = __bfloat162float(x[blk * 32 + lane_id()]);
  mxfp4_quantize_warp(v, codes + blk * 16, scales + blk);
}

cudaError_t launch_compress(const CompressArgs& a, cudaStream_t st) {
  if (a.max_blocks <= 0) return cudaSuccess;
  dim3 grid(a.max_blocks, a.B);
  // weights [m] + partial sums [RG][nchunks][16 bytes of floats]
  const int vec = a.dtype == SA_BF16 ? 8 : 4;
  const bool ik_plain = a.ik_raw != nullptr && a.ik_dtype != SA_MXFP4;
  const int nchunks = 2 * a.d / vec + (ik_plain ? a.dI / vec : 0);
  const size_t smem = sizeof(float) * ((size_t)a.m + (size_t)pool_groups(a.m) * nchunks * vec);
  cudaError_t e;
  if (a.dtype == SA_BF16) {
    if (smem > 48 * 1024 &&
        (e = cudaFuncSetAttribute(compress_kernel<SA_BF16>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
            cudaSuccess)
      return e;
    compress_kernel<SA_BF16><<<grid, kCompressThreads, smem, st>>>(a);
  } else {
    if (smem > 48 * 1024 &&
        (e = cudaFuncSetAttribute(compress_kernel<SA_F32>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
            cudaSuccess)
      return e;
    compress_kernel<SA_F32><<<grid, kCompressThreads, smem, st>>>(a);
  }
  return cudaGetLastError();
}

cudaError_t launch_mxfp4_quantize(const void* x_bf16, int64_t nblk, void* codes, void* scales,
                                  cudaStream_t st) {
  if (nblk <= 0) return cudaSuccess;
  const int threads = 256;
  const int64_t blocks = (nblk * 32 + threads - 1) / threads;
  mxfp4_quantize_kernel<<<(unsigned)blocks, threads, 0, st>>>(
      static_cast<const __nv_bfloat16*>(x_bf16), nblk, static_cast<uint8_t*>(codes),
      static_cast<uint8_t*>(scales));
  return cudaGetLastError();
}


// ---------------------------------------------------------------- ring write
// One CTA per (sequence, array): row b of array i into ring row pos[b] mod R,
// 4 bytes per thread and step.
__global__ void ring_write_kernel(RingWriteArgs a) {
  const int b = blockIdx.x, i = blockIdx.y;
  const int p = __ldg(a.pos + b);
  if (p < 0) {
    if (threadIdx.x == 0 && i == 0) set_err(a.err, SA_ERR_BOUNDS);
    return;
  }
  const int words = a.row_bytes[i] / 4;
  const uint32_t* src = static_cast<const uint32_t*>(a.rows[i]) + (int64_t)b * words;
  uint32_t* dst = static_cast<uint32_t*>(a.rings[i]) + ((int64_t)b * a.R + p % a.R) * words;
  for (int w = threadIdx.x; w < words; w += blockDim.x) dst[w] = __ldg(src + w);
}

cudaError_t launch_ring_write(const RingWriteArgs& a, cudaStream_t st) {
  if (a.B == 0) return cudaSuccess;
  ring_write_kernel<<<dim3((unsigned)a.B, (unsigned)a.n), 128, 0, st>>>(a);
  return cudaGetLastError();
}


// ------------------------------------------------ per-channel pooling
// One CTA per (sequence, block); thread c pools channel c (and c + blockDim,
// ...).  fp32 order, per channel: mu = max_i z_i (i ascending); den =
// sum_i exp(z_i - mu) in ascending i; x_c = sum_i (exp(z_i - mu) / den) * x_i
// by fused multiply-adds in ascending i; rounded to the storage type.
template <int DT>
__global__ void compress_channels_kernel(CompressChArgs a) {
  const int b = blockIdx.y;
  const int lo = __ldg(a.blk_lo + b), hi = __ldg(a.blk_hi + b);
  const int64_t j = (int64_t)lo + blockIdx.x;
  if (j >= hi) return;
  if (hi - lo > a.max_blocks || j < 0 || j >= a.N_cap) {
    if (threadIdx.x == 0) set_err(a.err, SA_ERR_BOUNDS);
    return;
  }
  const int m = a.m, R = a.R, d = a.d;
  const int64_t p0 = j * m;
  for (int c = threadIdx.x; c < d; c += blockDim.x) {
    const float* zc = a.z + (int64_t)b * R * d + c;
    auto row = [&](int i) -> int64_t { return ((p0 + i) % R) * d; };
    float mu = -INFINITY;
    for (int i = 0; i < m; ++i) mu = fmaxf(mu, __ldg(zc + row(i)));
    float den = 0.f;
    for (int i = 0; i < m; ++i) den += expf(__ldg(zc + row(i)) - mu);
    float acc = 0.f;
    for (int i = 0; i < m; ++i) {
      const float wi = expf(__ldg(zc + row(i)) - mu) / den;
      acc = fmaf(wi, Store<DT>::ld(a.x_raw, (int64_t)b * R * d + row(i) + c), acc);
    }
    Store<DT>::st(a.x_c, ((int64_t)b * a.N_cap + j) * d + c, acc);
  }
}

cudaError_t launch_compress_channels(const CompressChArgs& a, cudaStream_t st) {
  if (a.B == 0 || a.max_blocks == 0) return cudaSuccess;
  const dim3 grid((unsigned)a.max_blocks, (unsigned)a.B);
  const int threads = a.d < 128 ? ((a.d + 31) / 32) * 32 : 128;
  if (a.dtype == SA_BF16) compress_channels_kernel<SA_BF16><<<grid, threads, 0, st>>>(a);
  else compress_channels_kernel<SA_F32><<<grid, threads, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace sa
