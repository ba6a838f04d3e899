// Multi-query attention over a compressed-key part plus a sliding window, on
// CUDA cores in fp32 (fp32 inputs; any head count / width), and the exact
// log-sum-exp merges.
//
// Source: "오픈소스 LLM의 새 이정표: DeepSeek-V4 시리즈", section
// "압축 희소 어텐션(CSA)과 극압축 어텐션(HCA)" (CSA: top-k compressed entries plus a
// sliding-window branch; HCA: dense attention over all compressed entries) and
// "DeepSeek-V4 논문 읽기: 백만 토큰 컨텍스트를 저렴하게", sections "Compressed
// Sparse Attention (CSA)" steps 3-4 and "Heavily Compressed Attention (HCA)";
// one shared KV head: "EP 95. DeepSeek-V4 논문 읽기 — 노정석", section IDEAS.
//
// One CTA per (query row, split of the row's key list).  Keys are staged 32 at
// a time in shared memory as fp32; logits for all heads, an online softmax per
// head, and the O update run from shared memory.  With several splits a CTA
// writes a normalised partial (O_s, LSE_s) and the merge kernel combines them.
#include "kernels.cuh"

namespace sa {

constexpr int kAttnSimtThreads = 256;
constexpr int kSubKeys = 32;

template <int DT>
__global__ void __launch_bounds__(kAttnSimtThreads) attend_simt_kernel(AttnArgs a) {
  using S = Store<DT>;
  extern __shared__ float sm[];
  const int H = a.H, d = a.d;
  float* s_q = sm;                         // [H*d]
  float* s_o = s_q + H * d;                // [H*d]
  float* s_k = s_o + H * d;                // [32*d]
  float* s_v = s_k + kSubKeys * d;         // [32*d]
  float* s_p = s_v + kSubKeys * d;         // [H*32]
  float* s_m = s_p + H * kSubKeys;         // [H]
  float* s_l = s_m + H;                    // [H]
  float* s_al = s_l + H;                   // [H]
  int64_t* s_src = reinterpret_cast<int64_t*>(s_al + H + (H & 1));  // [32] source row, -1 masked
  int* s_isw = reinterpret_cast<int*>(s_src + kSubKeys);           // [32] 1: raw window row

  const int64_t row = blockIdx.x / a.nsplit;
  const int split = blockIdx.x % a.nsplit;
  const int b = (int)(row / a.T);
  const int p = __ldg(a.q_pos + row);
  int64_t nvis = p < 0 ? 0 : ((int64_t)p + 1) / a.m;
  if (nvis > a.N_cap) {
    if (split == 0 && threadIdx.x == 0) set_err(a.err, SA_ERR_BOUNDS);
    nvis = a.N_cap;
  }
  const int64_t n_comp = a.gather ? min64(a.k, nvis) : nvis;
  const int64_t n_win = p < 0 ? 0 : min64(a.W, (int64_t)p + 1);
  const int64_t n_keys = n_comp + n_win;
  const int64_t s_begin = (int64_t)split * a.split_tiles * kAttnTile;
  const int64_t s_end = min64(n_keys, s_begin + (int64_t)a.split_tiles * kAttnTile);

  for (int e = threadIdx.x; e < H * d; e += blockDim.x) {
    s_q[e] = S::ld(a.q, row * H * d + e);
    s_o[e] = 0.f;
  }
  for (int h = threadIdx.x; h < H; h += blockDim.x) { s_m[h] = -INFINITY; s_l[h] = 0.f; }
  __syncthreads();

  for (int64_t s0 = s_begin; s0 < s_end; s0 += kSubKeys) {
    if (threadIdx.x < kSubKeys) {
      const int64_t s = s0 + threadIdx.x;
      int64_t src = -1;
      int isw = 0;
      if (s < s_end) {
        if (s < n_comp) {
          int64_t j = a.gather ? (int64_t)__ldg(a.idx + row * a.k + s) : s;
          if (j < -1 || j >= nvis) { set_err(a.err, SA_ERR_BOUNDS); j = -1; }
          src = j < 0 ? -1 : (int64_t)b * a.N_cap + j;
        } else {
          const int64_t u = (int64_t)p - n_win + 1 + (s - n_comp);
          src = (int64_t)b * a.R + u % a.R;
          isw = 1;
        }
      }
      s_src[threadIdx.x] = src;
      s_isw[threadIdx.x] = isw;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < kSubKeys * d; e += blockDim.x) {
      const int i = e / d, c = e % d;
      const int64_t src = s_src[i];
      float kv = 0.f, vv = 0.f;
      if (src >= 0) {
        const void* K = s_isw[i] ? a.kr : a.kc;
        const void* V = s_isw[i] ? a.vr : a.vc;
        kv = S::ld(K, src * d + c);
        vv = S::ld(V, src * d + c);
      }
      s_k[e] = kv;
      s_v[e] = vv;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < H * kSubKeys; e += blockDim.x) {
      const int h = e / kSubKeys, i = e % kSubKeys;
      float lg = -INFINITY;
      if (s_src[i] >= 0) {
        float dot = 0.f;
        for (int c = 0; c < d; ++c) dot = fmaf(s_q[h * d + c], s_k[i * d + c], dot);
        lg = dot * a.sm_scale;
      }
      s_p[e] = lg;
    }
    __syncthreads();
    for (int h = threadIdx.x; h < H; h += blockDim.x) {
      float mx = s_m[h];
      for (int i = 0; i < kSubKeys; ++i) mx = fmaxf(mx, s_p[h * kSubKeys + i]);
      float alpha = 1.f, sum = 0.f;
      if (mx != -INFINITY) {
        alpha = (s_m[h] == -INFINITY) ? 0.f : expf(s_m[h] - mx);
        for (int i = 0; i < kSubKeys; ++i) {
          const float lg = s_p[h * kSubKeys + i];
          const float pv = (lg == -INFINITY) ? 0.f : expf(lg - mx);
          s_p[h * kSubKeys + i] = pv;
          sum += pv;
        }
        s_m[h] = mx;
      } else {
        for (int i = 0; i < kSubKeys; ++i) s_p[h * kSubKeys + i] = 0.f;
      }
      s_l[h] = s_l[h] * alpha + sum;
      s_al[h] = alpha;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < H * d; e += blockDim.x) {
      const int h = e / d, c = e % d;
      float acc = s_o[e] * s_al[h];
      for (int i = 0; i < kSubKeys; ++i) acc = fmaf(s_p[h * kSubKeys + i], s_v[i * d + c], acc);
      s_o[e] = acc;
    }
    __syncthreads();
  }

  float* out_l = a.nsplit > 1 ? a.part_lse + (row * a.nsplit + split) * H : a.lse + row * H;
  for (int e = threadIdx.x; e < H * d; e += blockDim.x) {
    const int h = e / d;
    const float l = s_l[h];
    const float v = l > 0.f ? s_o[e] / l : 0.f;
    if (a.nsplit > 1) a.part_o[(row * a.nsplit + split) * H * d + e] = v;
    else if (a.o_dtype == SA_BF16) Store<SA_BF16>::st(a.o, row * H * d + e, v);
    else Store<SA_F32>::st(a.o, row * H * d + e, v);
  }
  for (int h = threadIdx.x; h < H; h += blockDim.x)
    out_l[h] = s_l[h] > 0.f ? s_m[h] + logf(s_l[h]) : -INFINITY;
}

size_t attend_simt_smem(int H, int d) {
  return sizeof(float) * (2 * (size_t)H * d + 2 * kSubKeys * d + (size_t)H * kSubKeys + 3 * H + 2) +
         (sizeof(int64_t) + sizeof(int)) * kSubKeys + 16;
}

cudaError_t launch_attend_simt(const AttnArgs& a, cudaStream_t st) {
  const int64_t rows = (int64_t)a.B * a.T;
  if (rows == 0) return cudaSuccess;
  const size_t smem = attend_simt_smem(a.H, a.d);
  cudaError_t e;
  if (a.dtype == SA_BF16) {
    e = cudaFuncSetAttribute(attend_simt_kernel<SA_BF16>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attend_simt_kernel<SA_BF16><<<(unsigned)(rows * a.nsplit), kAttnSimtThreads, smem, st>>>(a);
  } else {
    e = cudaFuncSetAttribute(attend_simt_kernel<SA_F32>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attend_simt_kernel<SA_F32><<<(unsigned)(rows * a.nsplit), kAttnSimtThreads, smem, st>>>(a);
  }
  return cudaGetLastError();
}

// ------------------------------------------------------------------ merges
// Exact merge of partials over disjoint key sets:
//   LSE = log sum_i exp(LSE_i),  O = sum_i exp(LSE_i - LSE) * O_i.
// (The multi-branch design of "EP 95. DeepSeek-V4 논문 읽기 — 노정석", IDEAS, and
// the split-K partials of the kernels above.)  One warp per (row, head).

// Partials are laid out [row, split, head, :].  A CTA merges kMergeHeads
// heads of one query row.  All threads first fetch the split LSEs into shared
// memory at once (one memory round trip rather than nsplit dependent loads);
// kMergeHeads threads turn them into weights exp(LSE_s - LSE); then each
// thread issues up to kMergeBatch (16) independent 16-byte partial loads before it
// accumulates them.  Grid: (rows, ceil(H / kMergeHeads)).
constexpr int kMergeThreads = 256;
constexpr int kMergeHeads = 8;
constexpr int kMergeBatch = 16;

__global__ void __launch_bounds__(kMergeThreads) merge_splits_kernel(
    const float* __restrict__ part_o, const float* __restrict__ part_lse, int nsplit, int H,
    int d, void* __restrict__ o, int o_dtype, float* __restrict__ lse) {
  extern __shared__ float s_w[];                 // [nsplit][kMergeHeads]: LSEs, then weights
  const int64_t row = blockIdx.x;
  const int h0 = blockIdx.y * kMergeHeads;
  const int nh = min(kMergeHeads, H - h0);
  const float* pl = part_lse + row * nsplit * H + h0;
  for (int i = threadIdx.x; i < nsplit * kMergeHeads; i += blockDim.x) {
    const int s = i / kMergeHeads, hh = i % kMergeHeads;
    s_w[i] = hh < nh ? __ldg(pl + s * H + hh) : -INFINITY;
  }
  __syncthreads();
  if (threadIdx.x < nh) {
    const int hh = threadIdx.x;
    float mx = -INFINITY;
    for (int s = 0; s < nsplit; ++s) mx = fmaxf(mx, s_w[s * kMergeHeads + hh]);
    float L = -INFINITY;
    if (mx != -INFINITY) {
      float sum = 0.f;
      for (int s = 0; s < nsplit; ++s) sum += expf(s_w[s * kMergeHeads + hh] - mx);
      L = mx + logf(sum);
    }
    for (int s = 0; s < nsplit; ++s) {
      const float l = s_w[s * kMergeHeads + hh];
      s_w[s * kMergeHeads + hh] = L == -INFINITY ? 0.f : expf(l - L);
    }
    lse[row * H + h0 + hh] = L;
  }
  __syncthreads();
  const int d4 = d / 4;
  const int n4 = nh * d4;                        // float4 outputs of this CTA
  const int64_t stride4 = (int64_t)H * d4;       // float4 per split of the row
  const float4* po = reinterpret_cast<const float4*>(part_o + (row * nsplit * H + h0) * d);
  const int64_t out0 = (row * H + h0) * d;      // first output element of this CTA
  for (int e = threadIdx.x; e < n4; e += blockDim.x) {
    const int hh = e / d4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < nsplit; s0 += kMergeBatch) {
      float4 v[kMergeBatch];
#pragma unroll
      for (int j = 0; j < kMergeBatch; ++j)
        if (s0 + j < nsplit) v[j] = __ldg(po + (s0 + j) * stride4 + e);
#pragma unroll
      for (int j = 0; j < kMergeBatch; ++j) {
        if (s0 + j < nsplit) {
          const float wgt = s_w[(s0 + j) * kMergeHeads + hh];
          acc.x = fmaf(wgt, v[j].x, acc.x);
          acc.y = fmaf(wgt, v[j].y, acc.y);
          acc.z = fmaf(wgt, v[j].z, acc.z);
          acc.w = fmaf(wgt, v[j].w, acc.w);
        }
      }
    }
    if (o_dtype == SA_BF16) {
      const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
      const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
      uint2 u;
      u.x = *reinterpret_cast<const uint32_t*>(&lo);
      u.y = *reinterpret_cast<const uint32_t*>(&hi);
      reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(o) + out0)[e] = u;
    } else {
      reinterpret_cast<float4*>(static_cast<float*>(o) + out0)[e] = acc;
    }
  }
}

__global__ void merge_parts_kernel(MergeArgs a) {
  const int64_t g = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (g >= a.rows) return;
  const int lane = threadIdx.x & 31;
  float mx = -INFINITY;
  for (int s = 0; s < a.n; ++s) mx = fmaxf(mx, a.lse_parts[s][g]);
  float L = -INFINITY;
  if (mx != -INFINITY) {
    float sum = 0.f;
    for (int s = 0; s < a.n; ++s) sum += expf(a.lse_parts[s][g] - mx);
    L = mx + logf(sum);
  }
  for (int c = lane; c < a.d; c += 32) {
    float acc = 0.f;
    if (mx != -INFINITY) {
      for (int s = 0; s < a.n; ++s) {
        const float wgt = expf(a.lse_parts[s][g] - L);
        if (wgt > 0.f) acc = fmaf(wgt, a.o_parts[s][g * a.d + c], acc);
      }
    }
    if (a.o_dtype == SA_BF16)
      Store<SA_BF16>::st(a.o, g * a.d + c, acc);
    else
      Store<SA_F32>::st(a.o, g * a.d + c, acc);
  }
  if (lane == 0) a.lse[g] = L;
}

cudaError_t launch_merge_splits(const AttnArgs& a, cudaStream_t st) {
  if (a.nsplit <= 1) return cudaSuccess;
  const int64_t rows = (int64_t)a.B * a.T;
  if (a.d % 4) return cudaErrorInvalidValue;
  const size_t smem = sizeof(float) * (size_t)a.nsplit * kMergeHeads;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(merge_splits_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  const dim3 grid((unsigned)rows, (unsigned)((a.H + kMergeHeads - 1) / kMergeHeads));
  merge_splits_kernel<<<grid, kMergeThreads, smem, st>>>(a.part_o, a.part_lse, a.nsplit, a.H,
                                                          a.d, a.o, a.o_dtype, a.lse);
  return cudaGetLastError();
}

cudaError_t launch_merge(const MergeArgs& a, cudaStream_t st) {
  if (a.rows <= 0) return cudaSuccess;
  const int threads = 256;
  const int64_t blocks = (a.rows * 32 + threads - 1) / threads;
  merge_parts_kernel<<<(unsigned)blocks, threads, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace sa
