// Backward pass of the attention branches and of the block pooling, on CUDA
// cores in fp32.
//
// Source: "오픈소스 LLM의 새 이정표: DeepSeek-V4 시리즈", section
// "압축 희소 어텐션(CSA)과 극압축 어텐션(HCA)" (what the forward computes), and
// "EP 95. DeepSeek-V4 논문 읽기 — 노정석", section IDEAS: top-k selection is not
// differentiable, so the selection is a constant mask here -- gradients reach
// the queries, the attended cache rows and window rows, and through the
// pooling of the pass's blocks the raw rows and their logits; the indexer
// gets none.  The storage rounding of the caches is taken as the identity.
//
// Attention, per query row (H heads sharing one KV head) and key o of its
// key list, with P = exp(scale * q.k - LSE) from the forward's LSE:
//     dV_o += sum_h P dO_h;   dP = dO_h . V_o;   D_h = dO_h . O_h
//     dS = P (dP - D_h);      dq_h += scale sum_o dS K_o;   dK_o += scale sum_h dS q_h
// One CTA per (row, split of the key list in tiles of 32 keys): q, dO and a
// dq accumulator in shared memory; per tile the K/V rows (fp32), then S, P,
// dS, and the three products; dK/dV are added to the cache and ring rows
// with atomics (rows shared by several queries or splits), dq likewise.
//
// Pooling, per block with weights a = softmax(z_block) and the unrounded
// pooled row Xc = sum_i a_i X_i:
//     dX_i += a_i dXc;   dz_i += a_i (X_i - Xc) . dXc    (K and V both)
// One CTA per (sequence, block); the raw-row and logit gradients are added
// with atomics onto what the attention backward left there.
#include "kernels.cuh"

namespace sa {

namespace {

constexpr int kBwdThreads = 256;
constexpr int kBwdKeys = 32;          // keys per tile

template <int DT>
__global__ void __launch_bounds__(kBwdThreads) attend_backward_kernel(AttnBwdArgs a) {
  using S = Store<DT>;
  const int H = a.H, d = a.d, dp = d + 1;          // padded row stride of K/V tiles
  extern __shared__ float sm[];
  float* s_q = sm;                                 // [H][d]
  float* s_do = s_q + H * d;                       // [H][d]
  float* s_dq = s_do + H * d;                      // [H][d] accumulator
  float* s_k = s_dq + H * d;                       // [32][d+1]
  float* s_v = s_k + kBwdKeys * dp;                // [32][d+1]
  float* s_p = s_v + kBwdKeys * dp;                // [H][32]: P
  float* s_ds = s_p + H * kBwdKeys;                // [H][32]: dS
  float* s_lse = s_ds + H * kBwdKeys;              // [H]
  float* s_D = s_lse + H;                          // [H]
  int64_t* s_src = reinterpret_cast<int64_t*>(s_D + H + (H & 1));   // [32] source row, -1 masked
  int* s_isw = reinterpret_cast<int*>(s_src + kBwdKeys);           // [32] 1: window (ring) row

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
  const int64_t s_begin = (int64_t)split * a.split_tiles * kBwdKeys;
  const int64_t s_end = min64(n_keys, s_begin + (int64_t)a.split_tiles * kBwdKeys);
  if (s_begin >= s_end) return;

  for (int e = threadIdx.x; e < H * d; e += blockDim.x) {
    s_q[e] = S::ld(a.q, row * H * d + e);
    s_do[e] = a.dout[row * H * d + e];
    s_dq[e] = 0.f;
  }
  __syncthreads();
  // D_h = dO_h . O_h (one warp per head), LSE of the forward
  for (int h = threadIdx.x >> 5; h < H; h += blockDim.x >> 5) {
    float acc = 0.f;
    for (int c = threadIdx.x & 31; c < d; c += 32)
      acc = fmaf(s_do[h * d + c], a.o[(row * H + h) * d + c], acc);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if ((threadIdx.x & 31) == 0) {
      s_D[h] = acc;
      s_lse[h] = a.lse[row * H + h];
    }
  }

  for (int64_t s0 = s_begin; s0 < s_end; s0 += kBwdKeys) {
    __syncthreads();
    if (threadIdx.x < kBwdKeys) {
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
    for (int e = threadIdx.x; e < kBwdKeys * d; e += blockDim.x) {
      const int i = e / d, c = e % d;
      const int64_t src = s_src[i];
      float kv = 0.f, vv = 0.f;
      if (src >= 0) {
        kv = S::ld(s_isw[i] ? a.kr : a.kc, src * d + c);
        vv = S::ld(s_isw[i] ? a.vr : a.vc, src * d + c);
      }
      s_k[i * dp + c] = kv;
      s_v[i * dp + c] = vv;
    }
    __syncthreads();
    // P and dS: thread (i, h group) for key i = t % 32
    for (int e = threadIdx.x; e < H * kBwdKeys; e += blockDim.x) {
      const int i = e % kBwdKeys, h = e / kBwdKeys;
      float pr = 0.f, ds = 0.f;
      if (s_src[i] >= 0 && s_lse[h] != -INFINITY) {
        float dot = 0.f, dpv = 0.f;
        for (int c = 0; c < d; ++c) {
          dot = fmaf(s_q[h * d + c], s_k[i * dp + c], dot);
          dpv = fmaf(s_do[h * d + c], s_v[i * dp + c], dpv);
        }
        pr = expf(dot * a.sm_scale - s_lse[h]);
        ds = pr * (dpv - s_D[h]);
      }
      s_p[h * kBwdKeys + i] = pr;
      s_ds[h * kBwdKeys + i] = ds;
    }
    __syncthreads();
    // dq_h += scale * sum_i dS[h][i] K_i
    for (int e = threadIdx.x; e < H * d; e += blockDim.x) {
      const int h = e / d, c = e % d;
      float acc = 0.f;
#pragma unroll 8
      for (int i = 0; i < kBwdKeys; ++i) acc = fmaf(s_ds[h * kBwdKeys + i], s_k[i * dp + c], acc);
      s_dq[e] += a.sm_scale * acc;
    }
    // dK_i = scale * sum_h dS[h][i] q_h;  dV_i = sum_h P[h][i] dO_h
    for (int e = threadIdx.x; e < kBwdKeys * d; e += blockDim.x) {
      const int i = e / d, c = e % d;
      const int64_t src = s_src[i];
      if (src < 0) continue;
      float gk = 0.f, gv = 0.f;
      for (int h = 0; h < H; ++h) {
        gk = fmaf(s_ds[h * kBwdKeys + i], s_q[h * d + c], gk);
        gv = fmaf(s_p[h * kBwdKeys + i], s_do[h * d + c], gv);
      }
      float* dk = s_isw[i] ? a.dkr : a.dkc;
      float* dv = s_isw[i] ? a.dvr : a.dvc;
      atomicAdd(dk + src * d + c, a.sm_scale * gk);
      atomicAdd(dv + src * d + c, gv);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < H * d; e += blockDim.x) atomicAdd(a.dq + row * H * d + e, s_dq[e]);
}

// Pooling backward of block j = blk_lo[b] + blockIdx.x of sequence b = blockIdx.y.
template <int DT>
__global__ void __launch_bounds__(kBwdThreads) compress_backward_kernel(CompressBwdArgs a) {
  using S = Store<DT>;
  extern __shared__ float sw[];                    // [m] weights, [m] logit gradients
  float* s_dz = sw + a.m;
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
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    float mu = -INFINITY;
    for (int i = lane; i < m; i += 32) {
      const float zi = __ldg(a.z + (int64_t)b * R + (p0 + i) % R);
      sw[i] = zi;
      mu = fmaxf(mu, zi);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mu = fmaxf(mu, __shfl_xor_sync(0xffffffffu, mu, o));
    float sum = 0.f;
    for (int i = lane; i < m; i += 32) sum += expf(sw[i] - mu);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    for (int i = lane; i < m; i += 32) sw[i] = expf(sw[i] - mu) / sum;
  }
  for (int i = threadIdx.x; i < m; i += blockDim.x) s_dz[i] = 0.f;
  __syncthreads();
  // channel c of K and of V: the unrounded pooled value, then each raw row's
  // share of the gradient and of the logit gradient
  for (int c = threadIdx.x; c < 2 * d; c += blockDim.x) {
    const bool isv = c >= d;
    const int cc = isv ? c - d : c;
    const void* X = isv ? a.v_raw : a.k_raw;
    const float g = (isv ? a.dvc : a.dkc)[((int64_t)b * a.N_cap + j) * d + cc];
    float* dX = isv ? a.dvr : a.dkr;
    float xc = 0.f;
    for (int i = 0; i < m; ++i) xc = fmaf(sw[i], S::ld(X, ((int64_t)b * R + (p0 + i) % R) * d + cc), xc);
    for (int i = 0; i < m; ++i) {
      const int64_t r = (int64_t)b * R + (p0 + i) % R;
      const float xi = S::ld(X, r * d + cc);
      atomicAdd(dX + r * d + cc, sw[i] * g);
      atomicAdd(&s_dz[i], sw[i] * (xi - xc) * g);
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < m; i += blockDim.x)
    atomicAdd(a.dz + (int64_t)b * R + (p0 + i) % R, s_dz[i]);
}

}  // namespace

size_t attend_backward_smem(int H, int d) {
  return sizeof(float) * (3 * (size_t)H * d + 2 * (size_t)kBwdKeys * (d + 1) +
                          2 * (size_t)H * kBwdKeys + 2 * H + 2) +
         (sizeof(int64_t) + sizeof(int)) * kBwdKeys + 16;
}

cudaError_t launch_attend_backward(const AttnBwdArgs& a, cudaStream_t st) {
  const int64_t rows = (int64_t)a.B * a.T;
  if (rows == 0) return cudaSuccess;
  const size_t smem = attend_backward_smem(a.H, a.d);
  cudaError_t e;
  if (a.dtype == SA_BF16) {
    e = cudaFuncSetAttribute(attend_backward_kernel<SA_BF16>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attend_backward_kernel<SA_BF16><<<(unsigned)(rows * a.nsplit), kBwdThreads, smem, st>>>(a);
  } else {
    e = cudaFuncSetAttribute(attend_backward_kernel<SA_F32>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attend_backward_kernel<SA_F32><<<(unsigned)(rows * a.nsplit), kBwdThreads, smem, st>>>(a);
  }
  return cudaGetLastError();
}

int attend_backward_key_tile() { return kBwdKeys; }

cudaError_t launch_compress_backward(const CompressBwdArgs& a, cudaStream_t st) {
  if (a.max_blocks <= 0 || a.B <= 0) return cudaSuccess;
  const dim3 grid(a.max_blocks, a.B);
  const size_t smem = sizeof(float) * 2 * (size_t)a.m;
  if (a.dtype == SA_BF16)
    compress_backward_kernel<SA_BF16><<<grid, kBwdThreads, smem, st>>>(a);
  else
    compress_backward_kernel<SA_F32><<<grid, kBwdThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace sa
