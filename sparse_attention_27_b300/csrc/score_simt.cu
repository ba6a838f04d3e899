// Lightning-indexer scores on CUDA cores (fp32 inputs, or any shape the
// tensor-core kernel does not take):
//     s[r, j] = sum_h w[r,h] * max(0, q_I[r,h,:] . Ik_c[b,j,:]),  j < n(r)
// Source: "EP 95. DeepSeek-V4 논문 읽기 — 노정석", section IDEAS (lightning indexer
// selecting the top-k of the compressed cache), and "DeepSeek-V4 논문 읽기:
// 백만 토큰 컨텍스트를 저렴하게", section "Compressed Sparse Attention (CSA)" step 2.
// The weighted ReLU head sum is the reading taken where the pages give no
// formula.  fp32 FMA throughout, so fp32 inputs keep ~1e-6 relative error.
//
// Grid (query rows, entry tiles of 128); one thread per compressed entry; the
// row's indexer queries and weights sit in shared memory (broadcast reads).
#include "kernels.cuh"

namespace sa {

constexpr int kScoreSimtThreads = 128;

template <int DT>
__global__ void __launch_bounds__(kScoreSimtThreads) score_simt_kernel(ScoreArgs a) {
  using S = Store<DT>;
  extern __shared__ float s_q[];           // [HI*dI] then w [HI]
  const int r = blockIdx.x;
  const int b = r / a.T;
  const int p = __ldg(a.q_pos + r);
  int64_t n = p < 0 ? 0 : ((int64_t)p + 1) / a.m;
  if (n > a.N_cap) {
    if (blockIdx.y == 0 && threadIdx.x == 0) set_err(a.err, SA_ERR_BOUNDS);
    n = a.N_cap;
  }
  const int64_t j0 = (int64_t)blockIdx.y * kScoreSimtThreads;
  if (j0 >= n) return;
  const int HI = a.HI, dI = a.dI;
  float* s_w = s_q + HI * dI;
  for (int i = threadIdx.x; i < HI * dI; i += blockDim.x)
    s_q[i] = S::ld(a.q, (int64_t)r * HI * dI + i);
  for (int i = threadIdx.x; i < HI; i += blockDim.x) s_w[i] = __ldg(a.w + (int64_t)r * HI + i);
  __syncthreads();
  const int64_t j = j0 + threadIdx.x;
  if (j >= n) return;
  const int64_t kbase = ((int64_t)b * a.N_cap + j) * dI;
  float acc = 0.f;
  for (int h = 0; h < HI; ++h) {
    float dot = 0.f;
    for (int c = 0; c < dI; ++c) dot = fmaf(s_q[h * dI + c], S::ld(a.ik, kbase + c), dot);
    acc = fmaf(s_w[h], fmaxf(dot, 0.f), acc);
  }
  a.scores[(int64_t)r * a.ld + j] = acc;
}

cudaError_t launch_score_simt(const ScoreArgs& a, cudaStream_t st) {
  dim3 grid(a.B * a.T, (a.N_cap + kScoreSimtThreads - 1) / kScoreSimtThreads);
  size_t smem = sizeof(float) * (a.HI * a.dI + a.HI);
  if (a.dtype == SA_BF16)
    score_simt_kernel<SA_BF16><<<grid, kScoreSimtThreads, smem, st>>>(a);
  else
    score_simt_kernel<SA_F32><<<grid, kScoreSimtThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace sa
