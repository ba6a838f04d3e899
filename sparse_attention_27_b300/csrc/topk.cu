// Per-query top-k of the indexer scores: exact and deterministic.
//
// Source: "오픈소스 LLM의 새 이정표: DeepSeek-V4 시리즈", section
// "압축 희소 어텐션(CSA)과 극압축 어텐션(HCA)" (each query attends only its top-k
// compressed entries) and "DeepSeek-V4 논문 읽기: 백만 토큰 컨텍스트를 저렴하게",
// section "Compressed Sparse Attention (CSA)" step 3.  Ties go to the lower
// index and the output is in ascending index order (readings where the pages
// are silent).
//
// One kernel, topk_rows_kernel: a row's candidates are split over a cluster of
// up to 16 CTAs, one histogram pass finds the bin of the k-th largest key, an
// exact select runs inside that bin, and the output is emitted in index order
// with warp ballots (see there).
#include "kernels.cuh"
#include "topk_dev.cuh"

namespace sa {

// topk_rows_kernel: step A's input -- the row's fp32 scores, turned into
// keys with 16-byte loads, the row's largest key (over the cluster), and the
// histogram of the keys binned relative to it (FineBins: 1024 bins per
// octave from 6 octaves below the largest key) -- then topk_select.
template <int NT, int KPL>
__global__ void __launch_bounds__(NT, 1) topk_rows_kernel(TopkArgs a, int C, int chunk) {
  constexpr int CAP = NT * KPL;                  // keys one CTA holds
  extern __shared__ __align__(16) unsigned char smem_raw[];
  TopkSmem& S = *reinterpret_cast<TopkSmem*>(smem_raw);
  int* hist = reinterpret_cast<int*>(smem_raw + kTopkSmemBytes);   // [kFineBins]; later the union
  uint32_t* keys = reinterpret_cast<uint32_t*>(hist + kFineBins);   // [CAP]
  uint32_t* ck = keys + CAP;                                        // [kCandMax] this CTA's list
  int32_t* ci = reinterpret_cast<int32_t*>(ck + kCandMax);          // [kCandMax]
  const int tid = threadIdx.x;
  const int rank = C > 1 ? (int)cluster_rank() : 0;
  const int64_t row = blockIdx.x / C;
  const int k = a.k;
  int32_t* out = a.idx + row * k;
  const int p = __ldg(a.q_pos + row);
  const int n = p < 0 ? 0 : (int)min64(((int64_t)p + 1) / a.m, a.N_cap);
  if (p >= 0 && ((int64_t)p + 1) / a.m > a.N_cap && rank == 0 && tid == 0)
    set_err(a.err, SA_ERR_BOUNDS);
  if (n <= k) {                                  // same for the whole cluster: no barrier
    for (int i = rank * NT + tid; i < k; i += C * NT) out[i] = i < n ? i : -1;
    return;
  }
  const int lo = rank * chunk;                   // this CTA's first candidate
  const int cnt = max(0, min(n, lo + chunk) - lo);
  // ---- A. keys and the 13-bit histogram.  Thread tid holds the 16-byte
  // groups tid + q*NT; slots past cnt get key 0, below every real score's key
  // (score_key(-inf) > 0).
  const float* src = a.scores + row * a.ld + lo;
  const bool vec = (reinterpret_cast<uintptr_t>(src) & 15u) == 0;
  const int n4 = vec ? cnt / 4 : 0;              // whole 16-byte groups read as vectors
  float4 f[KPL / 4];
#pragma unroll
  for (int q = 0; q < KPL / 4; ++q) {
    const int g = tid + q * NT;
    if (g < n4) {
      f[q] = reinterpret_cast<const float4*>(src)[g];
    } else {
      const int i = 4 * g;
      f[q] = make_float4(i < cnt ? src[i] : 0.f, i + 1 < cnt ? src[i + 1] : 0.f,
                         i + 2 < cnt ? src[i + 2] : 0.f, i + 3 < cnt ? src[i + 3] : 0.f);
    }
  }
  for (int i = tid; i < kFineBins; i += NT) hist[i] = 0;      // while the loads fly
  if (tid == 0) S.kmax = 0u;
  __syncthreads();
  int nan_local = 0;
  uint32_t kmax = 0u;
  auto put = [&](int i, float v) -> uint32_t {
    if (i >= cnt) return 0u;
    const bool nan = is_nan_bits(v);
    nan_local |= nan;
    const uint32_t key = score_key(v);
    if (!nan) kmax = max(kmax, key);
    return key;
  };
#pragma unroll
  for (int q = 0; q < KPL / 4; ++q) {
    const int g = tid + q * NT;
    reinterpret_cast<uint4*>(keys)[g] =
        make_uint4(put(4 * g, f[q].x), put(4 * g + 1, f[q].y), put(4 * g + 2, f[q].z),
                   put(4 * g + 3, f[q].w));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
  if ((tid & 31) == 0 && kmax > 0u) atomicMax(&S.kmax, kmax);
  if (C > 1) cluster_sync(); else __syncthreads();   // every CTA's largest key is in place
  uint32_t mx = S.kmax;
  for (int r = 0; r < C; ++r) mx = max(mx, C > 1 ? *peer(&S.kmax, r) : mx);
  const uint32_t v = mx >> 13;
  const FineBins fb = mx == 0u ? kAbsoluteBins
                               : FineBins{13, v > 6u * 1024u ? v - 6u * 1024u : 0u};
  for (int i = tid; i < CAP; i += NT) {
    const uint32_t key = keys[i];
    if (key != 0u) atomicAdd(&hist[fb.bin(key)], 1);
  }
  nan_local = __syncthreads_or(nan_local);
  topk_select<NT, KPL>(S, keys, cnt, lo, hist, ck, ci, nan_local, k, C, rank, a.err,
                       [&](int pos, int j) { out[pos] = j; }, fb);
}

static size_t rows_smem(int nt, int kpl) {
  return kTopkSmemBytes + sizeof(uint32_t) * ((size_t)kFineBins + (size_t)nt * kpl + 2 * kCandMax);
}

template <int NT, int KPL>
static bool rows_cluster_probe(int C) {
  auto kern = topk_rows_kernel<NT, KPL>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)rows_smem(NT, KPL)) != cudaSuccess)
    return false;
  if (C <= 1) return true;
  if (C > 8 && cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
                   cudaSuccess)
    return false;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)C);
  cfg.blockDim = dim3(NT);
  cfg.dynamicSmemBytes = rows_smem(NT, KPL);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int nclusters = 0;
  if (cudaOccupancyMaxActiveClusters(&nclusters, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return nclusters > 0;
}

// Whether clusters of C CTAs (C = 1: plain CTAs) of a (NT, KPL) instance can
// be resident, with its shared memory set up; cached per device and C.
template <int NT, int KPL>
static bool rows_cluster_ok(int C) {
  static int cache[64][5];                       // [device][log2 C]: 0 unknown, 1 yes, 2 no
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  int lc = 0;
  while ((1 << lc) < C) ++lc;
  if (lc > 4) return false;
  if (cache[dev][lc] != 0) return cache[dev][lc] == 1;
  const bool ok = rows_cluster_probe<NT, KPL>(C);
  cache[dev][lc] = ok ? 1 : 2;
  return ok;
}

template <int NT, int KPL>
static cudaError_t launch_rows(const TopkArgs& a, int C, int chunk, cudaStream_t st) {
  auto kern = topk_rows_kernel<NT, KPL>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(a.rows * C));
  cfg.blockDim = dim3(NT);
  cfg.dynamicSmemBytes = rows_smem(NT, KPL);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = C > 1 ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, a, C, chunk);
}

bool topk_supported(int N_cap) { return N_cap <= kRowsMaxCluster * 1024 * kKplMax; }

cudaError_t launch_topk(const TopkArgs& a, int num_sms, cudaStream_t st) {
  if (a.rows <= 0) return cudaSuccess;
  // Cluster size: the largest power of two (at most 16) that keeps one wave
  // (rows * C <= SMs) and at least 4096 candidates per CTA; then the fewest
  // threads and keys per thread that hold a CTA's share.  A row that no
  // cluster size the device runs can hold is not supported.
  int C = 1;
  while (2 * C <= kRowsMaxCluster && (int64_t)a.rows * 2 * C <= num_sms &&
         a.N_cap / (2 * C) >= 4096)
    C *= 2;
  while (C < kRowsMaxCluster && (int64_t)C * 1024 * kKplMax < a.N_cap) C *= 2;
  for (; C >= 1; C /= 2) {
    if ((int64_t)C * 1024 * kKplMax < a.N_cap) break;            // cannot hold the row
    int chunk = (a.N_cap + C - 1) / C;
    chunk = (chunk + 3) & ~3;
    cudaError_t e = cudaErrorNotSupported;
    if (C == 1 && chunk <= 256 * 32) {
      if (rows_cluster_ok<256, 32>(C)) e = launch_rows<256, 32>(a, C, chunk, st);
    } else if (C == 1 && chunk <= 512 * 32) {
      if (rows_cluster_ok<512, 32>(C)) e = launch_rows<512, 32>(a, C, chunk, st);
    } else if (chunk <= 1024 * 8) {
      if (rows_cluster_ok<1024, 8>(C)) e = launch_rows<1024, 8>(a, C, chunk, st);
    } else if (chunk <= 1024 * 16) {
      if (rows_cluster_ok<1024, 16>(C)) e = launch_rows<1024, 16>(a, C, chunk, st);
    } else {
      if (rows_cluster_ok<1024, 32>(C)) e = launch_rows<1024, 32>(a, C, chunk, st);
    }
    if (e != cudaErrorNotSupported) return e;
  }
  return cudaErrorNotSupported;
}

}  // namespace sa
