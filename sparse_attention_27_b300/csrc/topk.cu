// Per-query top-k of the indexer scores: exact, deterministic radix select
// spread over a thread-block cluster.
//
// Source: "오픈소스 LLM의 새 이정표: DeepSeek-V4 시리즈", section
// "압축 희소 어텐션(CSA)과 극압축 어텐션(HCA)" (each query attends only its top-k
// compressed entries) and "DeepSeek-V4 논문 읽기: 백만 토큰 컨텍스트를 저렴하게",
// section "Compressed Sparse Attention (CSA)" step 3.  Ties go to the lower
// index and the output is in ascending index order (readings where the pages
// are silent).
//
// Design.  One cluster of C CTAs per query row; CTA c keeps the order-
// preserving 32-bit keys of candidates [c*chunk, (c+1)*chunk) in shared
// memory.  Three radix passes (11, 11, 10 bits, most significant first) find
// the exact k-th largest key T: each CTA histograms the keys that still match
// the prefix chosen so far, every CTA sums the C histograms through
// distributed shared memory, and picks the digit where the count of larger
// keys first reaches the remaining quota.  Histograms are double-buffered so
// one cluster barrier per pass suffices.  Then every key > T is kept, and of
// the keys == T the lowest indices fill what is left of k: each CTA learns the
// counts of the CTAs before it (DSMEM) and compacts its slice in index order,
// so the output comes out sorted without a sort.
#include "kernels.cuh"

namespace sa {

constexpr int kTopkThreads = 512;
constexpr int kBins = 2048;
constexpr int kMaxChunk = 49152;      // keys per CTA in shared memory
constexpr int kMaxCluster = 8;       // portable cluster size

struct TopkSmem {
  int hist[2][kBins];
  int scan[kTopkThreads / 32 + 1];
  __align__(8) int cnt[2];   // this CTA: keys > T, keys == T
  int nan_flag;
  int sel_bin, above;
};

__global__ void __launch_bounds__(kTopkThreads) topk_cluster_kernel(TopkArgs a, int C, int chunk) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  TopkSmem& S = *reinterpret_cast<TopkSmem*>(smem_raw);
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem_raw + sizeof(TopkSmem));
  const int tid = threadIdx.x;
  const int rank = (int)cluster_rank();
  const int64_t row = blockIdx.x / C;
  const int k = a.k;
  int32_t* out = a.idx + row * k;
  const int p = __ldg(a.q_pos + row);
  int64_t n = p < 0 ? 0 : ((int64_t)p + 1) / a.m;
  if (n > a.N_cap) {
    if (rank == 0 && tid == 0) set_err(a.err, SA_ERR_BOUNDS);
    n = a.N_cap;
  }
  if (n <= k) {                                   // everything visible is selected
    for (int64_t i = (int64_t)rank * kTopkThreads + tid; i < k; i += (int64_t)C * kTopkThreads)
      out[i] = i < n ? (int32_t)i : -1;
    return;
  }
  const int64_t lo = (int64_t)rank * chunk;
  const int cnt = (int)max64(0, min64(n, lo + chunk) - lo);
  const float* src = a.scores + row * a.ld + lo;
  int nan_local = 0;
  for (int i = tid; i < cnt; i += kTopkThreads) {
    const float f = src[i];
    nan_local |= is_nan_bits(f);
    keys[i] = score_key(f);
  }
  nan_local = __syncthreads_or(nan_local);
  if (tid == 0) S.nan_flag = nan_local;

  uint32_t prefix = 0, maskbits = 0;
  int krem = k;
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const int nb = pass == 2 ? 1024 : 2048;
    int* h = S.hist[pass & 1];
    for (int i = tid; i < nb; i += kTopkThreads) h[i] = 0;
    __syncthreads();
    for (int i = tid; i < cnt; i += kTopkThreads) {
      const uint32_t key = keys[i];
      if ((key & maskbits) == prefix) atomicAdd(&h[(key >> shift) & (nb - 1)], 1);
    }
    __syncthreads();
    cluster_sync();
    if (pass == 0) {
      int any_nan = 0;
#pragma unroll
      for (int r = 0; r < kMaxCluster; ++r)
        if (r < C) any_nan |= *static_cast<const int*>(__cluster_map_shared_rank(&S.nan_flag, r));
      if (any_nan) {                              // reject the row: all -1
        if (rank == 0 && tid == 0) set_err(a.err, SA_ERR_NAN);
        for (int64_t i = (int64_t)rank * kTopkThreads + tid; i < k; i += (int64_t)C * kTopkThreads)
          out[i] = -1;
        cluster_sync();                           // peers may still read our smem
        return;
      }
    }
    // Sum the C histograms.  Counting from the top digit down, thread t owns
    // bins nb-1-per*t .. nb-per*(t+1) (per = 4 for nb = 2048, 2 for 1024):
    // one 16- or 8-byte load from every CTA of the cluster, all issued before
    // any is used.
    const int per = nb / kTopkThreads;
    int loc[4] = {0, 0, 0, 0};
    if (per == 4) {
      int4 v[kMaxCluster];
#pragma unroll
      for (int r = 0; r < kMaxCluster; ++r)
        if (r < C) v[r] = *static_cast<const int4*>(__cluster_map_shared_rank(
                       reinterpret_cast<const int4*>(h + nb - 4 * (tid + 1)), r));
#pragma unroll
      for (int r = 0; r < kMaxCluster; ++r)
        if (r < C) { loc[0] += v[r].w; loc[1] += v[r].z; loc[2] += v[r].y; loc[3] += v[r].x; }
    } else {
      int2 v[kMaxCluster];
#pragma unroll
      for (int r = 0; r < kMaxCluster; ++r)
        if (r < C) v[r] = *static_cast<const int2*>(__cluster_map_shared_rank(
                       reinterpret_cast<const int2*>(h + nb - 2 * (tid + 1)), r));
#pragma unroll
      for (int r = 0; r < kMaxCluster; ++r)
        if (r < C) { loc[0] += v[r].y; loc[1] += v[r].x; }
    }
    int tot = loc[0] + loc[1] + loc[2] + loc[3];
    int base = block_exclusive_scan<kTopkThreads>(tot, S.scan, nullptr);
    for (int e = 0; e < per; ++e) {
      const int before = base, incl = base + loc[e];
      if (before < krem && incl >= krem) {
        S.sel_bin = nb - 1 - (tid * per + e);
        S.above = before;
      }
      base = incl;
    }
    __syncthreads();
    krem -= S.above;
    prefix |= (uint32_t)S.sel_bin << shift;
    maskbits |= (uint32_t)(nb - 1) << shift;
    __syncthreads();
  }
  const uint32_t T = prefix;                      // the k-th largest key; take krem of the == T

  // ---- compaction in index order
  const int per = (cnt + kTopkThreads - 1) / kTopkThreads;
  const int s0 = min(cnt, tid * per), s1 = min(cnt, s0 + per);
  int n_gt = 0, n_eq = 0;
  for (int i = s0; i < s1; ++i) {
    n_gt += keys[i] > T;
    n_eq += keys[i] == T;
  }
  int eq_total, gt_total;
  const int eq_base = block_exclusive_scan<kTopkThreads>(n_eq, S.scan, &eq_total);
  block_exclusive_scan<kTopkThreads>(n_gt, S.scan, &gt_total);
  if (tid == 0) { S.cnt[0] = gt_total; S.cnt[1] = eq_total; }
  __syncthreads();
  cluster_sync();
  int eq_before = 0, gt_before = 0;
  {
    int2 v[kMaxCluster];
#pragma unroll
    for (int r = 0; r < kMaxCluster; ++r)
      if (r < rank) v[r] = *static_cast<const int2*>(__cluster_map_shared_rank(
                       reinterpret_cast<const int2*>(S.cnt), r));
#pragma unroll
    for (int r = 0; r < kMaxCluster; ++r)
      if (r < rank) { gt_before += v[r].x; eq_before += v[r].y; }
  }
  const int quota = max(0, min(krem - eq_before, eq_total));
  const int sel_before = gt_before + min(eq_before, krem);
  const int my_eq_sel = max(0, min(quota - eq_base, n_eq));
  const int sel_base = block_exclusive_scan<kTopkThreads>(n_gt + my_eq_sel, S.scan, nullptr);
  int pos = sel_before + sel_base, eq_rank = eq_base;
  for (int i = s0; i < s1; ++i) {
    const uint32_t key = keys[i];
    if (key > T) {
      out[pos++] = (int32_t)(lo + i);
    } else if (key == T) {
      if (eq_rank < quota) out[pos++] = (int32_t)(lo + i);
      ++eq_rank;
    }
  }
  cluster_sync();                                 // keep smem alive for peers' DSMEM reads
}

bool topk_supported(int N_cap) { return N_cap <= kMaxChunk * kMaxCluster; }

cudaError_t launch_topk(const TopkArgs& a, int num_sms, cudaStream_t st) {
  if (a.rows <= 0) return cudaSuccess;
  // Cluster size: a power of two, enough CTAs to hold N_cap keys in shared
  // memory, doubled while there are too few rows to cover the SMs.
  int C = 1;
  while ((int64_t)C * kMaxChunk < a.N_cap) C *= 2;
  if (C > kMaxCluster) return cudaErrorInvalidValue;
  const int want = (num_sms + a.rows - 1) / a.rows;
  while (C < want && C < kMaxCluster && a.N_cap / (2 * C) >= 2048) C *= 2;
  int chunk = (a.N_cap + C - 1) / C;
  chunk = (chunk + 31) & ~31;
  if (chunk < 32) chunk = 32;
  const size_t smem = sizeof(TopkSmem) + sizeof(uint32_t) * (size_t)chunk;
  cudaError_t e = cudaFuncSetAttribute(topk_cluster_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(C * a.rows));
  cfg.blockDim = dim3(kTopkThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, topk_cluster_kernel, a, C, chunk);
}

}  // namespace sa
