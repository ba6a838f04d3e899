// Per-query top-k of the indexer scores: exact, deterministic radix select.
//
// Source: "오픈소스 LLM의 새 이정표: DeepSeek-V4 시리즈", section
// "압축 희소 어텐션(CSA)과 극압축 어텐션(HCA)" (each query attends only its top-k
// compressed entries) and "DeepSeek-V4 논문 읽기: 백만 토큰 컨텍스트를 저렴하게",
// section "Compressed Sparse Attention (CSA)" step 3.  Ties go to the lower
// index and the output is in ascending index order (readings where the pages
// are silent).
//
// Rows of up to 32768 candidates use topk_row_kernel (one CTA per row; a
// sample threshold cuts the row to a short candidate list first, see there).
// Longer rows: the row's candidates are split over a thread-block cluster of
// C CTAs (C = 1 while the row fits one CTA's shared memory); CTA c keeps the order-
// preserving 32-bit keys of candidates [c*chunk, (c+1)*chunk) in shared
// memory.  Three radix passes (11, 11, 10 bits, most significant first) find
// the exact k-th largest key T: each CTA histograms the keys that still match
// the prefix chosen so far (lanes of a warp that hit the same bin add once,
// through match.any), the C histograms are summed through distributed shared
// memory, and every CTA picks the digit where the count of larger keys first
// reaches the remaining quota.  Then every key > T is kept and, of the keys
// == T, the lowest indices fill what is left of k.  The output position of
// candidate i is (#keys > T before i) + min(#keys == T before i, quota), so
// each CTA compacts its slice in index order, 1024 keys at a time with warp
// ballots: the output comes out sorted without a sort.
#include "kernels.cuh"

namespace sa {

constexpr int kTopkThreads = 1024;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kBins = 2048;
constexpr int kMaxChunk = 49152;      // keys per CTA in shared memory (192 KB)
constexpr int kMaxCluster = 8;        // portable cluster size

struct TopkSmem {
  int hist[2][kBins];
  int scan[kTopkWarps + 1];
  int wgt[2 * kTopkWarps], weq[kTopkWarps];   // per-warp counts / min-max scratch
  __align__(8) int cnt[2];                // this CTA: keys > T, keys == T
  int nan_flag;
  int sel_bin, above;
};

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Sum of `v` over the CTA, returned to every thread.
__device__ __forceinline__ int block_sum(int v, int* scratch) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane == 0) scratch[w] = v;
  __syncthreads();
  int t = lane < kTopkWarps ? scratch[lane] : 0;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
  __syncthreads();
  return t;
}

template <bool kCluster>
__global__ void __launch_bounds__(kTopkThreads) topk_kernel(TopkArgs a, int C, int chunk) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  TopkSmem& S = *reinterpret_cast<TopkSmem*>(smem_raw);
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem_raw + sizeof(TopkSmem));
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rank = kCluster ? (int)cluster_rank() : 0;
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
  auto csync = [&]() {
    if constexpr (kCluster) cluster_sync(); else __syncthreads();
  };
  auto remote = [&](const void* p_, int r) -> const void* {
    if constexpr (kCluster) return __cluster_map_shared_rank(p_, r);
    else return p_;
  };

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
    for (int i0 = 0; i0 < cnt; i0 += kTopkThreads) {
      const int i = i0 + tid;
      const bool in = i < cnt;
      const uint32_t key = in ? keys[i] : 0u;
      const bool match = in && (key & maskbits) == prefix;
      const unsigned act = __ballot_sync(0xffffffffu, match);
      if (match) {
        const int bin = (int)((key >> shift) & (uint32_t)(nb - 1));
        const unsigned same = __match_any_sync(act, bin);
        if ((same & lanemask_lt()) == 0) atomicAdd(&h[bin], __popc(same));
      }
    }
    __syncthreads();
    csync();
    if (pass == 0) {
      int any_nan = 0;
#pragma unroll
      for (int r = 0; r < kMaxCluster; ++r)
        if (r < C) any_nan |= *static_cast<const int*>(remote(&S.nan_flag, r));
      if (any_nan) {                              // reject the row: all -1
        if (rank == 0 && tid == 0) set_err(a.err, SA_ERR_NAN);
        for (int64_t i = (int64_t)rank * kTopkThreads + tid; i < k; i += (int64_t)C * kTopkThreads)
          out[i] = -1;
        csync();                                  // peers may still read our smem
        return;
      }
    }
    // Sum the C histograms.  Counting from the top digit down, thread t owns
    // bins nb-1-per*t .. nb-per*(t+1) (per = 2 for nb = 2048, 1 for 1024):
    // one 8- or 4-byte load from every CTA of the cluster, all issued before
    // any is used.
    const int per = nb / kTopkThreads;
    int loc0 = 0, loc1 = 0;
    if (per == 2) {
      int2 v[kMaxCluster];
#pragma unroll
      for (int r = 0; r < kMaxCluster; ++r)
        if (r < C) v[r] = *static_cast<const int2*>(
                       remote(reinterpret_cast<const int2*>(h + nb - 2 * (tid + 1)), r));
#pragma unroll
      for (int r = 0; r < kMaxCluster; ++r)
        if (r < C) { loc0 += v[r].y; loc1 += v[r].x; }
    } else {
      int v[kMaxCluster];
#pragma unroll
      for (int r = 0; r < kMaxCluster; ++r)
        if (r < C) v[r] = *static_cast<const int*>(remote(h + nb - 1 - tid, r));
#pragma unroll
      for (int r = 0; r < kMaxCluster; ++r)
        if (r < C) loc0 += v[r];
    }
    const int base = block_exclusive_scan<kTopkThreads>(loc0 + loc1, S.scan, nullptr);
    {
      const int b0 = nb - 1 - tid * per;          // loc0 is bin b0, loc1 bin b0 - 1
      if (base < krem && base + loc0 >= krem) { S.sel_bin = b0; S.above = base; }
      if (per == 2) {
        const int before = base + loc0;
        if (before < krem && before + loc1 >= krem) { S.sel_bin = b0 - 1; S.above = before; }
      }
    }
    __syncthreads();
    krem -= S.above;
    prefix |= (uint32_t)S.sel_bin << shift;
    maskbits |= (uint32_t)(nb - 1) << shift;
    __syncthreads();
  }
  const uint32_t T = prefix;                      // the k-th largest key; take krem of the == T

  // ---- counts of this CTA's slice, then of the CTAs before it
  int n_gt = 0, n_eq = 0;
  for (int i = tid; i < cnt; i += kTopkThreads) {
    n_gt += keys[i] > T;
    n_eq += keys[i] == T;
  }
  const int gt_total = block_sum(n_gt, S.scan);
  const int eq_total = block_sum(n_eq, S.scan);
  if (tid == 0) { S.cnt[0] = gt_total; S.cnt[1] = eq_total; }
  __syncthreads();
  csync();
  int eq_before = 0, gt_before = 0;
  if constexpr (kCluster) {
    int2 v[kMaxCluster];
#pragma unroll
    for (int r = 0; r < kMaxCluster; ++r)
      if (r < rank) v[r] = *static_cast<const int2*>(remote(reinterpret_cast<const int2*>(S.cnt), r));
#pragma unroll
    for (int r = 0; r < kMaxCluster; ++r)
      if (r < rank) { gt_before += v[r].x; eq_before += v[r].y; }
  }

  // ---- compaction in index order, kTopkThreads keys per round.  Candidate i
  // (key > T, or key == T with eq(<i) < krem) goes to gt(<i) + min(eq(<i), krem),
  // with gt/eq counted over the whole row.
  int run_gt = gt_before, run_eq = eq_before;
  for (int i0 = 0; i0 < cnt; i0 += kTopkThreads) {
    const int i = i0 + tid;
    const uint32_t key = i < cnt ? keys[i] : 0u;
    const bool gt = i < cnt && key > T;
    const bool eq = i < cnt && key == T;
    const unsigned bg = __ballot_sync(0xffffffffu, gt), be = __ballot_sync(0xffffffffu, eq);
    if (lane == 0) { S.wgt[warp] = __popc(bg); S.weq[warp] = __popc(be); }
    __syncthreads();
    const int cg = lane < kTopkWarps ? S.wgt[lane] : 0;
    const int ce = lane < kTopkWarps ? S.weq[lane] : 0;
    int xg = cg, xe = ce;                         // inclusive scan over the warps
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int yg = __shfl_up_sync(0xffffffffu, xg, o), ye = __shfl_up_sync(0xffffffffu, xe, o);
      if (lane >= o) { xg += yg; xe += ye; }
    }
    const int pg = __shfl_sync(0xffffffffu, xg - cg, warp);   // keys of the warps before
    const int pe = __shfl_sync(0xffffffffu, xe - ce, warp);
    const int tg = __shfl_sync(0xffffffffu, xg, 31);          // this round's totals
    const int te = __shfl_sync(0xffffffffu, xe, 31);
    const int g_lt = run_gt + pg + __popc(bg & lanemask_lt());
    const int e_lt = run_eq + pe + __popc(be & lanemask_lt());
    if (gt) out[g_lt + min(e_lt, krem)] = (int32_t)(lo + i);
    else if (eq && e_lt < krem) out[g_lt + e_lt] = (int32_t)(lo + i);
    run_gt += tg;
    run_eq += te;
    __syncthreads();                              // per-warp counts are rewritten next round
  }
  if constexpr (kCluster) cluster_sync();         // keep smem alive for peers' DSMEM reads
}

// ------------------------------------------------------------------------
// Rows of at most kRowMax candidates: one CTA per row, no cluster.
//  1. keys -> shared memory; every 16th key is a sample;
//  2. a threshold Ts low enough that about 1.3 k keys reach it, read off the
//     samples (an order statistic of the sample, by the radix select below);
//  3. the keys >= Ts are compacted, in index order, into a candidate list;
//  4. the exact radix select runs on the candidates only: every key >= the
//     k-th largest T is >= Ts, so the list holds all of them and all ties at T.
// If the list comes out shorter than k or longer than its buffer (a skewed or
// tied row), steps 3-4 fall back to the radix select over all the row's keys.
constexpr int kRowMax = 32768;
constexpr int kTopkSmemBytes = (sizeof(TopkSmem) + 15) & ~15;   // keys start 16-byte aligned
constexpr int kCandMax = 8192;
constexpr int kSampleStride = 16;

// The kk-th largest of keys[0..m) (1 <= kk <= m), by three radix passes of
// 11, 11 and 10 bits; *take = how many keys equal to it belong to the top kk.
__device__ uint32_t radix_select(const uint32_t* keys, int m, int kk, TopkSmem& S, int* take) {
  const int tid = threadIdx.x;
  uint32_t prefix = 0, maskbits = 0;
  int krem = kk;
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const int nb = pass == 2 ? 1024 : 2048;
    int* h = S.hist[pass & 1];
    for (int i = tid; i < nb; i += kTopkThreads) h[i] = 0;
    __syncthreads();
    for (int i0 = 0; i0 < m; i0 += kTopkThreads) {
      const int i = i0 + tid;
      const bool in = i < m;
      const uint32_t key = in ? keys[i] : 0u;
      const bool match = in && (key & maskbits) == prefix;
      const unsigned act = __ballot_sync(0xffffffffu, match);
      if (match) {
        const int bin = (int)((key >> shift) & (uint32_t)(nb - 1));
        const unsigned same = __match_any_sync(act, bin);
        if ((same & lanemask_lt()) == 0) atomicAdd(&h[bin], __popc(same));
      }
    }
    __syncthreads();
    const int per = nb / kTopkThreads;
    const int loc0 = h[nb - 1 - tid * per];
    const int loc1 = per == 2 ? h[nb - 2 - tid * per] : 0;
    const int base = block_exclusive_scan<kTopkThreads>(loc0 + loc1, S.scan, nullptr);
    const int b0 = nb - 1 - tid * per;
    if (base < krem && base + loc0 >= krem) { S.sel_bin = b0; S.above = base; }
    if (per == 2) {
      const int before = base + loc0;
      if (before < krem && before + loc1 >= krem) { S.sel_bin = b0 - 1; S.above = before; }
    }
    __syncthreads();
    krem -= S.above;
    prefix |= (uint32_t)S.sel_bin << shift;
    maskbits |= (uint32_t)(nb - 1) << shift;
    __syncthreads();
  }
  *take = krem;
  return prefix;
}

// Rounds of the list passes: each thread takes kKpt consecutive entries.
constexpr int kKpt = 8;
constexpr int kRound = kKpt * kTopkThreads;

// keys[ib .. ib+7] by two 16-byte shared loads (entries past m read as 0 and
// are masked by the callers).  Lists are 16-byte aligned and padded to a
// multiple of 8 entries, so a group that starts below m is in bounds.
__device__ __forceinline__ void load8(const uint32_t* keys, int ib, int m, uint32_t* kk) {
  if (ib < m) {
    const uint4 u0 = *reinterpret_cast<const uint4*>(keys + ib);
    const uint4 u1 = *reinterpret_cast<const uint4*>(keys + ib + 4);
    kk[0] = u0.x; kk[1] = u0.y; kk[2] = u0.z; kk[3] = u0.w;
    kk[4] = u1.x; kk[5] = u1.y; kk[6] = u1.z; kk[7] = u1.w;
  } else {
#pragma unroll
    for (int j = 0; j < kKpt; ++j) kk[j] = 0u;
  }
}

// Write, in list order, the entries with key > T and the first `take` with
// key == T: out[p] = idx_of(i) for the p-th such entry.  The counts of a
// thread's entries (key > T in the high half, key == T in the low half of one
// int) are prefix-summed over the CTA once per round.
template <typename IdxOf>
__device__ void emit_selected(const uint32_t* keys, int m, uint32_t T, int take, TopkSmem& S,
                              int32_t* out, IdxOf idx_of) {
  const int tid = threadIdx.x;
  int run_gt = 0, run_eq = 0;
  for (int i0 = 0; i0 < m; i0 += kRound) {
    const int ib = i0 + tid * kKpt;
    uint32_t kk[kKpt];
    int ng = 0, ne = 0;
    load8(keys, ib, m, kk);
#pragma unroll
    for (int j = 0; j < kKpt; ++j) {
      ng += ib + j < m && kk[j] > T;
      ne += ib + j < m && kk[j] == T;
    }
    int tot;
    const int pre = block_exclusive_scan<kTopkThreads>((ng << 16) | ne, S.scan, &tot);
    int g_lt = run_gt + (pre >> 16), e_lt = run_eq + (pre & 0xFFFF);
#pragma unroll
    for (int j = 0; j < kKpt; ++j) {
      if (ib + j >= m) break;
      if (kk[j] > T) {
        out[g_lt + min(e_lt, take)] = idx_of(ib + j);
        ++g_lt;
      } else if (kk[j] == T) {
        if (e_lt < take) out[g_lt + e_lt] = idx_of(ib + j);
        ++e_lt;
      }
    }
    run_gt += tot >> 16;
    run_eq += tot & 0xFFFF;
  }
}

// Min and max of v over the CTA, returned to every thread.
__device__ __forceinline__ void block_minmax(uint32_t lo, uint32_t hi, uint32_t* mn, uint32_t* mx,
                                             int* scratch /* >= 2 * kTopkWarps */) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  uint32_t a = lo, b = hi;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a = min(a, __shfl_xor_sync(0xffffffffu, a, o));
    b = max(b, __shfl_xor_sync(0xffffffffu, b, o));
  }
  if (lane == 0) { scratch[2 * w] = (int)a; scratch[2 * w + 1] = (int)b; }
  __syncthreads();
  a = lane < kTopkWarps ? (uint32_t)scratch[2 * lane] : 0xffffffffu;
  b = lane < kTopkWarps ? (uint32_t)scratch[2 * lane + 1] : 0u;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a = min(a, __shfl_xor_sync(0xffffffffu, a, o));
    b = max(b, __shfl_xor_sync(0xffffffffu, b, o));
  }
  __syncthreads();
  *mn = a;
  *mx = b;
}

// A key Ts such that at least r of keys[0..m) are >= Ts (1 <= r <= m), close
// to the r-th largest: the lower edge of the linear bin (2048 bins over
// [min, max]) that holds the r-th largest key.
__device__ uint32_t threshold_at_least(const uint32_t* keys, int m, int r, TopkSmem& S) {
  const int tid = threadIdx.x;
  uint32_t lo = 0xffffffffu, hi = 0u;
  for (int i = tid; i < m; i += kTopkThreads) { lo = min(lo, keys[i]); hi = max(hi, keys[i]); }
  uint32_t kmin, kmax;
  block_minmax(lo, hi, &kmin, &kmax, S.wgt);
  const uint64_t span = (uint64_t)(kmax - kmin) + 1;
  int* h = S.hist[0];
  for (int i = tid; i < kBins; i += kTopkThreads) h[i] = 0;
  __syncthreads();
  for (int i = tid; i < m; i += kTopkThreads)
    atomicAdd(&h[(int)(((uint64_t)(keys[i] - kmin) * kBins) / span)], 1);
  __syncthreads();
  const int loc0 = h[kBins - 1 - 2 * tid], loc1 = h[kBins - 2 - 2 * tid];
  const int base = block_exclusive_scan<kTopkThreads>(loc0 + loc1, S.scan, nullptr);
  if (base < r && base + loc0 >= r) S.sel_bin = kBins - 1 - 2 * tid;
  else if (base + loc0 < r && base + loc0 + loc1 >= r) S.sel_bin = kBins - 2 - 2 * tid;
  __syncthreads();
  const uint64_t b = (uint64_t)S.sel_bin;
  __syncthreads();
  // smallest key whose bin is >= b
  return kmin + (uint32_t)((b * span + kBins - 1) / kBins);
}

__global__ void __launch_bounds__(kTopkThreads) topk_row_kernel(TopkArgs a, int n_pad) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  TopkSmem& S = *reinterpret_cast<TopkSmem*>(smem_raw);
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem_raw + kTopkSmemBytes);   // [n_pad]
  uint32_t* samp = keys + n_pad;                                             // [n_pad / 16]
  uint32_t* ck = samp + n_pad / kSampleStride;                               // [kCandMax]
  int32_t* ci = reinterpret_cast<int32_t*>(ck + kCandMax);                   // [kCandMax]
  const int tid = threadIdx.x;
  const int64_t row = blockIdx.x;
  const int k = a.k;
  int32_t* out = a.idx + row * k;
  const int p = __ldg(a.q_pos + row);
  int n = p < 0 ? 0 : (int)min64(((int64_t)p + 1) / a.m, a.N_cap);
  if (p >= 0 && ((int64_t)p + 1) / a.m > a.N_cap && tid == 0) set_err(a.err, SA_ERR_BOUNDS);
  if (n <= k) {
    for (int i = tid; i < k; i += kTopkThreads) out[i] = i < n ? i : -1;
    return;
  }
  const float* src = a.scores + row * a.ld;
  int nan_local = 0;
  int n4 = 0;
  if ((reinterpret_cast<uintptr_t>(src) & 15u) == 0) {       // 16-byte loads, four in flight
    n4 = n / 4;
    const float4* src4 = reinterpret_cast<const float4*>(src);
    uint4* keys4 = reinterpret_cast<uint4*>(keys);
#pragma unroll 4
    for (int i = tid; i < n4; i += kTopkThreads) {
      const float4 f = src4[i];
      nan_local |= is_nan_bits(f.x) | is_nan_bits(f.y) | is_nan_bits(f.z) | is_nan_bits(f.w);
      keys4[i] = make_uint4(score_key(f.x), score_key(f.y), score_key(f.z), score_key(f.w));
    }
  }
  for (int i = 4 * n4 + tid; i < n; i += kTopkThreads) {
    const float f = src[i];
    nan_local |= is_nan_bits(f);
    keys[i] = score_key(f);
  }
  if (__syncthreads_or(nan_local)) {
    if (tid == 0) set_err(a.err, SA_ERR_NAN);
    for (int i = tid; i < k; i += kTopkThreads) out[i] = -1;
    return;
  }
  const int ns = (n + kSampleStride - 1) / kSampleStride;
  for (int i = tid; i < ns; i += kTopkThreads) samp[i] = keys[i * kSampleStride];
  __syncthreads();
  int rs = (int)(((int64_t)k * ns * 13 + (int64_t)n * 10 - 1) / ((int64_t)n * 10));   // ~1.3 k/16
  rs = max(1, min(rs, ns));
  const uint32_t Ts = threshold_at_least(samp, ns, rs, S);
  // ---- candidates: keys >= Ts, in index order
  int count = 0;
  for (int i0 = 0; i0 < n; i0 += kRound) {
    const int ib = i0 + tid * kKpt;
    uint32_t kk[kKpt];
    int nc = 0;
    load8(keys, ib, n, kk);
#pragma unroll
    for (int j = 0; j < kKpt; ++j) nc += ib + j < n && kk[j] >= Ts;
    int tot;
    int pos = count + block_exclusive_scan<kTopkThreads>(nc, S.scan, &tot);
#pragma unroll
    for (int j = 0; j < kKpt; ++j) {
      if (ib + j < n && kk[j] >= Ts) {
        if (pos < kCandMax) { ck[pos] = kk[j]; ci[pos] = ib + j; }
        ++pos;
      }
    }
    count += tot;
  }
  __syncthreads();
  int take;
  if (count >= k && count <= kCandMax) {
    const uint32_t T = radix_select(ck, count, k, S, &take);
    emit_selected(ck, count, T, take, S, out, [&](int i) { return ci[i]; });
  } else {
    const uint32_t T = radix_select(keys, n, k, S, &take);
    emit_selected(keys, n, T, take, S, out, [&](int i) { return (int32_t)i; });
  }
}

bool topk_supported(int N_cap) { return N_cap <= kMaxChunk * kMaxCluster; }

cudaError_t launch_topk(const TopkArgs& a, int num_sms, cudaStream_t st) {
  if (a.rows <= 0) return cudaSuccess;
  if (a.N_cap <= kRowMax) {
    const int n_pad = (a.N_cap + 63) & ~63;   // keeps every list 16-byte aligned
    const size_t smem = kTopkSmemBytes + sizeof(uint32_t) * (size_t)(n_pad + n_pad / kSampleStride) +
                        (sizeof(uint32_t) + sizeof(int32_t)) * (size_t)kCandMax;
    cudaError_t e = cudaFuncSetAttribute(topk_row_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    topk_row_kernel<<<(unsigned)a.rows, kTopkThreads, smem, st>>>(a, n_pad);
    return cudaGetLastError();
  }
  // Cluster size: a power of two, enough CTAs to hold N_cap keys in shared
  // memory, doubled while there are too few rows to cover the SMs and each
  // CTA keeps at least 4096 keys (1: no cluster).
  int C = 1;
  while ((int64_t)C * kMaxChunk < a.N_cap) C *= 2;
  if (C > kMaxCluster) return cudaErrorInvalidValue;
  const int want = (num_sms + a.rows - 1) / a.rows;
  while (C < want && C < kMaxCluster && a.N_cap / (2 * C) >= 4096) C *= 2;
  int chunk = (a.N_cap + C - 1) / C;
  chunk = (chunk + 31) & ~31;
  if (chunk < 32) chunk = 32;
  const size_t smem = sizeof(TopkSmem) + sizeof(uint32_t) * (size_t)chunk;
  if (C == 1) {
    cudaError_t e = cudaFuncSetAttribute(topk_kernel<false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    topk_kernel<false><<<(unsigned)a.rows, kTopkThreads, smem, st>>>(a, 1, chunk);
    return cudaGetLastError();
  }
  cudaError_t e = cudaFuncSetAttribute(topk_kernel<true>,
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
  return cudaLaunchKernelEx(&cfg, topk_kernel<true>, a, C, chunk);
}

}  // namespace sa
