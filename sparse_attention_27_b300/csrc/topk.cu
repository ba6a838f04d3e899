// Per-query top-k of the indexer scores: exact, deterministic radix select.
//
// Source: "오픈소스 LLM의 새 이정표: DeepSeek-V4 시리즈", section
// "압축 희소 어텐션(CSA)과 극압축 어텐션(HCA)" (each query attends only its top-k
// compressed entries) and "DeepSeek-V4 논문 읽기: 백만 토큰 컨텍스트를 저렴하게",
// section "Compressed Sparse Attention (CSA)" step 3.  Ties go to the lower
// index and the output is in ascending index order (readings where the pages
// are silent).
//
// Rows of up to 32768 candidates use topk_row_kernel (one CTA per row, keys
// in registers, one histogram pass and an exact select inside one bin; see
// there).  Longer rows: the row's candidates are split over a thread-block cluster of
// C CTAs (C = 1 while the row fits one CTA's shared memory); CTA c keeps the order-
// preserving 32-bit keys of candidates [c*chunk, (c+1)*chunk) in shared
// memory.  Three radix passes (11, 11, 10 bits, most significant first) find
// the exact k-th largest key T: each CTA histograms the keys that still match
// the prefix chosen so far (one shared-memory atomic per key), the C
// histograms are summed through distributed shared memory, and every CTA picks the digit where the count of larger keys first
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
  int wg[kTopkWarps], we[kTopkWarps];     // row kernel: per-warp keys > T, keys == T
  int wc[kTopkWarps];                     // row kernel: per-warp keys in the selected bin
  int sel_bin, above;
  int ncand, take;                        // row kernel: keys in the selected bin, ties kept
  uint32_t T;                             // row kernel: the k-th largest key
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
      if (in && (key & maskbits) == prefix) atomicAdd(&h[(key >> shift) & (uint32_t)(nb - 1)], 1);
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
// Rows of at most kRowMax candidates: one CTA of NT threads per row; the row's
// keys sit in shared memory in index order.  Warp w owns candidates
// [w*32*kKpl, (w+1)*32*kKpl) and reads them 32 at a time (candidate
// w*32*kKpl + 32j + l in lane l, bank-conflict free), so a ballot over one j
// lists keys in index order.  Three passes over the row:
//  A. keys -> shared memory (16-byte loads) and a histogram of their top 13
//     bits (sign, exponent, 4 mantissa bits: 8192 bins, one atomic per key);
//     a scan of it gives the bin holding the k-th largest key;
//  B. that bin's keys are gathered with their indices, and every warp counts
//     its keys in higher bins; the exact k-th largest T comes from the bin's
//     keys alone (rank counting for a few, radix passes over the 19 low bits
//     otherwise; over the whole row if the bin overflows kCandMax);
//  C. emission in index order: out[#(> T) before i + min(#(== T) before i, take)].
constexpr int kRowMax = 32768;
constexpr int kKpl = 32;                                   // keys per thread
constexpr int kTopkSmemBytes = (sizeof(TopkSmem) + 15) & ~15;
constexpr int kFineShift = 19;                             // bin = key >> 19
constexpr int kFineBins = 1 << (32 - kFineShift);          // 8192
constexpr int kCandMax = 4096;                             // gathered keys of one bin
constexpr int kRankMax = 256;

// Over the histogram h[0..nb) (higher bin = larger keys): the bin b where the
// count of keys in bins >= b first reaches krem (1 <= krem <= total), and the
// count of keys in bins > b, to S.sel_bin / S.above.  Synchronises the CTA.
template <int NT>
__device__ void find_bin(const int* h, int nb, int krem, TopkSmem& S) {
  constexpr int NW = NT / 32;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int per = (nb + NT - 1) / NT;            // bins per thread, highest first
  int sum = 0;
  for (int q = 0; q < per; ++q) {
    const int b = nb - 1 - tid * per - q;
    sum += b >= 0 ? h[b] : 0;
  }
  int x = sum;                                   // inclusive scan within the warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) S.scan[w] = x;
  __syncthreads();
  int wt = lane < NW ? S.scan[lane] : 0;         // warp totals, scanned by every warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, wt, o);
    if (lane >= o) wt += y;
  }
  const int wbase = __shfl_sync(0xffffffffu, wt, (w + 31) & 31);
  int base = (w > 0 ? wbase : 0) + x - sum;
  for (int q = 0; q < per; ++q) {
    const int b = nb - 1 - tid * per - q;
    const int c = b >= 0 ? h[b] : 0;
    if (c > 0 && base < krem && base + c >= krem) { S.sel_bin = b; S.above = base; }
    base += c;
  }
  __syncthreads();
}

// The kk-th largest of those keys[0..m) whose top `top` bits equal prefix0's
// (1 <= kk <= their count), by radix passes of up to 11 bits over the bits
// below; *take = how many keys equal to it belong to the top kk.
template <int NT>
__device__ uint32_t radix_select(const uint32_t* keys, int m, int kk, TopkSmem& S, int* take,
                                 int top, uint32_t prefix0) {
  const int tid = threadIdx.x;
  uint32_t prefix = prefix0, maskbits = top > 0 ? (~0u << (32 - top)) : 0u;
  int krem = kk;
  int low = 32 - top;                            // bits still open
  while (low > 0) {
    const int nbits = min(11, low);
    const int shift = low - nbits;
    const int nb = 1 << nbits;
    int* h = S.hist[1];
    for (int i = tid; i < nb; i += NT) h[i] = 0;
    __syncthreads();
    for (int i = tid; i < m; i += NT) {
      const uint32_t key = keys[i];
      if ((key & maskbits) == prefix) atomicAdd(&h[(key >> shift) & (uint32_t)(nb - 1)], 1);
    }
    __syncthreads();
    find_bin<NT>(h, nb, krem, S);
    krem -= S.above;
    prefix |= (uint32_t)S.sel_bin << shift;
    maskbits |= (uint32_t)(nb - 1) << shift;
    low = shift;
    __syncthreads();
  }
  *take = krem;
  return prefix;
}

template <int NT>
__global__ void __launch_bounds__(NT, 1) topk_row_kernel(TopkArgs a) {
  constexpr int NW = NT / 32;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  TopkSmem& S = *reinterpret_cast<TopkSmem*>(smem_raw);
  int* hist = reinterpret_cast<int*>(smem_raw + kTopkSmemBytes);            // [kFineBins]
  uint32_t* keys = reinterpret_cast<uint32_t*>(hist + kFineBins);            // [NT * kKpl]
  uint32_t* ck = keys + NT * kKpl;                                           // [kCandMax]
  int32_t* ci = reinterpret_cast<int32_t*>(ck + kCandMax);                   // [kCandMax]
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int64_t row = blockIdx.x;
  const int k = a.k;
  int32_t* out = a.idx + row * k;
  const int p = __ldg(a.q_pos + row);
  const int n = p < 0 ? 0 : (int)min64(((int64_t)p + 1) / a.m, a.N_cap);
  if (p >= 0 && ((int64_t)p + 1) / a.m > a.N_cap && tid == 0) set_err(a.err, SA_ERR_BOUNDS);
  if (n <= k) {
    for (int i = tid; i < k; i += NT) out[i] = i < n ? i : -1;
    return;
  }
  // ---- A. keys and the 13-bit histogram.  Thread tid holds the 16-byte
  // groups tid + q*NT; slots past n get key 0, below every real score's key
  // (score_key(-inf) > 0).
  const float* src = a.scores + row * a.ld;
  const bool vec = (reinterpret_cast<uintptr_t>(src) & 15u) == 0;
  const int n4 = vec ? n / 4 : 0;                // whole 16-byte groups read as vectors
  float4 f[kKpl / 4];
#pragma unroll
  for (int q = 0; q < kKpl / 4; ++q) {
    const int g = tid + q * NT;
    if (g < n4) {
      f[q] = reinterpret_cast<const float4*>(src)[g];
    } else {
      const int i = 4 * g;
      f[q] = make_float4(i < n ? src[i] : 0.f, i + 1 < n ? src[i + 1] : 0.f,
                         i + 2 < n ? src[i + 2] : 0.f, i + 3 < n ? src[i + 3] : 0.f);
    }
  }
  for (int i = tid; i < kFineBins; i += NT) hist[i] = 0;      // while the loads fly
  __syncthreads();
  int nan_local = 0;
  auto put = [&](int i, float v) -> uint32_t {
    if (i >= n) return 0u;
    nan_local |= is_nan_bits(v);
    const uint32_t key = score_key(v);
    atomicAdd(&hist[key >> kFineShift], 1);
    return key;
  };
#pragma unroll
  for (int q = 0; q < kKpl / 4; ++q) {
    const int g = tid + q * NT;
    reinterpret_cast<uint4*>(keys)[g] =
        make_uint4(put(4 * g, f[q].x), put(4 * g + 1, f[q].y), put(4 * g + 2, f[q].z),
                   put(4 * g + 3, f[q].w));
  }
  if (__syncthreads_or(nan_local)) {
    if (tid == 0) set_err(a.err, SA_ERR_NAN);
    for (int i = tid; i < k; i += NT) out[i] = -1;
    return;
  }
  find_bin<NT>(hist, kFineBins, k, S);
  const uint32_t sel = (uint32_t)S.sel_bin;
  const int r = k - S.above;                     // 1 <= r <= keys in bin sel
  // ---- B. the bin's keys and indices; per-warp counts of keys above the bin
  const unsigned lt = lanemask_lt();
  const uint32_t* wkeys = keys + w * 32 * kKpl + lane;   // this lane's keys, stride 32
  const int i0 = w * 32 * kKpl + lane;
  int above_w = 0, in_w = 0;
  uint32_t mine = 0;                             // bit j: this lane's slot j is in bin sel
#pragma unroll 4
  for (int j = 0; j < kKpl; ++j) {
    const uint32_t key = wkeys[32 * j];
    const uint32_t hb = key >> kFineShift;       // slots past n: key 0, never above sel
    above_w += __popc(__ballot_sync(0xffffffffu, hb > sel));
    const bool in = key != 0u && hb == sel;
    in_w += __popc(__ballot_sync(0xffffffffu, in));
    mine |= (uint32_t)in << j;
  }
  if (lane == 0) { S.wg[w] = above_w; S.we[w] = 0; S.wc[w] = in_w; }
  __syncthreads();
  int cw = lane < NW ? S.wc[lane] : 0;           // list offset of this warp's bin keys
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, cw, o);
    if (lane >= o) cw += y;
  }
  const int c = __shfl_sync(0xffffffffu, cw, 31);
  int pos = w > 0 ? __shfl_sync(0xffffffffu, cw, w - 1) : 0;
  for (int j = 0; j < kKpl && __any_sync(0xffffffffu, mine >> j); ++j) {
    const bool in = (mine >> j) & 1u;
    const unsigned b = __ballot_sync(0xffffffffu, in);
    const int at = pos + __popc(b & lt);
    if (in && at < kCandMax) { ck[at] = wkeys[32 * j]; ci[at] = i0 + 32 * j; }
    pos += __popc(b);
  }
  __syncthreads();
  uint32_t T;
  int take;
  if (c <= kCandMax) {
    if (c <= kRankMax) {
      if (tid < c) {
        const uint32_t x = ck[tid];
        int gt = 0, eq = 0;
        for (int i = 0; i < c; ++i) {
          const uint32_t y = ck[i];
          gt += y > x;
          eq += y == x;
        }
        if (gt < r && r <= gt + eq) { S.T = x; S.take = r - gt; }   // equal x: equal writes
      }
      __syncthreads();
      T = S.T;
      take = S.take;
    } else {
      T = radix_select<NT>(ck, c, r, S, &take, 32 - kFineShift, sel << kFineShift);
    }
    for (int i = tid; i < c; i += NT) {          // the bin's share of the per-warp counts
      const int wi = ci[i] / (32 * kKpl);
      if (ck[i] > T) atomicAdd(&S.wg[wi], 1);
      else if (ck[i] == T) atomicAdd(&S.we[wi], 1);
    }
    __syncthreads();
  } else {                                       // the bin overflowed the list: whole row
    T = radix_select<NT>(keys, NT * kKpl, k, S, &take, 0, 0u);
    int g = 0, e = 0;
#pragma unroll 4
    for (int j = 0; j < kKpl; ++j) {
      const uint32_t key = wkeys[32 * j];
      g += __popc(__ballot_sync(0xffffffffu, key > T));
      e += __popc(__ballot_sync(0xffffffffu, key == T));
    }
    if (lane == 0) { S.wg[w] = g; S.we[w] = e; }
    __syncthreads();
  }
  // ---- C. emission in index order
  int incl = lane < NW ? (S.wg[lane] << 16) | S.we[lane] : 0;   // each count <= 32*kKpl
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  const int excl = __shfl_sync(0xffffffffu, incl, (w + 31) & 31);
  int g_run = w > 0 ? excl >> 16 : 0, e_run = w > 0 ? excl & 0xFFFF : 0;
#pragma unroll 4
  for (int j = 0; j < kKpl; ++j) {
    const uint32_t key = wkeys[32 * j];
    const bool is_gt = key > T, is_eq = key == T;
    const unsigned bg = __ballot_sync(0xffffffffu, is_gt);
    const unsigned be = __ballot_sync(0xffffffffu, is_eq);
    const int gb = g_run + __popc(bg & lt), eb = e_run + __popc(be & lt);
    if (is_gt) out[gb + min(eb, take)] = i0 + 32 * j;
    else if (is_eq && eb < take) out[gb + eb] = i0 + 32 * j;
    g_run += __popc(bg);
    e_run += __popc(be);
  }
}

bool topk_supported(int N_cap) { return N_cap <= kMaxChunk * kMaxCluster; }

cudaError_t launch_topk(const TopkArgs& a, int num_sms, cudaStream_t st) {
  if (a.rows <= 0) return cudaSuccess;
  if (a.N_cap <= kRowMax) {
    auto go = [&](auto kern, int nt) -> cudaError_t {
      const size_t smem = kTopkSmemBytes +
                          sizeof(uint32_t) * ((size_t)kFineBins + (size_t)nt * kKpl + 2 * kCandMax);
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)smem);
      if (e != cudaSuccess) return e;
      kern<<<(unsigned)a.rows, nt, smem, st>>>(a);
      return cudaGetLastError();
    };
    if (a.N_cap <= 256 * kKpl) return go(topk_row_kernel<256>, 256);
    if (a.N_cap <= 512 * kKpl) return go(topk_row_kernel<512>, 512);
    return go(topk_row_kernel<1024>, 1024);
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
