// Per-row exact top-k select over a thread-block cluster (device code shared
// by the stand-alone top-k kernel, topk.cu, and the fused decode kernel,
// decode_fused.cu).  Internal header.
//
// Source: "오픈소스 LLM의 새 이정표: DeepSeek-V4 시리즈", section
// "압축 희소 어텐션(CSA)과 극압축 어텐션(HCA)" (each query attends only its top-k
// compressed entries) and "DeepSeek-V4 논문 읽기: 백만 토큰 컨텍스트를 저렴하게",
// section "Compressed Sparse Attention (CSA)" step 3.  Ties go to the lower
// index and the output is in ascending index order (readings where the pages
// are silent).
//
// A row's candidates are split over a cluster of C CTAs (C = 1: one CTA per
// row), CTA r holding a contiguous slice as order-preserving 32-bit keys in
// shared memory, in index order.  Warp w of a CTA owns its keys
// [w*32*KPL, (w+1)*32*KPL) and reads them 32 at a time (key w*32*KPL + 32j + l
// in lane l, bank-conflict free), so a ballot over one j lists keys in index
// order.  Three steps over the CTA's keys:
//  A. a histogram of their top 13 bits (sign, exponent, 4 mantissa bits: 8192
//     bins, one atomic per key; or a relative map of 1024 bins per octave, see
//     FineBins), summed over the cluster through distributed shared memory,
//     gives the bin holding the row's k-th largest key;
//  B. each CTA lists its keys in that bin with their indices and counts, per
//     warp, its keys in higher bins; every CTA then copies all the cluster's
//     lists into one and finds the exact k-th largest T in it (rank counting
//     for a few keys, radix passes over the 19 low bits otherwise).  If a list
//     overflows (a heavily tied row), T comes instead from radix passes whose
//     histograms are summed over the cluster, and the counts from a full pass;
//  C. emission in index order: out[#(> T) before i + min(#(== T) before i, take)],
//     the counts of lower-ranked CTAs included.
#pragma once
#include <type_traits>

#include "common.cuh"

namespace sa {

constexpr int kTopkWarpsMax = 32;          // warps of the largest CTA (1024 threads)
constexpr int kBins = 2048;                // radix pass histogram (11 bits)

struct TopkSmem {
  int hist[2][kBins];
  int scan[kTopkWarpsMax + 1];
  __align__(8) int cnt[2];                // this CTA: keys > T, keys == T
  int nan_flag;
  int wg[kTopkWarpsMax], we[kTopkWarpsMax];   // per-warp keys > T, keys == T
  int wc[kTopkWarpsMax];                  // per-warp keys in the selected bin
  int gsum[64];                           // the 13-bit histogram in 64 groups
  int sel_bin, above;
  int take;                               // keys equal to T that are kept
  uint32_t T;                             // the k-th largest key
  uint32_t kmax;                          // this CTA's largest key (relative bins)
};

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

constexpr int kKplMax = 32;                                // keys per thread of the top-k kernels
                                                           // (topk_select itself takes up to 64)
constexpr int kTopkSmemBytes = (sizeof(TopkSmem) + 15) & ~15;
constexpr int kFineShift = 19;                             // bin = key >> 19
constexpr int kFineBins = 1 << (32 - kFineShift);          // 8192
constexpr int kCandMax = 4096;                             // listed keys of one bin
constexpr int kRankMax = 256;
constexpr int kRowsMaxCluster = 16;

// The first-level bins of a row's keys, kFineBins of them, monotone in the
// key.  Absolute (shift 19, lo 0): bin = the key's top 13 bits.  Relative
// (shift 13): bin = (key >> 13) - lo, the values at or below lo in bin 0 and
// those at or above lo + kFineBins - 1 in the last bin -- 1024 bins per octave
// of the score over a window of 8 octaves placed by the caller.  A bin's keys
// share their top `top` bits (prefix), which the exact select then leaves
// alone; the two end bins of the relative map share none.
struct FineBins {
  int shift;
  uint32_t lo;
  __device__ __forceinline__ uint32_t bin(uint32_t key) const {
    const uint32_t v = key >> shift;
    return v <= lo ? 0u : min(v - lo, (uint32_t)(kFineBins - 1));
  }
  __device__ __forceinline__ bool clamped(uint32_t b) const {
    return shift != kFineShift && (b == 0 || b == (uint32_t)(kFineBins - 1));
  }
  __device__ __forceinline__ int top(uint32_t b) const { return clamped(b) ? 0 : 32 - shift; }
  __device__ __forceinline__ uint32_t prefix(uint32_t b) const {
    return clamped(b) ? 0u : (lo + b) << shift;
  }
};
constexpr FineBins kAbsoluteBins{kFineShift, 0u};

// Sum of v over the CTA, returned to every thread.
template <int NT>
__device__ __forceinline__ int block_sum_nt(int v, int* scratch) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane == 0) scratch[w] = v;
  __syncthreads();
  int t = lane < NT / 32 ? scratch[lane] : 0;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
  __syncthreads();
  return t;
}

// The same shared-memory object in CTA r of this cluster.
template <typename T>
__device__ __forceinline__ const T* peer(const T* p, int r) {
  return static_cast<const T*>(__cluster_map_shared_rank((void*)p, (unsigned)r));
}

// Count of bin b summed over the C CTAs of the cluster (C = 1: this CTA); the
// C loads are independent and issued together.
__device__ __forceinline__ int bin_count(const int* h, int b, int C) {
  if (C == 1) return h[b];
  int v[kRowsMaxCluster];
#pragma unroll
  for (int r = 0; r < kRowsMaxCluster; ++r) v[r] = r < C ? peer(h, r)[b] : 0;
  int s = 0;
#pragma unroll
  for (int r = 0; r < kRowsMaxCluster; ++r) s += v[r];
  return s;
}

// Over the histogram h[0..nb) summed over the cluster's C CTAs (higher bin =
// larger keys): the bin b where the count of keys in bins >= b first reaches
// krem (1 <= krem <= total), and the count of keys in bins > b, to
// S.sel_bin / S.above.  Synchronises the CTA.
template <int NT>
__device__ void find_bin(const int* h, int nb, int krem, TopkSmem& S, int C) {
  constexpr int NW = NT / 32;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int per = (nb + NT - 1) / NT;            // bins per thread, highest first
  const int top = nb - tid * per;                // this thread's bins: [top - per, top)
  const bool vec8 = C > 1 && per == 8;           // 8 bins from every CTA: two 16-byte loads each
  int loc[8] = {0, 0, 0, 0, 0, 0, 0, 0};         // vec8: counts of bins top-1 .. top-8
  int sum = 0;
  if (!vec8) {
    for (int q = 0; q < per; ++q)
      if (top - 1 - q >= 0) sum += bin_count(h, top - 1 - q, C);
  } else {
    int4 u[kRowsMaxCluster], v[kRowsMaxCluster];
#pragma unroll
    for (int r = 0; r < kRowsMaxCluster; ++r) {
      if (r < C) {
        const int4* p4 = reinterpret_cast<const int4*>(peer(h, r) + top - 8);
        u[r] = p4[0];
        v[r] = p4[1];
      } else {
        u[r] = v[r] = make_int4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int r = 0; r < kRowsMaxCluster; ++r) {
      loc[0] += v[r].w; loc[1] += v[r].z; loc[2] += v[r].y; loc[3] += v[r].x;
      loc[4] += u[r].w; loc[5] += u[r].z; loc[6] += u[r].y; loc[7] += u[r].x;
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) sum += loc[q];
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
  if (sum > 0 && base < krem && base + sum >= krem) {   // the one thread holding the bin
    if (vec8) {
      bool done = false;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (!done && base + loc[q] >= krem) { S.sel_bin = top - 1 - q; S.above = base; done = true; }
        base += loc[q];
      }
    } else {
      for (int q = 0; q < per; ++q) {
        const int c = bin_count(h, top - 1 - q, C);
        if (base + c >= krem) { S.sel_bin = top - 1 - q; S.above = base; break; }
        base += c;
      }
    }
  }
  __syncthreads();
}

// find_bin for the 8192-bin histogram summed over a cluster of C > 1 CTAs,
// in two steps that read little of the peers' shared memory: the 64 group
// sums of 128 bins (gsum, written by every CTA before the cluster barrier)
// give the group holding the krem-th largest key, then only that group's 128
// bins are read from each CTA.  One warp works; synchronises the CTA.
__device__ __forceinline__ void find_bin_cluster(const int* h, const int* gsum, int krem, TopkSmem& S, int C) {
  const int tid = threadIdx.x, lane = tid & 31;
  if (tid < 32) {
    int g0 = 0, g1 = 0;                          // groups 63 - 2l and 62 - 2l, over the cluster
    {
      int a[kRowsMaxCluster], b[kRowsMaxCluster];
#pragma unroll
      for (int r = 0; r < kRowsMaxCluster; ++r) {
        a[r] = r < C ? peer(gsum, r)[63 - 2 * lane] : 0;
        b[r] = r < C ? peer(gsum, r)[62 - 2 * lane] : 0;
      }
#pragma unroll
      for (int r = 0; r < kRowsMaxCluster; ++r) { g0 += a[r]; g1 += b[r]; }
    }
    int x = g0 + g1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    int base = x - g0 - g1, G = -1, aboveG = 0;
    if (base < krem && base + g0 >= krem) { G = 63 - 2 * lane; aboveG = base; }
    else if (base + g0 < krem && base + g0 + g1 >= krem) { G = 62 - 2 * lane; aboveG = base + g0; }
    const int src = __ffs(__ballot_sync(0xffffffffu, G >= 0)) - 1;
    G = __shfl_sync(0xffffffffu, G, src);
    aboveG = __shfl_sync(0xffffffffu, aboveG, src);
    // bins G*128 + 127 - 4l - q (q < 4) of every CTA: one 16-byte load each
    int c4[4] = {0, 0, 0, 0};
    {
      int4 v[kRowsMaxCluster];
#pragma unroll
      for (int r = 0; r < kRowsMaxCluster; ++r)
        v[r] = r < C ? *reinterpret_cast<const int4*>(peer(h, r) + G * 128 + 124 - 4 * lane)
                     : make_int4(0, 0, 0, 0);
#pragma unroll
      for (int r = 0; r < kRowsMaxCluster; ++r) {
        c4[0] += v[r].w; c4[1] += v[r].z; c4[2] += v[r].y; c4[3] += v[r].x;
      }
    }
    int s2 = c4[0] + c4[1] + c4[2] + c4[3];
    int x2 = s2;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x2, o);
      if (lane >= o) x2 += y;
    }
    int b2 = aboveG + x2 - s2, bin = -1, above = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (bin < 0 && b2 < krem && b2 + c4[q] >= krem) { bin = G * 128 + 127 - 4 * lane - q; above = b2; }
      b2 += c4[q];
    }
    if (bin >= 0) { S.sel_bin = bin; S.above = above; }
  }
  __syncthreads();
}

// find_bin over one CTA's own 8192-bin histogram h (shared memory) in two
// steps: the 64 group sums of 128 bins (each warp sums whole groups with
// 16-byte loads), then one warp finds the group holding the krem-th largest
// key and the bin inside it.  S.sel_bin, S.above as find_bin; synchronises
// the CTA.
template <int NT>
__device__ void find_bin_groups(const int* h, int krem, TopkSmem& S) {
  constexpr int NW = NT / 32;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  for (int g = w; g < 64; g += NW) {
    const int4 v = reinterpret_cast<const int4*>(h + g * 128)[lane];
    int s = v.x + v.y + v.z + v.w;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) S.gsum[g] = s;
  }
  __syncthreads();
  if (w == 0) {
    const int g0 = S.gsum[63 - 2 * lane], g1 = S.gsum[62 - 2 * lane];   // descending groups
    int x = g0 + g1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    const int base = x - g0 - g1;
    int G = -1, aboveG = 0;
    if (base < krem && base + g0 >= krem) { G = 63 - 2 * lane; aboveG = base; }
    else if (base + g0 < krem && base + g0 + g1 >= krem) { G = 62 - 2 * lane; aboveG = base + g0; }
    const int src = __ffs(__ballot_sync(0xffffffffu, G >= 0)) - 1;
    G = __shfl_sync(0xffffffffu, G, src);
    aboveG = __shfl_sync(0xffffffffu, aboveG, src);
    // bins G*128 + 127 - 4l - q (q < 4): one 16-byte load per lane
    const int4 v = *reinterpret_cast<const int4*>(h + G * 128 + 124 - 4 * lane);
    const int c4[4] = {v.w, v.z, v.y, v.x};
    const int s2 = c4[0] + c4[1] + c4[2] + c4[3];
    int x2 = s2;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x2, o);
      if (lane >= o) x2 += y;
    }
    int b2 = aboveG + x2 - s2, bin = -1, above = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (bin < 0 && b2 < krem && b2 + c4[q] >= krem) { bin = G * 128 + 127 - 4 * lane - q; above = b2; }
      b2 += c4[q];
    }
    if (bin >= 0) { S.sel_bin = bin; S.above = above; }
  }
  __syncthreads();
}

// The kk-th largest of those keys[0..m) whose top `top` bits equal prefix0's
// (1 <= kk <= their count over the cluster), by radix passes of up to 11 bits
// over the bits below, the per-pass histograms summed over the cluster's C
// CTAs; *take = how many keys equal to it belong to the top kk.  In a
// cluster every CTA must call it with the same top and prefix0.
template <int NT>
__device__ uint32_t radix_select(const uint32_t* keys, int m, int kk, TopkSmem& S, int* take,
                                 int top, uint32_t prefix0, int C) {
  const int tid = threadIdx.x;
  uint32_t prefix = prefix0, maskbits = top > 0 ? (~0u << (32 - top)) : 0u;
  int krem = kk;
  int low = 32 - top;                            // bits still open
  for (int pass = 0; low > 0; ++pass) {
    const int nbits = min(11, low);
    const int shift = low - nbits;
    const int nb = 1 << nbits;
    int* h = S.hist[pass & 1];                   // alternate: peers may still read the last one
    for (int i = tid; i < nb; i += NT) h[i] = 0;
    __syncthreads();
    for (int i = tid; i < m; i += NT) {
      const uint32_t key = keys[i];                // 0: an empty slot, never a real key
      if (key != 0u && (key & maskbits) == prefix)
        atomicAdd(&h[(key >> shift) & (uint32_t)(nb - 1)], 1);
    }
    if (C > 1) cluster_sync(); else __syncthreads();
    find_bin<NT>(h, nb, krem, S, C);
    krem -= S.above;
    prefix |= (uint32_t)S.sel_bin << shift;
    maskbits |= (uint32_t)(nb - 1) << shift;
    low = shift;
    __syncthreads();
  }
  *take = krem;
  return prefix;
}

// The selection of one row, after its candidates' keys and their 13-bit
// histogram are built: steps A (the cluster's bin search) to C (emission) of
// the description above.  keys: this CTA's CAP = NT * KPL key slots (slot i =
// candidate lo + i; slots at or past cnt hold key 0); hist: [kFineBins], its
// space reused for the union lists uk/ui ([kCandMax] each); ck/ci: this CTA's
// list ([kCandMax] each); nan_local: this thread saw a NaN candidate.
// emit(pos, j) writes candidate j at output position pos (pos < k); a
// rejected row (a NaN anywhere in the cluster) gets emit(pos, -1) for every
// pos, spread over the cluster.  Every CTA of the cluster calls it; it
// synchronises the CTA and the cluster.  Requires 1 <= k < the row's count.
template <int NT, int KPL, class Emit>
__device__ void topk_select(TopkSmem& S, const uint32_t* keys, int cnt, int lo, int* hist,
                            uint32_t* ck, int32_t* ci, int nan_local, int k, int C, int rank,
                            int32_t* err, Emit emit, const FineBins fb = kAbsoluteBins) {
  constexpr int NW = NT / 32;
  constexpr int CAP = NT * KPL;                  // key slots of this CTA
  uint32_t* uk = reinterpret_cast<uint32_t*>(hist);                 // [kCandMax] union keys
  int32_t* ui = reinterpret_cast<int32_t*>(uk + kCandMax);          // [kCandMax] union indices
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  auto csync = [&]() { if (C > 1) cluster_sync(); else __syncthreads(); };
  if (tid == 0) S.nan_flag = nan_local;
  if (C > 1) {                                   // group sums of 128 bins for the peers
    for (int g = w; g < 64; g += NW) {
      const int4 v = reinterpret_cast<const int4*>(hist + g * 128)[lane];
      int s = v.x + v.y + v.z + v.w;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      if (lane == 0) S.gsum[g] = s;
    }
  }
  csync();                                       // every CTA's histogram and flag are final
  int any_nan = nan_local;
  if (C > 1) any_nan = __any_sync(0xffffffffu, lane < C && *peer(&S.nan_flag, lane) != 0);
  if (any_nan) {                                 // reject the row: all -1
    if (rank == 0 && tid == 0) set_err(err, SA_ERR_NAN);
    for (int i = rank * NT + tid; i < k; i += C * NT) emit(i, -1);
    if (C > 1) cluster_sync();                   // peers may still read our flag
    return;
  }
  if (C > 1) find_bin_cluster(hist, S.gsum, k, S, C);
  else find_bin<NT>(hist, kFineBins, k, S, 1);
  const uint32_t sel = (uint32_t)S.sel_bin;
  const int r1 = k - S.above;                    // 1 <= r1 <= keys of the row in bin sel
  // ---- B. this CTA's keys in bin sel (list) and per-warp counts above it
  const unsigned lt = lanemask_lt();
  const uint32_t* wkeys = keys + w * 32 * KPL + lane;   // this lane's keys, stride 32
  const int i0 = w * 32 * KPL + lane;
  int above_w = 0, in_w = 0;
  using Mask = typename std::conditional<(KPL > 32), uint64_t, uint32_t>::type;
  Mask mine = 0;                                 // bit j: this lane's slot j is in bin sel
#pragma unroll 4
  for (int j = 0; j < KPL; ++j) {
    const uint32_t key = wkeys[32 * j];
    const uint32_t hb = fb.bin(key);             // empty slots: key 0, never above sel
    above_w += __popc(__ballot_sync(0xffffffffu, hb > sel));
    const bool in = key != 0u && hb == sel;
    in_w += __popc(__ballot_sync(0xffffffffu, in));
    mine |= (Mask)in << j;
  }
  if (lane == 0) { S.wg[w] = above_w; S.we[w] = 0; S.wc[w] = in_w; }
  __syncthreads();
  int cw = lane < NW ? S.wc[lane] : 0;           // list offset of this warp's keys
  int aw = lane < NW ? S.wg[lane] : 0;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, cw, o);
    const int z = __shfl_up_sync(0xffffffffu, aw, o);
    if (lane >= o) { cw += y; aw += z; }
  }
  const int c_mine = __shfl_sync(0xffffffffu, cw, 31);
  const int a_mine = __shfl_sync(0xffffffffu, aw, 31);
  if (tid == 0) { S.cnt[0] = a_mine; S.cnt[1] = c_mine; }
  int pos = w > 0 ? __shfl_sync(0xffffffffu, cw, w - 1) : 0;
  for (int j = 0; j < KPL && __any_sync(0xffffffffu, (mine >> j) != 0); ++j) {
    const bool in = (mine >> j) & 1u;
    const unsigned b = __ballot_sync(0xffffffffu, in);
    const int at = pos + __popc(b & lt);
    if (in && at < kCandMax) { ck[at] = wkeys[32 * j]; ci[at] = lo + i0 + 32 * j; }
    pos += __popc(b);
  }
  __syncthreads();
  csync();                                       // lists and counts final; hists no longer read
  // list sizes and above-counts of the cluster: lane r of every warp reads
  // CTA r's, and shuffles give the prefix sums (every CTA gets the same)
  int cr = 0, ar = 0;
  if (lane < C) {
    const int* rc = C > 1 ? peer(S.cnt, lane) : S.cnt;
    ar = rc[0];
    cr = rc[1];
  }
  int cs = cr, as = ar;                          // inclusive over the ranks
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, cs, o), z = __shfl_up_sync(0xffffffffu, as, o);
    if (lane >= o) { cs += y; as += z; }
  }
  const int c_all = __shfl_sync(0xffffffffu, cs, 31);
  const bool overflow = __any_sync(0xffffffffu, cr > kCandMax) || c_all > kCandMax;
  int offr[kRowsMaxCluster];                     // where CTA r's list starts in the union
#pragma unroll
  for (int r = 0; r < kRowsMaxCluster; ++r) offr[r] = __shfl_sync(0xffffffffu, cs - cr, r);
  const int off_mine = __shfl_sync(0xffffffffu, cs - cr, rank);
  const int above_before = __shfl_sync(0xffffffffu, as - ar, rank);
  uint32_t T;
  int take, gt_before = above_before, eq_before = 0;
  if (!overflow) {
    // the union of the lists, rank by rank (index order is not needed here)
    for (int i = tid; i < c_all; i += NT) {
      int r = 0, base = 0;
#pragma unroll
      for (int q = 1; q < kRowsMaxCluster; ++q)
        if (q < C && i >= offr[q]) { r = q; base = offr[q]; }
      uk[i] = C > 1 ? peer(ck, r)[i - base] : ck[i];
      ui[i] = C > 1 ? peer(ci, r)[i - base] : ci[i];
    }
    __syncthreads();
    if (c_all <= kRankMax) {
      if (tid < c_all) {
        const uint32_t x = uk[tid];
        int gt = 0, eq = 0;
        for (int i = 0; i < c_all; ++i) {
          const uint32_t y = uk[i];
          gt += y > x;
          eq += y == x;
        }
        if (gt < r1 && r1 <= gt + eq) { S.T = x; S.take = r1 - gt; }   // equal x: equal writes
      }
      __syncthreads();
      T = S.T;
      take = S.take;
    } else {
      T = radix_select<NT>(uk, c_all, r1, S, &take, fb.top(sel), fb.prefix(sel), 1);
    }
    // the union's share of the counts: per warp of this CTA, and before it
    int gb = 0, eb = 0;
    for (int i = tid; i < c_all; i += NT) {
      const uint32_t x = uk[i];
      const int idx = ui[i];
      if (i >= off_mine && i < off_mine + c_mine) {
        const int wi = (idx - lo) / (32 * KPL);
        if (x > T) atomicAdd(&S.wg[wi], 1);
        else if (x == T) atomicAdd(&S.we[wi], 1);
      } else if (i < off_mine) {
        gb += x > T;
        eb += x == T;
      }
    }
    const int both = block_sum_nt<NT>((gb << 16) | eb, S.scan);   // each <= kCandMax
    gt_before += both >> 16;
    eq_before += both & 0xFFFF;
    __syncthreads();
  } else {                                       // heavily tied: cluster-wide radix passes
    // over every key of the row: within an end bin of a relative map (no
    // shared prefix) the bin's r1-th largest is the row's k-th largest
    T = radix_select<NT>(keys, CAP, fb.clamped(sel) ? k : r1, S, &take, fb.top(sel),
                         fb.prefix(sel), C);
    int g = 0, e = 0;
#pragma unroll 4
    for (int j = 0; j < KPL; ++j) {
      const uint32_t key = wkeys[32 * j];
      g += __popc(__ballot_sync(0xffffffffu, key > T));
      e += __popc(__ballot_sync(0xffffffffu, key == T));
    }
    if (lane == 0) { S.wg[w] = g; S.we[w] = e; }
    __syncthreads();
    if (C > 1) {
      int gs = lane < NW ? S.wg[lane] : 0, es = lane < NW ? S.we[lane] : 0;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        gs += __shfl_xor_sync(0xffffffffu, gs, o);
        es += __shfl_xor_sync(0xffffffffu, es, o);
      }
      if (tid == 0) { S.cnt[0] = gs; S.cnt[1] = es; }   // peers read cnt only after this sync
      cluster_sync();
      const int gr = lane < rank ? peer(S.cnt, lane)[0] : 0;
      const int er = lane < rank ? peer(S.cnt, lane)[1] : 0;
      gt_before = gr;
      eq_before = er;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        gt_before += __shfl_xor_sync(0xffffffffu, gt_before, o);
        eq_before += __shfl_xor_sync(0xffffffffu, eq_before, o);
      }
    } else {
      gt_before = 0;
    }
  }
  // ---- C. emission in index order
  int incl = lane < NW ? (S.wg[lane] << 16) | S.we[lane] : 0;   // each count <= 32*KPL
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  const int excl = __shfl_sync(0xffffffffu, incl, (w + 31) & 31);
  int g_run = gt_before + (w > 0 ? excl >> 16 : 0);
  int e_run = eq_before + (w > 0 ? excl & 0xFFFF : 0);
#pragma unroll 4
  for (int j = 0; j < KPL; ++j) {
    const uint32_t key = wkeys[32 * j];
    const bool is_gt = key > T, is_eq = key == T;
    const unsigned bg = __ballot_sync(0xffffffffu, is_gt);
    const unsigned be = __ballot_sync(0xffffffffu, is_eq);
    const int gb = g_run + __popc(bg & lt), eb = e_run + __popc(be & lt);
    if (is_gt) emit(gb + min(eb, take), lo + i0 + 32 * j);
    else if (is_eq && eb < take) emit(gb + eb, lo + i0 + 32 * j);
    g_run += __popc(bg);
    e_run += __popc(be);
  }
  if (C > 1) cluster_sync();                     // peers may still read our lists and counts
}

}  // namespace sa
