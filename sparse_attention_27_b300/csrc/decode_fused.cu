// Fused CSA decode: the whole CSA layer for each sequence's new token in one
// launch -- compression of the block the token closes, lightning-indexer
// scores, top-k, sparse attention over the selected compressed rows plus the
// sliding window, and the merge of the partial results.
//
// Source: "오픈소스 LLM의 새 이정표: DeepSeek-V4 시리즈", section
// "압축 희소 어텐션(CSA)과 극압축 어텐션(HCA)" (compress m entries into one, attend
// the top-k compressed entries plus a sliding window), "DeepSeek-V4 논문 읽기:
// 백만 토큰 컨텍스트를 저렴하게", section "Compressed Sparse Attention (CSA)" steps
// 1-4 and "KV Cache 관리: 저장 구조까지 변경" (compressed cache, sliding-window
// cache, uncompressed tail), "EP 95. DeepSeek-V4 논문 읽기 — 노정석", section
// IDEAS (lightning indexer, one shared KV head; kernels fused into one, the
// "mega-kernel" of the chapter list).
//
// One thread-block cluster of C CTAs per sequence (one query token each), one
// CTA per SM, 512 threads.  CTA r of the cluster owns a contiguous slice of
// the sequence's visible compressed entries (whole 128-entry tiles).  Phases:
//  1. scores: warp 0 streams the slice's indexer-key tiles by TMA through a
//     ring of 32 KB stages (two 128-entry tiles per copy: the copy engine's
//     cost is per request, so larger requests stream faster per SM); warp 1 issues tcgen05 MMAs D[j, h] =
//     Ik_c[j] . q_I[h] (M = 128 entries, N = 64 heads, K = 64) into six TMEM
//     accumulators; three warpgroups (warps 4-7, 8-11, 12-15; tiles
//     round-robin) fold ReLU and the head weights in fp32 and write each score
//     as an order-preserving 32-bit key into shared memory -- the scores never
//     go to global memory.  Warps 12-15 first pool the blocks this step
//     compresses (the block the new token closes) and write them to the
//     caches; the producer loads a tile holding such a block only after them.
//  2. top-k: the row's exact top-k over the cluster (topk_dev.cuh: a 13-bit
//     histogram summed over distributed shared memory, an exact select in
//     the k-th key's bin, emission in index order) into the idx output; each
//     CTA then reads its share of the key list back through L2.
//  3. attention: the key list (selected rows ascending, padded to a multiple
//     of 4, then the window) is cut into tiles of 64 keys, and CTA r attends
//     its contiguous share of the tiles: warps 12-15 gather K/V rows by 16-byte
//     cp.async into 128B-swizzled stages; warp 1 issues S = Q.K^T (M = 64
//     heads, N = 64 keys, K = 128) and O += P.V (N = 128, K = 64) into TMEM;
//     warps 4-7 run the online softmax (the running max raised only when it
//     grows by more than 32 in log2 units, then O rescaled in TMEM).
//  4. merge: each CTA leaves its normalised partial O (fp32) and LSE in
//     shared memory; after a cluster barrier CTA r merges heads
//     [r*64/C, (r+1)*64/C) from all C partials over distributed shared memory
//     and writes O and LSE.
// Every mbarrier wait is bounded (SA_ERR_DEVICE_TIMEOUT, then the CTA drops
// its remaining work); every thread of every CTA passes the same cluster
// barriers whatever happens, and the CTA frees its TMEM before it exits.
#include <cudaTypedefs.h>

#include "compress_dev.cuh"
#include "kernels.cuh"
#include "topk_dev.cuh"

namespace sa {

namespace {

constexpr int kThreads = 512;
constexpr int kTile = 128;                     // indexer entries per score tile (MMA M)
constexpr int kHI = 64, kDI = 64;              // indexer heads, indexer key width
constexpr int kD = 128;                        // head dim
constexpr int kHeads = 64;                     // attention MMA M
constexpr int kKeys = 64;                      // keys per attention tile
constexpr int kStageTiles = 2;                 // score tiles per stage (one TMA box of 256 rows)
constexpr int kTileBytes = kTile * kDI * 2;    // 16 KB: one score tile
constexpr int kABytes = kStageTiles * kTileBytes;   // 32 KB: one score stage
constexpr int kBBytes = kHI * kDI * 2;         // 8 KB: the row's indexer queries
constexpr int kQBytes = kHeads * kD * 2;       // 16 KB: the row's query heads
constexpr int kHalf = kKeys * 128;             // 8 KB: 64 dims of a K or V tile
constexpr int kKVBytes = 4 * kHalf;            // 32 KB: one K/V stage
constexpr int kPBytes = kHeads * kKeys * 2;    // 8 KB
constexpr int kEpiGroups = 3;                  // score epilogue warpgroups (tiles round-robin)
constexpr int kAcc = 6;                        // score accumulators (64 TMEM columns each)
constexpr int kTmemCols = 512;                 // score: 6 x 64; attention: S 2 x 64 + O 128
constexpr int kMaxStagesA = 6, kMaxStagesKV = 6;
constexpr int kMaxPool = 128;                  // largest block size m this kernel pools
constexpr float kRescaleThreshold = 32.f;      // log2 units

// warp roles
constexpr int kWarpTma = 0;                    // score tiles, B and Q loads
constexpr int kWarpMma = 1;                    // MMA issuer and TMEM owner
constexpr int kWarpEpi = 4;                    // score epilogue: warps 4-11
constexpr int kWarpSoft = 4;                   // softmax: warps 4-7
constexpr int kWarpAux = 12;                   // pooling, then K/V producers: warps 12-15
constexpr int kBarPool = 1;                    // named barrier of the pooling warps

struct Ctl {
  uint64_t a_full[kMaxStagesA], a_empty[kMaxStagesA];
  uint64_t b_full, q_full, fresh;
  uint64_t t_full[kAcc], t_empty[kAcc];
  uint64_t kv_full[kMaxStagesKV], kv_empty[kMaxStagesKV];
  uint64_t s_full[2], s_empty[2], p_full[2], p_empty[2];
  uint32_t tmem;
  int abort;
  uint32_t smax;                               // largest key of this CTA's first score tile
  uint32_t bin_lo;                             // the row's relative first-level bins (FineBins::lo)
  __align__(16) float w[kHI];                  // indexer head weights of the row
  float pw[kMaxPool];                          // pooling weights of one block
  float lse[kHeads];                           // this CTA's partial LSE
};
static_assert(offsetof(Ctl, w) % 16 == 0, "the epilogue reads w as float4");

struct TMaps {
  CUtensorMap ik;                              // [B*N_cap, 64] bf16, box 64 x 256
  CUtensorMap qi;                              // [B*64, 64] bf16, box 64 x 64
  CUtensorMap q;                               // [B*H, 128] bf16, box 64 x 64
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Byte offset of 16-byte chunk c (0..7) of 128-byte row r in a 1024-aligned
// block with the 128-byte swizzle.
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}

// The row's geometry, the same in every CTA of the cluster.
struct RowPlan {
  int b, p;
  int n;               // visible compressed entries
  int n_comp;          // selected entries: min(k, n)
  int n_comp_pad;      // rounded up to a multiple of 4
  int n_win;           // window rows
  bool all;            // n <= k (or k = 0): every visible entry is selected, no scoring
  int tpc;             // score tiles per CTA
  int qt;              // attention tiles per CTA
};

__device__ __forceinline__ RowPlan plan_row(const FusedDecodeArgs& a, int b) {
  RowPlan P;
  P.b = b;
  P.p = __ldg(a.q_pos + b);
  const int64_t nraw = P.p < 0 ? 0 : ((int64_t)P.p + 1) / a.m;
  P.n = (int)min64(nraw, a.N_cap);
  P.n_comp = min(a.k, P.n);
  P.n_comp_pad = (P.n_comp + 3) & ~3;
  P.n_win = P.p < 0 ? 0 : (int)min64(a.W, (int64_t)P.p + 1);
  P.all = P.n <= a.k || a.k == 0;
  const int ntiles = (P.n + kTile - 1) / kTile;
  P.tpc = (ntiles + a.C - 1) / a.C;
  const int ntl = (P.n_comp_pad + P.n_win + kKeys - 1) / kKeys;
  P.qt = (ntl + a.C - 1) / a.C;
  return P;
}

// Which CTA pools fresh block j: the owner of the score tile holding it, or
// the last CTA for a block outside the scored entries.
__device__ __forceinline__ int pool_owner(const RowPlan& P, int64_t j, int C) {
  if (P.all || j >= P.n) return C - 1;
  return (int)min64(C - 1, (j / kTile) / P.tpc);
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
    csa_decode_kernel(const __grid_constant__ TMaps tm, FusedDecodeArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  Ctl& C = *reinterpret_cast<Ctl*>(smem_raw);
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + sizeof(Ctl) + 1023) & ~uintptr_t(1023));
  unsigned char* sB = base;                                        // kBBytes
  unsigned char* sQ = sB + kBBytes;                                // kQBytes
  uint32_t* keys = reinterpret_cast<uint32_t*>(sQ + kQBytes);      // [a.cap]
  int32_t* sel = reinterpret_cast<int32_t*>(keys + a.cap);         // [a.selcap]
  unsigned char* X = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(sel + a.selcap) + 1023) & ~uintptr_t(1023));
  // region X, by phase: score stages | top-k scratch | K/V stages | partial O
  unsigned char* sA = X;
  int* hist = reinterpret_cast<int*>(X);                           // [kFineBins]
  uint32_t* ck = reinterpret_cast<uint32_t*>(X + 4 * kFineBins);   // [kCandMax]
  int32_t* ci = reinterpret_cast<int32_t*>(ck + kCandMax);         // [kCandMax]
  TopkSmem& TS = *reinterpret_cast<TopkSmem*>(ci + kCandMax);
  unsigned char* sKV = X;                                          // [stages_kv][kKVBytes]
  // the P tiles of the attention take the score keys' space, dead once the
  // top-k has passed its last cluster barrier
  unsigned char* sP = reinterpret_cast<unsigned char*>(keys);      // [2][kPBytes]
  float* sO = reinterpret_cast<float*>(X);                         // [64][128]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Cn = a.C;
  const int rank = Cn > 1 ? (int)cluster_rank() : 0;
  const int b = blockIdx.x / Cn;
  const RowPlan P = plan_row(a, b);
  volatile int* abort_flag = &C.abort;

  // this CTA's score tiles and entries
  const int ntiles = (P.n + kTile - 1) / kTile;
  const int t_lo = P.all ? 0 : min(ntiles, rank * P.tpc);
  const int t_hi = P.all ? 0 : min(ntiles, t_lo + P.tpc);
  const int lo = t_lo * kTile;
  const int cnt = max(0, min(P.n, t_hi * kTile) - lo);
  // this CTA's attention tiles of the key list
  const int ntl = (P.n_comp_pad + P.n_win + kKeys - 1) / kKeys;
  const int at_lo = min(ntl, rank * P.qt);
  const int nt_att = min(ntl, at_lo + P.qt) - at_lo;
  // the blocks this step pools: [blk_lo, blk_hi) of the sequence
  const int fb_lo = __ldg(a.blk_lo + b), fb_hi = __ldg(a.blk_hi + b);
  const bool fresh_ok = fb_hi - fb_lo <= a.max_blocks;
  int t_fresh = 0x7fffffff;                      // first score tile of this CTA holding one
  if (fresh_ok && a.m <= kMaxPool) {
    for (int j = max(fb_lo, 0); j < fb_hi && j < a.N_cap; ++j)
      if (pool_owner(P, j, Cn) == rank && j < P.n) t_fresh = min(t_fresh, j / kTile);
  }

  if (tid == 0) {
    for (int s = 0; s < a.stages_a; ++s) { mbar_init(&C.a_full[s], 1); mbar_init(&C.a_empty[s], 1); }
    mbar_init(&C.b_full, 1);
    mbar_init(&C.q_full, 1);
    mbar_init(&C.fresh, 128);
    for (int s = 0; s < kAcc; ++s) { mbar_init(&C.t_full[s], 1); mbar_init(&C.t_empty[s], 128); }
    for (int s = 0; s < a.stages_kv; ++s) {
      mbar_init(&C.kv_full[s], 32);
      mbar_init(&C.kv_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&C.s_full[s], 1);
      mbar_init(&C.s_empty[s], 128);
      mbar_init(&C.p_full[s], 128);
      mbar_init(&C.p_empty[s], 1);
    }
    C.abort = 0;
    C.smax = 0u;
    if (rank == 0) {
      if (P.p >= 0 && ((int64_t)P.p + 1) / a.m > a.N_cap) set_err(a.err, SA_ERR_BOUNDS);
      if (!fresh_ok || fb_lo < 0) set_err(a.err, SA_ERR_BOUNDS);
    }
    mbar_fence_init();
  }
  if (tid < kHI) C.w[tid] = __ldg(a.w + (int64_t)b * kHI + tid);
  // key slots past this CTA's scored tiles stay 0 (below every real key)
  for (int i = (t_hi - t_lo) * kTile + tid; i < a.cap; i += kThreads) keys[i] = 0u;
  if (warp == kWarpMma) tmem_alloc(&C.tmem, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = C.tmem;
  // The top-k bins its keys relative to the row's largest sampled key: the
  // first score tile of every CTA, published by the warpgroup that scores it.
  // The cluster exchanges the samples through one barrier whose arrive comes
  // early (the sampling warps right after their first tile, every other
  // thread now) and whose wait comes only before the histogram.
  const bool sample_x = Cn > 1 && !P.all;
  const bool sampler = warp >= kWarpEpi && warp < kWarpEpi + 4;   // epilogue group 0: tile 0
  if (sample_x && !sampler) cluster_arrive_release();

  if (warp == kWarpTma && lane == 0) {
    tma_prefetch_desc(&tm.ik);
    tma_prefetch_desc(&tm.qi);
    tma_prefetch_desc(&tm.q);
    mbar_arrive_expect_tx(&C.q_full, kQBytes);
    tma_load_2d(&tm.q, &C.q_full, sQ, 0, b * a.H);
    tma_load_2d(&tm.q, &C.q_full, sQ + kHeads * 128, 64, b * a.H);
    if (t_hi > t_lo) {
      mbar_arrive_expect_tx(&C.b_full, kBBytes);
      tma_load_2d(&tm.qi, &C.b_full, sB, 0, b * kHI);
    }
  }

  // ========================================================= 1. scores
  int nan_local = 0;
  const int nt_score = t_hi - t_lo;
  if (warp == kWarpTma) {
    if (lane == 0) {
      int issued = 0;
      bool waited_fresh = false;
      for (int t = t_lo; t < t_hi && !*abort_flag; t += kStageTiles, ++issued) {
        if (t + kStageTiles - 1 >= t_fresh && !waited_fresh) {   // pooled rows in memory first
          if (!mbar_wait(&C.fresh, 0, a.err)) { *abort_flag = 1; break; }
          waited_fresh = true;
        }
        const int st = issued % a.stages_a;
        const uint32_t ph = (uint32_t)((issued / a.stages_a) & 1);
        if (!mbar_wait(&C.a_empty[st], ph ^ 1, a.err)) { *abort_flag = 1; break; }
        mbar_arrive_expect_tx(&C.a_full[st], kABytes);
        tma_load_2d(&tm.ik, &C.a_full[st], sA + st * kABytes, 0,
                    (int32_t)((int64_t)b * a.N_cap + (int64_t)t * kTile));
      }
      // every issued copy has landed before region X is used for anything else
      for (int u = max(0, issued - a.stages_a); u < issued; ++u)
        mbar_wait(&C.a_full[u % a.stages_a], (uint32_t)((u / a.stages_a) & 1), a.err);
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    if (lane == 0 && nt_score > 0) {
      constexpr uint32_t idesc = idesc_bf16(kTile, kHI);
      bool ok = mbar_wait(&C.b_full, 0, a.err);
      const uint32_t b_base = smem_u32(sB);
      for (int o = 0; o < nt_score && ok && !*abort_flag; ++o) {
        const int u = o / kStageTiles, half = o % kStageTiles;   // stage, tile within it
        const int st = u % a.stages_a, acc = o % kAcc;
        if ((half == 0 && !mbar_wait(&C.a_full[st], (uint32_t)((u / a.stages_a) & 1), a.err)) ||
            !mbar_wait(&C.t_empty[acc], (uint32_t)(((o / kAcc) & 1) ^ 1), a.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a_base = smem_u32(sA + st * kABytes + half * kTileBytes);
#pragma unroll
        for (int kk = 0; kk < kDI / 16; ++kk)
          tc_mma_f16(tmem + acc * kHI, sdesc_kmajor_sw128(a_base + kk * 32),
                     sdesc_kmajor_sw128(b_base + kk * 32), idesc, kk > 0 ? 1u : 0u);
        tc_commit(&C.t_full[acc]);
        if (half == kStageTiles - 1 || o == nt_score - 1) tc_commit(&C.a_empty[st]);
      }
      if (!ok) *abort_flag = 1;
    }
    __syncwarp();
  }
  // The score epilogue of warpgroup grp (tiles o = grp (mod kEpiGroups));
  // warp w reads TMEM lanes 32*(w%4)..
  auto score_epilogue = [&](int grp) {
    const int quad = warp & 3;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const float4* w4 = reinterpret_cast<const float4*>(C.w);
    bool arrived = false;                        // the sampling warps' cluster arrive
    for (int o = grp; o < nt_score; o += kEpiGroups) {
      const int acc = o % kAcc;
      // warp-uniform: the TMEM loads below are warp-collective
      if (!__all_sync(0xffffffffu, !*abort_flag &&
                                       mbar_wait(&C.t_full[acc], (uint32_t)((o / kAcc) & 1), a.err))) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
      uint32_t v[64];
      tmem_ld32_async(tmem + lane_base + acc * kHI, v);
      tmem_ld32_async(tmem + lane_base + acc * kHI + 32, v + 32);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&C.t_empty[acc]);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float4 wv = w4[i];
        s0 = fmaf(wv.x, fmaxf(__uint_as_float(v[4 * i + 0]), 0.f), s0);
        s1 = fmaf(wv.y, fmaxf(__uint_as_float(v[4 * i + 1]), 0.f), s1);
        s2 = fmaf(wv.z, fmaxf(__uint_as_float(v[4 * i + 2]), 0.f), s2);
        s3 = fmaf(wv.w, fmaxf(__uint_as_float(v[4 * i + 3]), 0.f), s3);
      }
      const float s = (s0 + s1) + (s2 + s3);
      const int jl = o * kTile + quad * 32 + lane;          // slot in this CTA's keys
      const bool real = lo + jl < P.n;
      nan_local |= real && is_nan_bits(s);
      keys[jl] = real ? score_key(s) : 0u;
      if (o == 0) {                                         // the sample: tile 0, group 0
        if (real) atomicMax(&C.smax, score_key(s));
        if (sample_x) cluster_arrive_release();
        arrived = true;
      }
    }
    // no tile 0 here, or stopped before it: the arrive all the same, so that
    // every thread of the cluster passes the barrier
    if (grp == 0 && sample_x && !arrived) cluster_arrive_release();
  };
  if (warp >= kWarpEpi && warp < kWarpEpi + 8) {
    score_epilogue((warp - kWarpEpi) >> 2);
  } else if (warp >= kWarpAux) {
    // pool this CTA's share of the step's blocks (K, V and the indexer key),
    // then release the producer's wait on them
    const int t = tid - kWarpAux * 32;                       // 0..127
    const int ckv = kD / 8, cik = kDI / 8;                   // 16-byte chunks per row
    const int nchunks = 2 * ckv + cik;
    if (fresh_ok && a.m <= kMaxPool) {
      for (int j = max(fb_lo, 0); j < fb_hi; ++j) {
        if (pool_owner(P, j, Cn) != rank) continue;
        if (j >= a.N_cap) {
          if (t == 0) set_err(a.err, SA_ERR_BOUNDS);
          continue;
        }
        const int64_t p0 = (int64_t)j * a.m;
        if (t < 32) pool_weights_warp(a.z + (int64_t)b * a.R, p0, a.m, a.R, C.pw);
        named_bar_sync(kBarPool, 128);
        if (t < nchunks) {
          const char* src;
          char* dst;
          int width, off;
          if (t < ckv) {
            src = static_cast<const char*>(a.k_raw); dst = static_cast<char*>(a.k_c);
            width = kD; off = t * 8;
          } else if (t < 2 * ckv) {
            src = static_cast<const char*>(a.v_raw); dst = static_cast<char*>(a.v_c);
            width = kD; off = (t - ckv) * 8;
          } else {
            src = static_cast<const char*>(a.ik_raw); dst = static_cast<char*>(a.ik_c);
            width = kDI; off = (t - 2 * ckv) * 8;
          }
          src += (int64_t)b * a.R * width * 2;
          float acc[8];
          pool_chunk<SA_BF16>(src, (int64_t)width * 2, off * 2, p0, a.m, a.R, C.pw, acc);
          store_chunk<SA_BF16>(dst + (((int64_t)b * a.N_cap + j) * width + off) * 2, acc);
          // the score tile holding this row is read by TMA (the async proxy)
          asm volatile("fence.proxy.async;" ::: "memory");
        }
        named_bar_sync(kBarPool, 128);                     // before pw is reused
      }
    }
    mbar_arrive(&C.fresh);
    score_epilogue(2);                           // then the third epilogue warpgroup
  }
  tc_fence_before();
  nan_local = __syncthreads_or(nan_local);
  tc_fence_after();

  // ========================================================== 2. top-k
  const int k = a.k;
  int32_t* out_idx = a.idx + (int64_t)b * k;
  const int sel_lo = at_lo * kKeys;              // first list position this CTA attends
  if (!P.all) {
    if (sample_x) cluster_wait_acquire();         // every CTA's sample is in place
    if (tid == 0) {
      uint32_t mx = C.smax;
      for (int r = 0; r < Cn; ++r) mx = max(mx, Cn > 1 ? *peer(&C.smax, r) : mx);
      // 1024 bins per octave from 6 octaves below the sample's largest key to
      // 2 above it (no sample: the absolute bins)
      const uint32_t v = mx >> 13;
      C.bin_lo = mx == 0u ? 0xFFFFFFFFu : (v > 6u * 1024u ? v - 6u * 1024u : 0u);
    }
    for (int i = tid; i < kFineBins; i += kThreads) hist[i] = 0;
    __syncthreads();
    const FineBins fb = C.bin_lo == 0xFFFFFFFFu ? kAbsoluteBins : FineBins{13, C.bin_lo};
    for (int i = tid; i < cnt; i += kThreads) atomicAdd(&hist[fb.bin(keys[i])], 1);
    __syncthreads();
    auto emit = [&](int pos, int j) { out_idx[pos] = j; };
    if (a.cap == 8192)
      topk_select<kThreads, 16>(TS, keys, cnt, lo, hist, ck, ci, nan_local, k, Cn, rank, a.err,
                                emit, fb);
    else
      topk_select<kThreads, 32>(TS, keys, cnt, lo, hist, ck, ci, nan_local, k, Cn, rank, a.err,
                                emit, fb);
    // the selection is complete in global memory (topk_select ends with a
    // cluster barrier after the emission): this CTA's share of the key list,
    // read through L2 (other CTAs wrote it), padding slots -1
    for (int s = tid; s < P.qt * kKeys; s += kThreads) {
      const int pos = sel_lo + s;
      sel[s] = pos < P.n_comp ? __ldcg(out_idx + pos) : -1;
    }
    __syncthreads();
  } else {
    // every visible entry is selected, in order
    for (int i = rank * kThreads + tid; i < k; i += Cn * kThreads) out_idx[i] = i < P.n ? i : -1;
    for (int s = tid; s < P.qt * kKeys; s += kThreads) {
      const int pos = sel_lo + s;
      sel[s] = pos < P.n_comp ? pos : -1;
    }
    // the pooled rows (global memory, written by the pooling CTA) are visible
    // to every CTA of the cluster
    if (Cn > 1) cluster_sync(); else __syncthreads();
  }
  tc_fence_after();

  // ====================================================== 3. attention
  const int nprod = min(4, a.stages_kv);        // producer warps: at most one per stage
  if (warp >= kWarpAux) {
    const int pw_ = warp - kWarpAux;
    if (pw_ < nprod) {
      const __nv_bfloat16* kc = static_cast<const __nv_bfloat16*>(a.k_c);
      const __nv_bfloat16* vc = static_cast<const __nv_bfloat16*>(a.v_c);
      const __nv_bfloat16* kr = static_cast<const __nv_bfloat16*>(a.k_raw);
      const __nv_bfloat16* vr = static_cast<const __nv_bfloat16*>(a.v_raw);
      for (int n = pw_; n < nt_att; n += nprod) {
        if (*abort_flag) break;
        const int st = n % a.stages_kv;
        if (!mbar_wait(&C.kv_empty[st], (uint32_t)(((n / a.stages_kv) & 1) ^ 1), a.err)) {
          *abort_flag = 1;
          break;
        }
        unsigned char* stage = sKV + st * kKVBytes;
        const uint32_t kd = smem_u32(stage), vd = kd + 2 * kHalf;
        // lane l resolves the source rows of keys 2l and 2l+1 as (row << 1 | raw),
        // -1 for a key with no row (masked: zero-filled); then each cp.async
        // instruction copies two whole 256-byte rows (half-warp per key, one
        // 16-byte chunk per lane), four full lines per instruction
        int64_t src2[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int s = (at_lo + n) * kKeys + 2 * lane + q;   // list position
          int64_t code = -1;
          if (s < P.n_comp) {
            const int j = sel[s - sel_lo];
            if (j >= 0 && j < P.n) code = ((int64_t)b * a.N_cap + j) << 1;
            else if (j != -1) set_err(a.err, SA_ERR_BOUNDS);
          } else if (s >= P.n_comp_pad && s < P.n_comp_pad + P.n_win) {
            const int64_t u = (int64_t)P.p - P.n_win + 1 + (s - P.n_comp_pad);
            code = (((int64_t)b * a.R + u % a.R) << 1) | 1;
          }
          src2[q] = code;
        }
        const int hw = lane >> 4, ch = lane & 15;
#pragma unroll 4
        for (int pr = 0; pr < kKeys / 2; ++pr) {
          const int64_t c0 = __shfl_sync(0xffffffffu, src2[0], pr);
          const int64_t c1 = __shfl_sync(0xffffffffu, src2[1], pr);
          const int64_t code = hw ? c1 : c0;
          const int key = 2 * pr + hw;
          const bool raw = code >= 0 && (code & 1);
          const __nv_bfloat16* ks = raw ? kr : kc;
          const __nv_bfloat16* vs = raw ? vr : vc;
          const uint32_t bytes = code >= 0 ? 16u : 0u;
          const int64_t off = (code >= 0 ? (code >> 1) : 0) * kD + ch * 8;
          const uint32_t o = (ch >> 3) * kHalf + swz(key, ch & 7);
          cp_async16(kd + o, (code >= 0 ? ks : kr) + off, bytes);
          cp_async16(vd + o, (code >= 0 ? vs : vr) + off, bytes);
        }
        asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
        fence_proxy_async_smem();
        mbar_arrive(&C.kv_full[st]);
      }
      asm volatile("cp.async.wait_group 0;" ::: "memory");
    }
  } else if (warp == kWarpMma) {
    if (lane == 0 && nt_att > 0) {
      constexpr uint32_t idS = idesc_bf16(kHeads, kKeys, 0, 0);
      constexpr uint32_t idO = idesc_bf16(kHeads, kD, 0, 1);
      const uint32_t qa = smem_u32(sQ);
      bool ok = mbar_wait(&C.q_full, 0, a.err);
      auto pv = [&](int m_) -> bool {             // O += P(m_) . V(m_)
        const int pb = m_ & 1;
        if (!mbar_wait(&C.p_full[pb], (uint32_t)((m_ >> 1) & 1), a.err)) return false;
        tc_fence_after();
        const uint32_t pa = smem_u32(sP + pb * kPBytes);
        const uint32_t va = smem_u32(sKV + (m_ % a.stages_kv) * kKVBytes) + 2 * kHalf;
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk)
          tc_mma_f16(tmem + 128, sdesc_kmajor_sw128(pa + kk * 32),
                     sdesc_mnmajor_sw128(va + kk * 2048, kHalf, 1024), idO,
                     (m_ > 0 || kk > 0) ? 1u : 0u);
        tc_commit(&C.kv_empty[m_ % a.stages_kv]);
        tc_commit(&C.p_empty[pb]);
        return true;
      };
      for (int n = 0; n < nt_att && ok; ++n) {
        if (*abort_flag) { ok = false; break; }
        const int st = n % a.stages_kv, sb = n & 1;
        if (!mbar_wait(&C.kv_full[st], (uint32_t)((n / a.stages_kv) & 1), a.err) ||
            !mbar_wait(&C.s_empty[sb], (uint32_t)(((n >> 1) & 1) ^ 1), a.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t ka = smem_u32(sKV + st * kKVBytes);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
          tc_mma_f16(tmem + sb * 64,
                     sdesc_kmajor_sw128(qa + (kk >> 2) * (kHeads * 128) + (kk & 3) * 32),
                     sdesc_kmajor_sw128(ka + (kk >> 2) * kHalf + (kk & 3) * 32), idS,
                     kk > 0 ? 1u : 0u);
        tc_commit(&C.s_full[sb]);
        if (n > 0 && !pv(n - 1)) { ok = false; break; }
      }
      if (ok && !pv(nt_att - 1)) ok = false;
      if (!ok) *abort_flag = 1;
    }
    __syncwarp();
  } else if (warp >= kWarpSoft && warp < kWarpSoft + 4) {
    // S and O through the 16x256b TMEM shape: lane l holds heads h0 = 16q + l/4
    // and h1 = h0 + 8 (q = this warp's TMEM quarter), keys 8g + 2(l%4) and +1
    // of every 8-key group g
    const int quad = warp & 3;
    const int l4 = lane & 3;
    const int h0 = quad * 16 + (lane >> 2), h1 = h0 + 8;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const float c2 = a.sm_scale * 1.4426950408889634f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    bool ok = true;
    for (int n = 0; n < nt_att && ok; ++n) {
      // (before the wait for S) key i of the tile is real iff it is a selected
      // row naming a visible entry (a -1 from a rejected row is ignored) or a
      // window row.  Lane l tests keys 2l and 2l+1; two ballots give the
      // tile's even and odd keys, and this lane keeps the bits of its keys
      // 8g + 2(l%4) + j as bit 2g + j of keep16.
      const int s0 = (at_lo + n) * kKeys;
      const bool ok0 = h0 < a.H, ok1 = h1 < a.H;
      auto is_real = [&](int sk) -> bool {
        if (sk < P.n_comp) {
          const int jj = sel[sk - sel_lo];
          return jj >= 0 && jj < P.n;
        }
        return sk >= P.n_comp_pad && sk < P.n_comp_pad + P.n_win;
      };
      const uint32_t re = __ballot_sync(0xffffffffu, is_real(s0 + 2 * lane));
      const uint32_t ro = __ballot_sync(0xffffffffu, is_real(s0 + 2 * lane + 1));
      uint32_t keep16 = 0;
#pragma unroll
      for (int g = 0; g < 8; ++g)
        keep16 |= (((re >> (4 * g + l4)) & 1u) << (2 * g)) |
                  (((ro >> (4 * g + l4)) & 1u) << (2 * g + 1));
      const int sb = n & 1, pb = n & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(&C.s_full[sb], (uint32_t)((n >> 1) & 1), a.err));
      if (!ok) break;
      tc_fence_after();
      float v[32];
      {
        uint32_t r[32];
        tmem_ld16x256b_x8_async(tmem + lane_base + sb * 64, r);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
      }
      tc_fence_before();
      mbar_arrive(&C.s_empty[sb]);
      if (keep16 != 0xFFFFu || !ok0 || !ok1) {
#pragma unroll
        for (int g = 0; g < 8; ++g) {
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const bool keep = (keep16 >> (2 * g + j)) & 1u;
            if (!keep || !ok0) v[4 * g + j] = -INFINITY;
            if (!keep || !ok1) v[4 * g + 2 + j] = -INFINITY;
          }
        }
      }
      float x0 = -INFINITY, x1 = -INFINITY;
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        x0 = fmaxf(x0, fmaxf(v[4 * g], v[4 * g + 1]));
        x1 = fmaxf(x1, fmaxf(v[4 * g + 2], v[4 * g + 3]));
      }
      x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, 1));
      x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, 1));
      x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, 2));
      x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, 2));
      float al0 = 1.f, al1 = 1.f;
      bool need = false;
      auto raise = [&](float mt, float& m_, float& al) {
        if (mt > m_) {
          if (m_ == -INFINITY) {
            m_ = mt;
          } else if (mt > m_ + kRescaleThreshold) {
            al = fast_exp2(m_ - mt);
            m_ = mt;
            need = true;
          }
        }
      };
      raise(x0 * c2, m0, al0);
      raise(x1 * c2, m1, al1);
      if (__any_sync(0xffffffffu, need)) {
        // rescale O once PV(n-1) is done (it signals p_empty of its P buffer)
        ok = __all_sync(0xffffffffu, mbar_wait(&C.p_empty[(n - 1) & 1],
                                               (uint32_t)(((n - 1) >> 1) & 1), a.err));
        if (!ok) break;
        tc_fence_after();
        const uint32_t tO = tmem + lane_base + 128;
#pragma unroll 1
        for (int c = 0; c < kD; c += 32) {
          float o[16];
          tmem_ld16x256b_x4(tO + c, o);
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            o[4 * g] *= al0;
            o[4 * g + 1] *= al0;
            o[4 * g + 2] *= al1;
            o[4 * g + 3] *= al1;
          }
          tmem_st16x256b_x4(tO + c, o);
        }
        tmem_st_wait();
      }
      l0 *= al0;
      l1 *= al1;
      // P buffer pb is free once PV(n-2) is done
      ok = __all_sync(0xffffffffu,
                      mbar_wait(&C.p_empty[pb], (uint32_t)(((n >> 1) & 1) ^ 1), a.err));
      if (!ok) break;
      {
        unsigned char* prow = sP + pb * kPBytes + 4 * l4;
        const float r0 = m0 == -INFINITY ? 0.f : m0, r1 = m1 == -INFINITY ? 0.f : m1;
        float u0 = 0.f, u1 = 0.f;
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          const __nv_bfloat162 p0 = __floats2bfloat162_rn(fast_exp2(fmaf(v[4 * g], c2, -r0)),
                                                          fast_exp2(fmaf(v[4 * g + 1], c2, -r0)));
          const __nv_bfloat162 p1 = __floats2bfloat162_rn(fast_exp2(fmaf(v[4 * g + 2], c2, -r1)),
                                                          fast_exp2(fmaf(v[4 * g + 3], c2, -r1)));
          u0 += __low2float(p0) + __high2float(p0);
          u1 += __low2float(p1) + __high2float(p1);
          *reinterpret_cast<__nv_bfloat162*>(prow + swz(h0, g)) = p0;
          *reinterpret_cast<__nv_bfloat162*>(prow + swz(h1, g)) = p1;
        }
        l0 += u0;
        l1 += u1;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&C.p_full[pb]);
    }
    // ---- this CTA's partial: O = all PVs (the last one signals p_empty)
    if (ok && nt_att > 0)
      ok = __all_sync(0xffffffffu, mbar_wait(&C.p_empty[(nt_att - 1) & 1],
                                             (uint32_t)(((nt_att - 1) >> 1) & 1), a.err));
    if (!ok) *abort_flag = 1;
    tc_fence_after();
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    const bool have0 = ok && nt_att > 0 && l0 > 0.f, have1 = ok && nt_att > 0 && l1 > 0.f;
    const float inv0 = have0 ? 1.f / l0 : 0.f, inv1 = have1 ? 1.f / l1 : 0.f;
    // the partial goes to shared memory over the K/V stages, which no copy or
    // MMA touches any more (the last PV is complete)
    const uint32_t tO = tmem + lane_base + 128;
#pragma unroll 1
    for (int c = 0; c < kD; c += 32) {
      float o[16];
      if (nt_att > 0) {
        tmem_ld16x256b_x4(tO + c, o);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) o[i] = 0.f;
      }
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const int col = c + 8 * g + 2 * l4;
        *reinterpret_cast<float2*>(sO + h0 * kD + col) =
            make_float2(o[4 * g] * inv0, o[4 * g + 1] * inv0);
        *reinterpret_cast<float2*>(sO + h1 * kD + col) =
            make_float2(o[4 * g + 2] * inv1, o[4 * g + 3] * inv1);
      }
    }
    if (l4 == 0) {
      C.lse[h0] = have0 ? (m0 + log2f(l0)) * 0.6931471805599453f : -INFINITY;
      C.lse[h1] = have1 ? (m1 + log2f(l1)) * 0.6931471805599453f : -INFINITY;
    }
  }
  tc_fence_before();
  if (Cn > 1) cluster_sync(); else __syncthreads();   // every CTA's partial is final

  // ========================================================== 4. merge
  {
    const int hpc = kHeads / Cn;                 // heads merged by this CTA
    for (int it = tid; it < hpc * 32; it += kThreads) {
    const int hh = it >> 5, c4 = it & 31;        // head of this CTA's share, float4 column
    const int h = rank * hpc + hh;
    if (h < a.H) {
      float L[16];
      float mx = -INFINITY;
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        L[r] = -INFINITY;
        if (r < Cn) L[r] = Cn > 1 ? *peer(&C.lse[h], r) : C.lse[h];
        mx = fmaxf(mx, L[r]);
      }
      float lse_out = -INFINITY;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      if (mx != -INFINITY) {
        float sum = 0.f;
#pragma unroll
        for (int r = 0; r < 16; ++r)
          if (r < Cn) sum += expf(L[r] - mx);
        lse_out = mx + logf(sum);
        float4 v[16];
#pragma unroll
        for (int r = 0; r < 16; ++r)
          if (r < Cn)
            v[r] = Cn > 1 ? *peer(reinterpret_cast<const float4*>(sO + h * kD) + c4, r)
                          : reinterpret_cast<const float4*>(sO + h * kD)[c4];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          if (r < Cn) {
            const float wgt = L[r] == -INFINITY ? 0.f : expf(L[r] - lse_out);
            acc.x = fmaf(wgt, v[r].x, acc.x);
            acc.y = fmaf(wgt, v[r].y, acc.y);
            acc.z = fmaf(wgt, v[r].z, acc.z);
            acc.w = fmaf(wgt, v[r].w, acc.w);
          }
        }
      }
      const int64_t o0 = ((int64_t)b * a.H + h) * kD + 4 * c4;
      if (a.o_dtype == SA_BF16) {
        const __nv_bfloat162 lo2 = __floats2bfloat162_rn(acc.x, acc.y);
        const __nv_bfloat162 hi2 = __floats2bfloat162_rn(acc.z, acc.w);
        uint2 u;
        u.x = *reinterpret_cast<const uint32_t*>(&lo2);
        u.y = *reinterpret_cast<const uint32_t*>(&hi2);
        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.o) + o0) = u;
      } else {
        *reinterpret_cast<float4*>(static_cast<float*>(a.o) + o0) = acc;
      }
      if (c4 == 0) a.lse[(int64_t)b * a.H + h] = lse_out;
    }
    }
  }
  if (Cn > 1) cluster_sync();                    // peers have read this CTA's partial
  if (warp == kWarpTma && lane == 0) {           // no copy may still be landing at exit
    mbar_wait(&C.q_full, 0, a.err);
    if (t_hi > t_lo) mbar_wait(&C.b_full, 0, a.err);
  }
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------- host side

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* ptr = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// bf16 matrix [rows, cols] (cols * 2 bytes per row), box 64 columns x box_rows
// rows, 128-byte swizzle, zero fill out of range.
static bool tmap_bf16(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                      uint32_t box_rows) {
  auto enc = encode_fn();
  if (!enc || rows == 0) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Shared memory of one CTA for the given key capacity, list capacity and
// stage counts (the phases' scratch shares region X).
static size_t fused_smem(int cap, int selcap, int stages_a, int stages_kv) {
  const size_t fixed = round_up(sizeof(Ctl), 16) + 1024 + kBBytes + kQBytes +
                       4 * (size_t)cap + 4 * (size_t)selcap;
  const size_t topk = 4 * (size_t)kFineBins + 8 * (size_t)kCandMax + sizeof(TopkSmem);
  const size_t x = std::max(std::max((size_t)stages_a * kABytes, topk),
                            std::max((size_t)stages_kv * kKVBytes, (size_t)kHeads * kD * 4));
  return fixed + 1024 + x;
}

constexpr size_t kSmemMax = 232448;              // 227 KB per block on sm_100-class parts
static_assert(4 * 8192 >= 2 * kPBytes, "the P tiles fit the smallest key array");
static_assert((kBBytes + kQBytes) % 1024 == 0, "the P tiles start on a 1024-byte boundary");

bool fused_decode_plan(FusedDecodeArgs& a, int num_sms) {
  if (a.B <= 0) return false;
  const int ntiles = (a.N_cap + kTile - 1) / kTile;
  // cluster size: the fewest CTAs whose key space holds the row (16384 keys
  // per CTA at most), then doubled while the grid stays within one wave
  int C = 1;
  while (C < 16 && (int64_t)((ntiles + C - 1) / C) * kTile > 16384) C *= 2;
  if ((int64_t)((ntiles + C - 1) / C) * kTile > 16384) return false;
  while (C < 16 && (int64_t)a.B * 2 * C <= num_sms && (ntiles + 2 * C - 1) / (2 * C) >= 8)
    C *= 2;
  const int tpc = (ntiles + C - 1) / C;
  a.C = C;
  a.cap = tpc * kTile <= 8192 ? 8192 : 16384;
  const int ntl = ((std::min(a.k, a.N_cap) + 3) / 4 * 4 + a.W + kKeys - 1) / kKeys;
  a.selcap = std::max(1, (ntl + C - 1) / C) * kKeys;
  // stage counts: as many as fit
  int sa_ = kMaxStagesA, skv = kMaxStagesKV;
  while (sa_ > 2 && fused_smem(a.cap, a.selcap, sa_, 2) > kSmemMax) --sa_;
  while (skv > 2 && fused_smem(a.cap, a.selcap, 2, skv) > kSmemMax) --skv;
  a.stages_a = sa_;
  a.stages_kv = skv;
  return fused_smem(a.cap, a.selcap, sa_, skv) <= kSmemMax;
}

cudaError_t launch_fused_decode(const FusedDecodeArgs& a, cudaStream_t st) {
  TMaps tm;
  // with no compressed entries nothing is scored and the key map is never
  // used: it then describes the query rows instead, so that it still encodes
  const bool no_keys = (uint64_t)a.B * a.N_cap == 0;
  if (!tmap_bf16(&tm.ik, no_keys ? a.q_idx : a.ik_c,
                 no_keys ? (uint64_t)a.B * kHI : (uint64_t)a.B * a.N_cap, kDI,
                 kStageTiles * kTile) ||
      !tmap_bf16(&tm.qi, a.q_idx, (uint64_t)a.B * kHI, kDI, kHI) ||
      !tmap_bf16(&tm.q, a.q, (uint64_t)a.B * a.H, kD, kHeads))
    return cudaErrorInvalidValue;
  const size_t smem = fused_smem(a.cap, a.selcap, a.stages_a, a.stages_kv);
  cudaError_t e = cudaFuncSetAttribute(csa_decode_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if (a.C > 8) {
    e = cudaFuncSetAttribute(csa_decode_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return cudaErrorNotSupported;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(a.B * a.C));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = a.C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.C > 1 ? 1 : 0;
  if (a.C > 1) {
    int nclusters = 0;
    if (cudaOccupancyMaxActiveClusters(&nclusters, csa_decode_kernel, &cfg) != cudaSuccess ||
        nclusters <= 0) {
      cudaGetLastError();
      return cudaErrorNotSupported;
    }
  }
  return cudaLaunchKernelEx(&cfg, csa_decode_kernel, tm, a);
}

}  // namespace sa
