// The whole hybrid decode step -- both layers, CSA and HCA, for every
// sequence's new token -- as one persistent launch over a queue of work items.
//
// Source: "오픈소스 LLM의 새 이정표: DeepSeek-V4 시리즈", section
// "압축 희소 어텐션(CSA)과 극압축 어텐션(HCA)" (CSA: compress m entries into one,
// attend the top-k compressed entries plus a sliding window; HCA: compress
// m' >> m entries into one and attend all of them densely, plus the window),
// "DeepSeek-V4 논문 읽기: 백만 토큰 컨텍스트를 저렴하게", sections "Compressed
// Sparse Attention (CSA)" steps 1-4, "Heavily Compressed Attention (HCA)" and
// "KV Cache 관리: 저장 구조까지 변경", and "EP 95. DeepSeek-V4 논문 읽기 — 노정석",
// section IDEAS (lightning indexer; kernels fused into one "mega-kernel").
//
// One CTA of 512 threads per SM, launched once per step.  CTAs take work
// items from four queues (see "the queues" below) until none is left.  Item
// kinds, per sequence b:
//   POOL(b)     pool the CSA block(s) and the HCA block(s) the token closes
//               (compress_dev.cuh: the same fp32 order as csa_compress);
//   SCORE(b,u)  tcgen05 indexer scores of 32 tiles of 128 entries (TMA stages
//               of two tiles, six TMEM accumulators, three epilogue
//               warpgroups), written as order-preserving keys to a workspace
//               row; consecutive SCORE items stream through one pipeline;
//   TOPKA(b,r)  slice r of the row's exact top-k: from the row's 13-bit score
//               histogram (summed by the SCORE items) the bin of the k-th
//               largest key; the slice's keys in that bin listed, the keys
//               above it counted;
//   TOPKB(b,r)  once every TOPKA(b, *) is done: the exact k-th largest key from
//               the lists, then the slice's selected entries written to their
//               places in the idx output (ascending index order);
//   CSA(b,z)    sparse attention over a contiguous share of the key list
//               (selected rows, then the window): cp.async row gathers, QK^T
//               and PV on tcgen05, online softmax; a normalised partial O and
//               LSE to the workspace; the last share to finish merges them
//               into O and LSE;
//   HCA(b,z)    the same over all compressed HCA rows plus the window.
// Dependencies (release/acquire counters in the workspace):
//   SCORE(b, tile holding a block pooled this step) after POOL(b);
//   TOPKA(b, *) after POOL(b) and every SCORE(b, *); TOPKB(b, *) after every
//   TOPKA(b, *); CSA(b, *) after every TOPKB(b, *); HCA(b, *) after POOL(b).
// While later rows are scored, the top-k and attention of earlier rows run
// on other SMs as soon as their inputs are ready.
// Every wait (mbarrier or counter) is bounded: on a timeout the CTA records
// SA_ERR_DEVICE_TIMEOUT, raises the workspace abort flag, and every CTA stops
// taking items.
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
constexpr int kTileBytes = kTile * kDI * 2;    // 16 KB
constexpr int kABytes = kStageTiles * kTileBytes;   // 32 KB
constexpr int kBBytes = kHI * kDI * 2;         // 8 KB: one sequence's indexer queries
constexpr int kQBytes = kHeads * kD * 2;       // 16 KB
constexpr int kHalf = kKeys * 128;             // 8 KB: 64 dims of a K or V tile
constexpr int kKVBytes = 4 * kHalf;            // 32 KB: one K/V stage
constexpr int kPBytes = kHeads * kKeys * 2;    // 8 KB
constexpr int kEpiGroups = 3;
constexpr int kAcc = 6;
constexpr int kTmemCols = 512;
constexpr int kStagesA = 6, kStagesKV = 5;
constexpr int kProducers = 4;                  // K/V gather warps (12-15)
constexpr int kMaxPool = 128;                  // largest block size pooled
constexpr int kTopkKpl = 64;                   // keys per thread: rows of up to 32768 entries
constexpr int kKeyCap = kThreads * kTopkKpl;
constexpr int kMaxParts = 16;                  // attention shares per sequence and layer
constexpr int kRing = 4;                       // item slots between the claiming warp and the rest
constexpr float kRescaleThreshold = 32.f;

constexpr int kWarpTma = 0, kWarpMma = 1, kWarpEpi = 4, kWarpSoft = 4, kWarpProd = 12;

enum ItemKind : int { kStop = 0, kPool = 1, kScore = 2, kTopkA = 3, kCsa = 4, kHca = 5, kTopkB = 6 };
constexpr int kSlices = 4;                     // top-k slices of a row (kKeyCap / kSlices entries)
constexpr int kSliceKeys = kKeyCap / kSlices;  // 8192
constexpr int kSliceKpt = kSliceKeys / kThreads;   // 16 keys per thread
constexpr int kCandSlice = 4096;               // listed candidates of one slice
constexpr int kInfo = 16;                      // row info ints: sel, r1, overflow, -, then per slice (above, listed)

// workspace counters (int32): [0] next item, [1] abort, then per sequence
constexpr int kCtrHead = 32;
enum CtrArray : int { kPoolDone = 0, kScoreDone, kNan, kTopkADone, kTopkDone, kCsaParts, kHcaParts,
                     kNumCtr };

struct Ctl {
  uint64_t it_full[kRing], it_empty[kRing];
  uint64_t a_full[kStagesA], a_empty[kStagesA];
  uint64_t b_full[2], b_empty[2];
  uint64_t t_full[kAcc], t_empty[kAcc];
  uint64_t kv_full[kStagesKV], kv_empty[kStagesKV];
  uint64_t s_full[2], s_empty[2], p_full[2], p_empty[2];
  uint64_t q_full;
  int4 ring[kRing];
  uint32_t tmem;
  int abort;
  int bcast;
  __align__(16) float pw[2][kMaxPool];          // pooling weights of two blocks
  __align__(16) float wgt[kEpiGroups][kHI];    // head weights of each epilogue group's item
};
static_assert(offsetof(Ctl, wgt) % 16 == 0, "the epilogue reads wgt as float4");
static_assert((kHI * sizeof(float)) % 16 == 0, "each group's weights start 16-byte aligned");

struct TMaps {
  CUtensorMap ik;                              // [B*N_cap, 64] bf16, box 64 x 256
  CUtensorMap qi;                              // [B*64, 64] bf16, box 64 x 64
  CUtensorMap q;                               // [B*H, 128] bf16, box 64 x 64
  CUtensorMap qh;                              // the HCA queries, same shape
  CUtensorMap hk, hv;                          // HCA caches [B*N2_cap, 128] bf16, box 64 x 64
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
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}
__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_add(int* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int atom_acq_rel_add(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v)
               : "memory");
  return old;
}

// Score-key rows are N_cap rounded up to 4 keys apart (16-byte aligned rows).
__host__ __device__ __forceinline__ int64_t key_stride(int N_cap) { return (N_cap + 3) & ~3; }

// Per-row 13-bit score histograms [B][8192] and top-k row info [B][kInfo]
// follow the counters (all zeroed by the launch).
__host__ __device__ __forceinline__ int64_t ctr_ints(int B) {
  return ((int64_t)kCtrHead + (int64_t)kNumCtr * B + 63) / 64 * 64;
}
__device__ __forceinline__ int* hist_of(const StepArgs& a, int b) {
  return a.ctr + ctr_ints(a.B) + (int64_t)b * kFineBins;
}
__device__ __forceinline__ int* info_of(const StepArgs& a, int b) {
  return a.ctr + ctr_ints(a.B) + (int64_t)a.B * kFineBins + (int64_t)b * kInfo;
}

__device__ __forceinline__ int* ctr_of(const StepArgs& a, int which, int b) {
  return a.ctr + kCtrHead + which * a.B + b;
}
__device__ __forceinline__ bool aborted(const StepArgs& a) {
  return *reinterpret_cast<volatile const int*>(a.ctr + 1) != 0;
}
__device__ __forceinline__ void raise_abort(const StepArgs& a) {
  atomicExch(a.ctr + 1, 1);
}

// Wait until *p >= target (acquire).  Gives up on the abort flag or after
// kWaitLimitNs (SA_ERR_DEVICE_TIMEOUT, abort raised).
__device__ bool wait_ge(const StepArgs& a, const int* p, int target) {
  if (ld_acquire(p) >= target) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
    __nanosleep(64);
    if (ld_acquire(p) >= target) return true;
    if (aborted(a)) return false;
    if (global_ns() - t0 > kWaitLimitNs) {
      set_err(a.err, SA_ERR_DEVICE_TIMEOUT);
      raise_abort(a);
      return false;
    }
  }
}

// ------------------------------------------------------------ the queues
// Four queues, each a counter in the workspace: the independent items (the
// POOL items, then every sequence's SCORE items in sequence order, then the
// HCA items) and three dependent queues (sequence, then slice or share): CSA,
// TOPKB and TOPKA, in that priority.  A CTA takes the highest-priority
// dependent head whose dependencies are done, else the next independent item;
// only when no independent item is left does it take the next dependent item
// ready or not (TOPKA, then TOPKB, then CSA) and wait for its dependencies.
// Nothing waits forever: SCORE and HCA items wait only for POOL items, which
// come first in their queue and wait for nothing; a TOPKA item is taken
// unready only once every independent item is taken, a TOPKB item only once
// every TOPKA item is, a CSA item only once every TOPKB item is -- each by a
// running CTA that finishes its earlier items first.
enum Queue : int { kQInd = 0, kQTopkA = 2, kQTopkB = 3, kQCsa = 4 };   // counter slots (1: abort)

__device__ __forceinline__ int ld_volatile(const int* p) {
  return *reinterpret_cast<volatile const int*>(p);
}
// Independent item i: POOL(i < B), SCORE(b, u), HCA(b, z).  .w: an id unique
// over all queues.
__device__ __forceinline__ int4 independent_item(const StepArgs& a, int i) {
  if (i < a.B) return make_int4(kPool, i, 0, i);
  const int s0 = i - a.B;
  if (s0 < a.B * a.ns) return make_int4(kScore, s0 / a.ns, s0 % a.ns, i);
  const int h0 = s0 - a.B * a.ns;
  return make_int4(kHca, h0 / a.nh, h0 % a.nh, i);
}
__device__ __forceinline__ int n_independent(const StepArgs& a) {
  return a.B * (1 + a.ns + a.nh);
}
// Queue q's item h as (kind, sequence, part, id).
__device__ __forceinline__ int4 dependent_item(const StepArgs& a, int q, int h) {
  const int nind = n_independent(a), nt = a.B * kSlices;
  if (q == kQTopkA) return make_int4(kTopkA, h / kSlices, h % kSlices, nind + h);
  if (q == kQTopkB) return make_int4(kTopkB, h / kSlices, h % kSlices, nind + nt + h);
  return make_int4(kCsa, h / a.na, h % a.na, nind + 2 * nt + h);
}
__device__ int4 claim_item(const StepArgs& a) {
  const int nind = n_independent(a);
  constexpr int kNq = 3;                         // dependent queues, highest priority first
  const int qs[kNq] = {kQCsa, kQTopkB, kQTopkA};
  const int lens[kNq] = {a.B * a.na, a.B * kSlices, a.B * kSlices};
  const int per[kNq] = {max(a.na, 1), kSlices, kSlices};
  // ready dependent items first.  Each try costs two memory round trips:
  // the queue heads together, then the flags their items wait for
  for (int tries = 0; tries < 4; ++tries) {
    int h[kNq];
#pragma unroll
    for (int u = 0; u < kNq; ++u) h[u] = ld_volatile(a.ctr + qs[u]);
    bool ready[kNq];
#pragma unroll
    for (int u = 0; u < kNq; ++u) {
      ready[u] = false;
      if (h[u] >= lens[u]) continue;
      const int b = h[u] / per[u];
      if (u == 0) ready[u] = ld_acquire(a.ctr + kCtrHead + kTopkDone * a.B + b) >= kSlices;
      else if (u == 1) ready[u] = ld_acquire(a.ctr + kCtrHead + kTopkADone * a.B + b) >= kSlices;
      else ready[u] = ld_acquire(a.ctr + kCtrHead + kPoolDone * a.B + b) >= 1 &&
                      ld_acquire(a.ctr + kCtrHead + kScoreDone * a.B + b) >= kEpiGroups * a.ns;
    }
    int u = 0;
    while (u < kNq && !ready[u]) ++u;
    if (u == kNq) break;
    if (atomicCAS(a.ctr + qs[u], h[u], h[u] + 1) == h[u]) return dependent_item(a, qs[u], h[u]);
  }
  int i = atomicAdd(a.ctr + kQInd, 1);
  if (i < nind) return independent_item(a, i);
  // no independent work left: the next dependent item, ready or not, in
  // dependency order of the queues
  for (int u = kNq - 1; u >= 0; --u) {
    i = atomicAdd(a.ctr + qs[u], 1);
    if (i < lens[u]) return dependent_item(a, qs[u], i);
  }
  return make_int4(kStop, 0, 0, 0);
}

// ----------------------------------------------------- row geometry
__device__ __forceinline__ int visible(int p, int m, int cap) {
  return p < 0 ? 0 : (int)min64(((int64_t)p + 1) / m, cap);
}

// One sequence's score item: tiles [t0, t1) of its visible entries.
struct ScoreGeom {
  int b, n, t0, t1;
  bool all;                                      // every visible entry selected: no scoring
};
__device__ __forceinline__ ScoreGeom score_geom(const StepArgs& a, int b, int u) {
  ScoreGeom G;
  G.b = b;
  const int p = __ldg(a.q_pos + b);
  G.n = visible(p, a.m, a.N_cap);
  G.all = G.n <= a.k || a.k == 0;
  const int ntiles = (G.n + kTile - 1) / kTile;
  G.t0 = min(ntiles, u * a.tps);
  G.t1 = G.all ? G.t0 : min(ntiles, G.t0 + a.tps);
  return G;
}

// One attention item: key-list tiles [t_lo, t_lo + nt) of one layer's row.
struct AttGeom {
  int b, p, z;
  int nvis, n_comp, n_comp_pad, n_win;
  int t_lo, nt;
  bool gather;                                   // CSA: list slots from idx
};
__device__ __forceinline__ AttGeom att_geom(const StepArgs& a, int b, int z, bool csa) {
  AttGeom G;
  G.b = b;
  G.z = z;
  G.p = __ldg(a.q_pos + b);
  G.gather = csa;
  G.nvis = csa ? visible(G.p, a.m, a.N_cap) : visible(G.p, a.m2, a.N2_cap);
  G.n_comp = csa ? min(a.k, G.nvis) : G.nvis;
  G.n_comp_pad = (G.n_comp + 3) & ~3;
  G.n_win = G.p < 0 ? 0 : (int)min64(a.W, (int64_t)G.p + 1);
  const int ntl = (G.n_comp_pad + G.n_win + kKeys - 1) / kKeys;
  const int tp = csa ? a.tpa : a.tph;
  G.t_lo = min(ntl, z * tp);
  G.nt = min(ntl, G.t_lo + tp) - G.t_lo;
  return G;
}

// Running counts of pipeline uses, so that mbarrier phases continue across
// items.  Each warp keeps its own copy; all copies advance identically.
struct Counters {
  int s_items;                                   // non-empty SCORE items (B buffer uses)
  int stages;                                    // score stages
  int tiles;                                     // score tiles
  int att_items;                                 // attention items (Q loads)
  int att_tiles;                                 // attention tiles
};

// One block to pool: sequence b, block j of a layer whose cache rows are cut
// into 16-byte chunks over n arrays (src raw ring [B, R, width], dst cache
// [B, cap, width], bf16), pooling logits z_b (the sequence's ring), block size m.
struct PoolJob {
  const char* src[3];
  char* dst[3];
  int width[3];
  int n, nch;                                    // arrays; 16-byte chunks per row over them
  int64_t j;
  int cap, m;
  const float* z_b;
};

__device__ __forceinline__ void job_chunk(const PoolJob& J, int c, int& q, int& off) {
  q = 0;
  while (c >= J.width[q] / 8) { c -= J.width[q] / 8; ++q; }
  off = c * 8;                                   // channel offset in array q
}

// POOL(b): the CSA block(s) and the HCA block(s) sequence b's token closes,
// two blocks at a time.  The blocks' raw rows are staged in shared memory by
// cp.async (one round trip) while one warp per block computes the weights;
// then thread (block, chunk c, row group g) computes partial g of chunk c
// from shared memory and the RG = min(m, 8) partials are added in order --
// the evaluation order of compress_dev.cuh, so the rows equal csa_compress's
// bit for bit.  Out of line: its registers do not count against the kernel's
// pipelines.
__device__ __noinline__ void pool_item(const StepArgs& a, Ctl& C, unsigned char* X, int b) {
  const int tid = threadIdx.x, warp = tid >> 5;
  const int fb_lo = __ldg(a.blk_lo + b), fb_hi = __ldg(a.blk_hi + b);
  const int hb_lo = __ldg(a.hblk_lo + b), hb_hi = __ldg(a.hblk_hi + b);
  const bool f_ok = fb_hi - fb_lo <= a.max_blocks && fb_lo >= 0;
  const bool h_ok = hb_hi - hb_lo <= a.max_blocks2 && hb_lo >= 0;
  if (tid == 0 && (!f_ok || !h_ok)) set_err(a.err, SA_ERR_BOUNDS);
  const int nf = f_ok ? max(0, fb_hi - fb_lo) : 0, nh = h_ok ? max(0, hb_hi - hb_lo) : 0;
  auto make_job = [&](int t, PoolJob& J) -> bool {        // job t: CSA blocks, then HCA blocks
    if (t < nf) {
      J.j = fb_lo + t; J.cap = a.N_cap; J.m = a.m; J.z_b = a.z + (int64_t)b * a.R;
      J.src[0] = static_cast<const char*>(a.k_raw); J.dst[0] = static_cast<char*>(a.k_c);
      J.src[1] = static_cast<const char*>(a.v_raw); J.dst[1] = static_cast<char*>(a.v_c);
      J.src[2] = static_cast<const char*>(a.ik_raw); J.dst[2] = static_cast<char*>(a.ik_c);
      J.width[0] = kD; J.width[1] = kD; J.width[2] = kDI; J.n = 3;
    } else {
      J.j = hb_lo + (t - nf); J.cap = a.N2_cap; J.m = a.m2; J.z_b = a.hz + (int64_t)b * a.R;
      J.src[0] = static_cast<const char*>(a.hk_raw); J.dst[0] = static_cast<char*>(a.hk_c);
      J.src[1] = static_cast<const char*>(a.hv_raw); J.dst[1] = static_cast<char*>(a.hv_c);
      J.src[2] = nullptr; J.dst[2] = nullptr;
      J.width[0] = kD; J.width[1] = kD; J.width[2] = 0; J.n = 2;
    }
    J.nch = 0;
    for (int q = 0; q < J.n; ++q) J.nch += J.width[q] / 8;
    if (J.j >= J.cap) {
      if (tid == 0) set_err(a.err, SA_ERR_BOUNDS);
      return false;
    }
    return true;
  };
  // shared memory: staged rows of two blocks (m x nch x 16 bytes each, at
  // most 128 x 40 x 16), then the partial sums (8 x 40 x 8 floats each)
  constexpr int kStageMax = kMaxPool * 40 * 16;
  constexpr int kPartMax = 8 * 40 * 8;
  for (int t0 = 0; t0 < nf + nh; t0 += 2) {
    PoolJob J[2];
    bool live[2];
    for (int u = 0; u < 2; ++u) live[u] = t0 + u < nf + nh && make_job(t0 + u, J[u]);
    // stage the raw rows
    for (int u = 0; u < 2; ++u) {
      if (!live[u]) continue;
      const PoolJob& P = J[u];
      const int64_t p0 = P.j * P.m;
      const uint32_t st = smem_u32(X + u * kStageMax);
      for (int e = tid; e < P.m * P.nch; e += kThreads) {
        const int i = e / P.nch, c = e % P.nch;
        int q, off;
        job_chunk(P, c, q, off);
        const char* src = P.src[q] + (((int64_t)b * a.R + (p0 + i) % a.R) * P.width[q] + off) * 2;
        cp_async16(st + (uint32_t)e * 16, src, 16);
      }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    if (warp < 2 && live[warp])                  // meanwhile: each block's weights
      pool_weights_warp(J[warp].z_b, J[warp].j * J[warp].m, J[warp].m, a.R, C.pw[warp]);
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncthreads();
    // partials
    float* part = reinterpret_cast<float*>(X + 2 * kStageMax);
    const int tasks0 = live[0] ? J[0].nch * pool_groups(J[0].m) : 0;
    const int tasks1 = live[1] ? J[1].nch * pool_groups(J[1].m) : 0;
    for (int t = tid; t < tasks0 + tasks1; t += kThreads) {
      const int u = t < tasks0 ? 0 : 1;
      const int tt = u ? t - tasks0 : t;
      const PoolJob& P = J[u];
      const int RG = pool_groups(P.m);
      const int c = tt % P.nch, g = tt / P.nch;
      const unsigned char* stg = X + u * kStageMax;
      float acc[8];
      pool_partial_by<8, 2>(
          [&](int i, float* f) {
            bf16x8_to_f32(*reinterpret_cast<const uint4*>(stg + (i * P.nch + c) * 16), f);
          },
          P.m, C.pw[u], g, RG, acc);
#pragma unroll
      for (int e = 0; e < 8; ++e) part[u * kPartMax + (g * P.nch + c) * 8 + e] = acc[e];
    }
    __syncthreads();
    // the partials of each chunk added in order, stored
    const int n0 = live[0] ? J[0].nch : 0, n1 = live[1] ? J[1].nch : 0;
    for (int t = tid; t < n0 + n1; t += kThreads) {
      const int u = t < n0 ? 0 : 1;
      const int c = u ? t - n0 : t;
      const PoolJob& P = J[u];
      const int RG = pool_groups(P.m);
      const float* pp = part + u * kPartMax;
      float acc[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = pp[c * 8 + e];
      for (int g = 1; g < RG; ++g)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] += pp[(g * P.nch + c) * 8 + e];
      int q, off;
      job_chunk(P, c, q, off);
      store_chunk<SA_BF16>(P.dst[q] + (((int64_t)b * P.cap + P.j) * P.width[q] + off) * 2, acc);
      // cache rows may be read by TMA (the async proxy) on other SMs
      asm volatile("fence.proxy.async;" ::: "memory");
    }
    __syncthreads();                             // staging, weights and partials free again
  }
  __syncthreads();
  if (tid == 0) red_release_add(ctr_of(a, kPoolDone, b), 1);
}

// The exact top-k of a row (the selection of topk_dev.cuh: the k largest
// keys, ties to the lower index, emitted in ascending index order), over
// kSlices slices of kSliceKeys entries, from the row's keys and 13-bit
// histogram in L2 (both written by its SCORE items), in two item kinds:
//   TOPKA(b, r): the histogram gives the bin `sel` of the k-th largest key
//     and the count of keys above it; slice r lists its keys in bin sel (in
//     index order) and counts its keys above the bin, into the workspace;
//   TOPKB(b, r), once every TOPKA(b, *) is done: the exact k-th largest T
//     (and how many keys equal to T are taken) from the union of the lists;
//     the slices before r give, from their counts and lists, how many of
//     their keys are > T and == T; slice r then emits each of its selected
//     keys at its position out[#(> T) before i + min(#(== T) before i, take)].
// Thread t holds 16 consecutive entries of the slice in registers.  A slice
// whose bin holds more than kCandSlice keys (a heavily tied row) sets the
// row's overflow flag, and every TOPKB of that row then takes T from radix
// passes over all the row's keys instead.
struct TopkRow {
  int p, n, k;
  bool all;                                      // n <= k or k == 0: every visible entry
};
__device__ __forceinline__ TopkRow topk_row(const StepArgs& a, int b) {
  TopkRow R;
  R.p = __ldg(a.q_pos + b);
  R.n = visible(R.p, a.m, a.N_cap);
  R.k = a.k;
  R.all = R.n <= R.k || R.k == 0;
  return R;
}
// This thread's 16 keys of slice r (entries at or past n: key 0).
__device__ __forceinline__ void slice_keys(const StepArgs& a, int b, int r, int n,
                                           uint32_t* kr) {
  const int i0 = r * kSliceKeys + kSliceKpt * threadIdx.x;
  const uint4* src = reinterpret_cast<const uint4*>(a.keys + (int64_t)b * key_stride(a.N_cap) + i0);
  uint4 v[kSliceKpt / 4];
#pragma unroll
  for (int u = 0; u < kSliceKpt / 4; ++u)
    v[u] = i0 + 4 * u < n ? __ldcg(src + u) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
  for (int u = 0; u < kSliceKpt / 4; ++u) {
    kr[4 * u + 0] = i0 + 4 * u + 0 < n ? v[u].x : 0u;
    kr[4 * u + 1] = i0 + 4 * u + 1 < n ? v[u].y : 0u;
    kr[4 * u + 2] = i0 + 4 * u + 2 < n ? v[u].z : 0u;
    kr[4 * u + 3] = i0 + 4 * u + 3 < n ? v[u].w : 0u;
  }
}

__device__ __noinline__ void topka_item(const StepArgs& a, Ctl& C, unsigned char* X, int b, int r) {
  const int tid = threadIdx.x;
  volatile int* abort_flag = &C.abort;
  int* hist = reinterpret_cast<int*>(X);                             // [8192]
  TopkSmem& S = *reinterpret_cast<TopkSmem*>(hist + kFineBins);
  if (tid == 0) {
    int ok = !*abort_flag;
    if (ok) ok = wait_ge(a, ctr_of(a, kPoolDone, b), 1);
    if (ok) ok = wait_ge(a, ctr_of(a, kScoreDone, b), kEpiGroups * a.ns);
    if (!ok) *abort_flag = 1;
    C.bcast = ok;
  }
  __syncthreads();
  const bool ok = C.bcast != 0;
  const TopkRow R = topk_row(a, b);
  const bool nan_any = __ldcg(ctr_of(a, kNan, b)) != 0;
  if (ok && !R.all && !nan_any) {
    // the row's histogram and this thread's keys: one round trip
    const int4* hrow4 = reinterpret_cast<const int4*>(hist_of(a, b));
    int4 hv[kFineBins / 4 / kThreads];
#pragma unroll
    for (int u = 0; u < kFineBins / 4 / kThreads; ++u) hv[u] = __ldcg(hrow4 + u * kThreads + tid);
    uint32_t kr[kSliceKpt];
    slice_keys(a, b, r, R.n, kr);
#pragma unroll
    for (int u = 0; u < kFineBins / 4 / kThreads; ++u)
      reinterpret_cast<int4*>(hist)[u * kThreads + tid] = hv[u];
    __syncthreads();
    find_bin_groups<kThreads>(hist, R.k, S);
    const uint32_t sel = (uint32_t)S.sel_bin;
    int in_t = 0, above_t = 0;
#pragma unroll
    for (int j = 0; j < kSliceKpt; ++j) {
      const uint32_t hb = kr[j] >> kFineShift;
      in_t += kr[j] != 0u && hb == sel;
      above_t += hb > sel;                     // key 0 (no entry) is never above
    }
    int listed = 0;
    int off = block_exclusive_scan<kThreads>(in_t, S.scan, &listed);
    const int above_r = block_sum_nt<kThreads>(above_t, S.scan);
    uint32_t* cand = a.tk_cand + ((int64_t)b * kSlices + r) * kCandSlice;
    if (in_t > 0) {
#pragma unroll
      for (int j = 0; j < kSliceKpt; ++j)
        if (kr[j] != 0u && (kr[j] >> kFineShift) == sel) {
          if (off < kCandSlice) cand[off] = kr[j];
          ++off;
        }
    }
    if (tid == 0) {
      int* info = info_of(a, b);
      info[4 + 2 * r] = above_r;
      info[5 + 2 * r] = listed;
      if (listed > kCandSlice) atomicOr(info + 2, 1);
      if (r == 0) { info[0] = (int)sel; info[1] = R.k - S.above; }
    }
  }
  __syncthreads();
  if (tid == 0 && ok) red_release_add(ctr_of(a, kTopkADone, b), 1);
}

__device__ __noinline__ void topkb_item(const StepArgs& a, Ctl& C, unsigned char* X, int b, int r) {
  const int tid = threadIdx.x;
  volatile int* abort_flag = &C.abort;
  uint32_t* uk = reinterpret_cast<uint32_t*>(X);                    // [kSlices * kCandSlice] or [kKeyCap]
  TopkSmem& S = *reinterpret_cast<TopkSmem*>(uk + kKeyCap);
  if (tid == 0) {
    int ok = !*abort_flag;
    if (ok) ok = wait_ge(a, ctr_of(a, kTopkADone, b), kSlices);
    if (!ok) *abort_flag = 1;
    C.bcast = ok;
  }
  __syncthreads();
  const bool ok = C.bcast != 0;
  const TopkRow R = topk_row(a, b);
  int32_t* out_idx = a.idx + (int64_t)b * R.k;
  const bool nan_any = __ldcg(ctr_of(a, kNan, b)) != 0;
  const int q_lo = r * ((R.k + kSlices - 1) / kSlices);
  const int q_hi = min(R.k, q_lo + (R.k + kSlices - 1) / kSlices);
  if (tid == 0 && r == 0 && R.p >= 0 && ((int64_t)R.p + 1) / a.m > a.N_cap)
    set_err(a.err, SA_ERR_BOUNDS);
  if (ok && R.all) {
    for (int i = q_lo + tid; i < q_hi; i += kThreads) out_idx[i] = i < R.n ? i : -1;
  } else if (ok && nan_any) {                    // reject the row: all -1
    if (tid == 0 && r == 0) set_err(a.err, SA_ERR_NAN);
    for (int i = q_lo + tid; i < q_hi; i += kThreads) out_idx[i] = -1;
  } else if (ok) {
    const int* info = info_of(a, b);
    const uint32_t sel = (uint32_t)__ldcg(info + 0);
    const int r1 = __ldcg(info + 1);
    const bool overflow = __ldcg(info + 2) != 0;
    int above[kSlices], listed[kSlices];
#pragma unroll
    for (int q = 0; q < kSlices; ++q) {
      above[q] = __ldcg(info + 4 + 2 * q);
      listed[q] = __ldcg(info + 5 + 2 * q);
    }
    uint32_t kr[kSliceKpt];
    slice_keys(a, b, r, R.n, kr);
    int c_all = 0, c_before = 0;                 // listed keys in all slices, in slices < r
#pragma unroll
    for (int q = 0; q < kSlices; ++q) {
      c_before += q < r ? listed[q] : 0;
      c_all += listed[q];
    }
    uint32_t T;
    int take, gt_before = 0, eq_before = 0;
    if (!overflow) {
      // the union of the lists, slice by slice (index order)
      int base = 0;
#pragma unroll
      for (int q = 0; q < kSlices; ++q) {
        const uint32_t* cand = a.tk_cand + ((int64_t)b * kSlices + q) * kCandSlice;
        for (int i = tid; i < listed[q]; i += kThreads) uk[base + i] = __ldcg(cand + i);
        base += listed[q];
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
        T = radix_select<kThreads>(uk, c_all, r1, S, &take, 32 - kFineShift, sel << kFineShift, 1);
      }
      // the slices before r: listed keys > T and == T
      int gb = 0, eb = 0;
      for (int i = tid; i < c_before; i += kThreads) {
        gb += uk[i] > T;
        eb += uk[i] == T;
      }
      const int both = block_sum_nt<kThreads>((gb << 16) | eb, S.scan);   // each <= 3 * 4096
      gt_before = both >> 16;
      eq_before = both & 0xFFFF;
#pragma unroll
      for (int q = 0; q < kSlices; ++q) gt_before += q < r ? above[q] : 0;
    } else {
      // heavily tied row: every key of the row to shared memory, radix passes
      const uint4* src = reinterpret_cast<const uint4*>(a.keys + (int64_t)b * key_stride(a.N_cap));
      for (int q4 = tid; q4 < kKeyCap / 4; q4 += kThreads) {
        uint4 v = 4 * q4 < R.n ? __ldcg(src + q4) : make_uint4(0u, 0u, 0u, 0u);
        if (4 * q4 + 0 >= R.n) v.x = 0u;
        if (4 * q4 + 1 >= R.n) v.y = 0u;
        if (4 * q4 + 2 >= R.n) v.z = 0u;
        if (4 * q4 + 3 >= R.n) v.w = 0u;
        reinterpret_cast<uint4*>(uk)[q4] = v;
      }
      __syncthreads();
      T = radix_select<kThreads>(uk, kKeyCap, r1, S, &take, 32 - kFineShift, sel << kFineShift, 1);
      int gb = 0, eb = 0;
      for (int i = tid; i < r * kSliceKeys; i += kThreads) {
        gb += uk[i] > T;
        eb += uk[i] == T;
      }
      gt_before = block_sum_nt<kThreads>(gb, S.scan);
      eq_before = block_sum_nt<kThreads>(eb, S.scan);
    }
    // this slice: per-thread counts, one scan, emission in index order
    int gt = 0, eq = 0;
#pragma unroll
    for (int j = 0; j < kSliceKpt; ++j) {
      gt += kr[j] > T;
      eq += kr[j] == T;
    }
    int tot = 0;                                 // both prefixes <= 8192: packed in one int
    const int pre = block_exclusive_scan<kThreads>((gt << 16) | eq, S.scan, &tot);
    int gb = gt_before + (pre >> 16), eb = eq_before + (pre & 0xFFFF);
    const int i0 = r * kSliceKeys + kSliceKpt * tid;
    if (gt + eq > 0) {
#pragma unroll
      for (int j = 0; j < kSliceKpt; ++j) {
        if (kr[j] > T) {
          out_idx[gb + min(eb, take)] = i0 + j;
          ++gb;
        } else if (kr[j] == T) {
          if (eb < take) out_idx[gb + eb] = i0 + j;
          ++eb;
        }
      }
    }
  }
  __syncthreads();
  if (tid == 0 && ok) red_release_add(ctr_of(a, kTopkDone, b), 1);
}

// CSA(b, zi) or HCA(b, zi): one share of a row's key list, then the merge of
// the row's shares by whichever finishes last.  n0: attention tiles before
// this item in this CTA (mbarrier phases continue over items); q_ph: parity
// of this item's Q load.  Returns the item's tile count.  Out of line: its
// registers do not count against the score pipeline's.
__device__ __noinline__ int att_item(const TMaps& tm, const StepArgs& a, Ctl& C,
                                     unsigned char* X, uint32_t tmem, int b, int zi, bool csa,
                                     int n0, uint32_t q_ph) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int* abort_flag = &C.abort;
  auto fail = [&]() {
    *abort_flag = 1;
    raise_abort(a);
  };
  unsigned char* sQ = X;
  unsigned char* sKV = X + kQBytes;
  unsigned char* sP = sKV + kStagesKV * kKVBytes;
  int32_t* sel = reinterpret_cast<int32_t*>(sP + 2 * kPBytes);
  const AttGeom G = att_geom(a, b, zi, csa);
  const int nparts = csa ? a.na : a.nh;
  if (tid == 0) {
    int ok = !*abort_flag;
    if (ok) ok = csa ? wait_ge(a, ctr_of(a, kTopkDone, b), kSlices)
                     : wait_ge(a, ctr_of(a, kPoolDone, b), 1);
    if (!ok) *abort_flag = 1;
    C.bcast = ok;
  }
  __syncthreads();
  const bool live = C.bcast != 0;
  const int nt = live ? G.nt : 0;
  const int sel_lo = G.t_lo * kKeys;
  if (csa) {                                 // this share's list slots, read through L2
    for (int s = tid; s < nt * kKeys; s += kThreads) {
      const int pos = sel_lo + s;
      sel[s] = pos < G.n_comp ? __ldcg(a.idx + (int64_t)b * a.k + pos) : -1;
    }
  }
  __syncthreads();
  const void* kc = csa ? a.k_c : a.hk_c;
  const void* vc = csa ? a.v_c : a.hv_c;
  const void* kr = csa ? a.k_raw : a.hk_raw;
  const void* vr = csa ? a.v_raw : a.hv_raw;
  const int ncap = csa ? a.N_cap : a.N2_cap;

  if (warp == kWarpTma && lane == 0 && nt > 0) {
    const CUtensorMap* qm = csa ? &tm.q : &tm.qh;
    mbar_arrive_expect_tx(&C.q_full, kQBytes);
    tma_load_2d(qm, &C.q_full, sQ, 0, b * a.H);
    tma_load_2d(qm, &C.q_full, sQ + kHeads * 128, 64, b * a.H);
  }
  const int nprod = kProducers;              // producer warps 12-15
  if (warp >= kWarpProd) {
    const int pw_ = warp - kWarpProd;
    const __nv_bfloat16* kcb = static_cast<const __nv_bfloat16*>(kc);
    const __nv_bfloat16* vcb = static_cast<const __nv_bfloat16*>(vc);
    const __nv_bfloat16* krb = static_cast<const __nv_bfloat16*>(kr);
    const __nv_bfloat16* vrb = static_cast<const __nv_bfloat16*>(vr);
    for (int n = pw_; n < nt; n += nprod) {
      if (*abort_flag) break;
      const int ng = n0 + n, st = ng % kStagesKV;
      if (!mbar_wait(&C.kv_empty[st], (uint32_t)(((ng / kStagesKV) & 1) ^ 1), a.err)) {
        fail();
        break;
      }
      unsigned char* stage = sKV + st * kKVBytes;
      const uint32_t kd = smem_u32(stage), vd = kd + 2 * kHalf;
      if (!G.gather && (G.t_lo + n + 1) * kKeys <= G.n_comp) {
        // a tile of 64 consecutive HCA cache rows: four TMA boxes (K and V,
        // 64 dims each) in the layout the gather below writes; lane 0's
        // arrival carries the bytes, the other lanes arrive at once
        if (lane == 0) {
          asm volatile("fence.proxy.async;" ::: "memory");   // rows pooled in this launch
          const int32_t row = (int32_t)((int64_t)b * ncap + (int64_t)(G.t_lo + n) * kKeys);
          mbar_arrive_expect_tx(&C.kv_full[st], kKVBytes);
          tma_load_2d(&tm.hk, &C.kv_full[st], stage, 0, row);
          tma_load_2d(&tm.hk, &C.kv_full[st], stage + kHalf, 64, row);
          tma_load_2d(&tm.hv, &C.kv_full[st], stage + 2 * kHalf, 0, row);
          tma_load_2d(&tm.hv, &C.kv_full[st], stage + 3 * kHalf, 64, row);
        } else {
          mbar_arrive(&C.kv_full[st]);
        }
        __syncwarp();
        continue;
      }
      // lane l resolves keys 2l and 2l+1 as (row << 1 | raw), -1 for a
      // masked key; each cp.async instruction then copies two whole rows
      int64_t src2[2];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int s = (G.t_lo + n) * kKeys + 2 * lane + q;   // list position
        int64_t code = -1;
        if (s < G.n_comp) {
          const int j = G.gather ? sel[s - sel_lo] : s;
          if (j >= 0 && j < G.nvis) code = ((int64_t)b * ncap + j) << 1;
          else if (j != -1) set_err(a.err, SA_ERR_BOUNDS);
        } else if (s >= G.n_comp_pad && s < G.n_comp_pad + G.n_win) {
          const int64_t u = (int64_t)G.p - G.n_win + 1 + (s - G.n_comp_pad);
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
        const __nv_bfloat16* ks = raw ? krb : kcb;
        const __nv_bfloat16* vs = raw ? vrb : vcb;
        const uint32_t bytes = code >= 0 ? 16u : 0u;
        const int64_t off = (code >= 0 ? (code >> 1) : 0) * kD + ch * 8;
        const uint32_t o = (ch >> 3) * kHalf + swz(key, ch & 7);
        cp_async16(kd + o, (code >= 0 ? ks : krb) + off, bytes);
        cp_async16(vd + o, (code >= 0 ? vs : vrb) + off, bytes);
      }
      // one tile in flight per producer: the MMA frees tile n's stage only
      // after it has issued S(n + 1), so a producer holding an unsignalled
      // tile while waiting for a stage could wait on itself
      asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
      fence_proxy_async_smem();
      mbar_arrive(&C.kv_full[st]);
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
  } else if (warp == kWarpMma) {
    if (lane == 0 && nt > 0) {
      constexpr uint32_t idS = idesc_bf16(kHeads, kKeys, 0, 0);
      constexpr uint32_t idO = idesc_bf16(kHeads, kD, 0, 1);
      const uint32_t qa = smem_u32(sQ);
      bool ok = mbar_wait(&C.q_full, q_ph, a.err);
      auto pv = [&](int m_) -> bool {        // O += P(m_) . V(m_); m_ local to the item
        const int mg = n0 + m_, pb = mg & 1;
        if (!mbar_wait(&C.p_full[pb], (uint32_t)((mg >> 1) & 1), a.err)) return false;
        tc_fence_after();
        const uint32_t pa = smem_u32(sP + pb * kPBytes);
        const uint32_t va = smem_u32(sKV + (mg % kStagesKV) * kKVBytes) + 2 * kHalf;
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk)
          tc_mma_f16(tmem + 128, sdesc_kmajor_sw128(pa + kk * 32),
                     sdesc_mnmajor_sw128(va + kk * 2048, kHalf, 1024), idO,
                     (m_ > 0 || kk > 0) ? 1u : 0u);
        tc_commit(&C.kv_empty[mg % kStagesKV]);
        tc_commit(&C.p_empty[pb]);
        return true;
      };
      for (int n = 0; n < nt && ok; ++n) {
        if (*abort_flag) { ok = false; break; }
        const int ng = n0 + n, st = ng % kStagesKV, sb = ng & 1;
        if (!mbar_wait(&C.kv_full[st], (uint32_t)((ng / kStagesKV) & 1), a.err) ||
            !mbar_wait(&C.s_empty[sb], (uint32_t)(((ng >> 1) & 1) ^ 1), a.err)) {
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
      if (ok && !pv(nt - 1)) ok = false;
      if (!ok) fail();
    }
    __syncwarp();
  } else if (warp >= kWarpSoft && warp < kWarpSoft + 4) {
    // S and O through the 16x256b TMEM shape: lane l holds heads
    // h0 = 16q + l/4 and h1 = h0 + 8, keys 8g + 2(l%4) and +1 of each
    // 8-key group g
    const int quad = warp & 3, l4 = lane & 3;
    const int h0 = quad * 16 + (lane >> 2), h1 = h0 + 8;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const float c2 = a.sm_scale * 1.4426950408889634f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    bool ok = true;
    for (int n = 0; n < nt && ok; ++n) {
      const int ng = n0 + n;
      const int s0 = (G.t_lo + n) * kKeys;
      const bool ok0 = h0 < a.H, ok1 = h1 < a.H;
      auto is_real = [&](int sk) -> bool {
        if (sk < G.n_comp) {
          if (!G.gather) return true;
          const int jj = sel[sk - sel_lo];
          return jj >= 0 && jj < G.nvis;
        }
        return sk >= G.n_comp_pad && sk < G.n_comp_pad + G.n_win;
      };
      const uint32_t re = __ballot_sync(0xffffffffu, is_real(s0 + 2 * lane));
      const uint32_t ro = __ballot_sync(0xffffffffu, is_real(s0 + 2 * lane + 1));
      uint32_t keep16 = 0;
#pragma unroll
      for (int g = 0; g < 8; ++g)
        keep16 |= (((re >> (4 * g + l4)) & 1u) << (2 * g)) |
                  (((ro >> (4 * g + l4)) & 1u) << (2 * g + 1));
      const int sb = ng & 1, pb = ng & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(&C.s_full[sb], (uint32_t)((ng >> 1) & 1), a.err));
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
        ok = __all_sync(0xffffffffu, mbar_wait(&C.p_empty[(ng - 1) & 1],
                                               (uint32_t)(((ng - 1) >> 1) & 1), a.err));
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
      // P buffer pb is free once PV(ng-2) is done
      ok = __all_sync(0xffffffffu,
                      mbar_wait(&C.p_empty[pb], (uint32_t)(((ng >> 1) & 1) ^ 1), a.err));
      if (!ok) break;
      {
        unsigned char* prow = sP + pb * kPBytes + 4 * l4;
        const float r0 = m0 == -INFINITY ? 0.f : m0, r1 = m1 == -INFINITY ? 0.f : m1;
        float u0 = 0.f, u1 = 0.f;
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          const __nv_bfloat162 p0 = __floats2bfloat162_rn(
              fast_exp2(fmaf(v[4 * g], c2, -r0)), fast_exp2(fmaf(v[4 * g + 1], c2, -r0)));
          const __nv_bfloat162 p1 = __floats2bfloat162_rn(
              fast_exp2(fmaf(v[4 * g + 2], c2, -r1)), fast_exp2(fmaf(v[4 * g + 3], c2, -r1)));
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
    // ---- this item's partial: O = all PVs (the last one signals p_empty)
    if (ok && nt > 0)
      ok = __all_sync(0xffffffffu, mbar_wait(&C.p_empty[(n0 + nt - 1) & 1],
                                             (uint32_t)(((n0 + nt - 1) >> 1) & 1), a.err));
    if (!ok) fail();
    tc_fence_after();
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    const bool have0 = ok && nt > 0 && l0 > 0.f, have1 = ok && nt > 0 && l1 > 0.f;
    const float inv0 = have0 ? 1.f / l0 : 0.f, inv1 = have1 ? 1.f / l1 : 0.f;
    float* po = (csa ? a.part_o : a.hpart_o) + ((int64_t)b * nparts + G.z) * kHeads * kD;
    float* pl = (csa ? a.part_lse : a.hpart_lse) + ((int64_t)b * nparts + G.z) * kHeads;
    const uint32_t tO = tmem + lane_base + 128;
#pragma unroll 1
    for (int c = 0; c < kD; c += 32) {
      float o[16];
      if (nt > 0) {
        tmem_ld16x256b_x4(tO + c, o);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) o[i] = 0.f;
      }
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const int col = c + 8 * g + 2 * l4;
        __stcg(reinterpret_cast<float2*>(po + h0 * kD + col),
               make_float2(o[4 * g] * inv0, o[4 * g + 1] * inv0));
        __stcg(reinterpret_cast<float2*>(po + h1 * kD + col),
               make_float2(o[4 * g + 2] * inv1, o[4 * g + 3] * inv1));
      }
    }
    if (l4 == 0) {
      __stcg(pl + h0, have0 ? (m0 + log2f(l0)) * 0.6931471805599453f : -INFINITY);
      __stcg(pl + h1, have1 ? (m1 + log2f(l1)) * 0.6931471805599453f : -INFINITY);
    }
  }
  if (warp == kWarpTma && lane == 0 && nt > 0)   // the Q copy has landed before X is reused
    mbar_wait(&C.q_full, q_ph, a.err);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // the last share of the row to finish merges the partials
  if (tid == 0) {
    const int old = atom_acq_rel_add(ctr_of(a, csa ? kCsaParts : kHcaParts, b), 1);
    C.bcast = old == nparts - 1;
  }
  __syncthreads();
  if (C.bcast) {
    const float* pob = (csa ? a.part_o : a.hpart_o) + (int64_t)b * nparts * kHeads * kD;
    const float* plb = (csa ? a.part_lse : a.hpart_lse) + (int64_t)b * nparts * kHeads;
    void* out = csa ? a.o : a.ho;
    float* out_lse = csa ? a.lse : a.hlse;
    for (int t = tid; t < kHeads * 32; t += kThreads) {
      const int h = t >> 5, c4 = t & 31;
      if (h >= a.H) continue;
      float L[kMaxParts];
      float mx = -INFINITY;
#pragma unroll
      for (int r = 0; r < kMaxParts; ++r) {
        L[r] = r < nparts ? __ldcg(plb + r * kHeads + h) : -INFINITY;
        mx = fmaxf(mx, L[r]);
      }
      float lse_out = -INFINITY;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      if (mx != -INFINITY) {
        float sum = 0.f;
#pragma unroll
        for (int r = 0; r < kMaxParts; ++r)
          if (r < nparts) sum += expf(L[r] - mx);
        lse_out = mx + logf(sum);
#pragma unroll
        for (int r = 0; r < kMaxParts; ++r) {
          if (r < nparts && L[r] != -INFINITY) {
            const float wgt = expf(L[r] - lse_out);
            const float4 v = __ldcg(reinterpret_cast<const float4*>(
                                        pob + ((int64_t)r * kHeads + h) * kD) + c4);
            acc.x = fmaf(wgt, v.x, acc.x);
            acc.y = fmaf(wgt, v.y, acc.y);
            acc.z = fmaf(wgt, v.z, acc.z);
            acc.w = fmaf(wgt, v.w, acc.w);
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
        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(out) + o0) = u;
      } else {
        *reinterpret_cast<float4*>(static_cast<float*>(out) + o0) = acc;
      }
      if (c4 == 0) out_lse[(int64_t)b * a.H + h] = lse_out;
    }
  }
  return nt;
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
    decode_step_kernel(const __grid_constant__ TMaps tm, const __grid_constant__ StepArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  Ctl& C = *reinterpret_cast<Ctl*>(smem_raw);
  unsigned char* X = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + sizeof(Ctl) + 1023) & ~uintptr_t(1023));
  // region X, by item kind:
  //  SCORE: stages [kStagesA][32 KB] | B [2][8 KB]
  //  TOPKA: histogram [8192] | TopkSmem;  TOPKB: candidate union or all keys [32768] | TopkSmem
  //  CSA/HCA: Q [16 KB] | K/V stages [kStagesKV][32 KB] | P [2][8 KB] | list slots
  //  POOL: two blocks' raw rows [2][128 x 40 x 16 B] | partial sums [2][8 x 40 x 8] floats
  unsigned char* sA = X;
  unsigned char* sB = X + kStagesA * kABytes;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int* abort_flag = &C.abort;

  if (tid == 0) {
    for (int s = 0; s < kRing; ++s) { mbar_init(&C.it_full[s], 1); mbar_init(&C.it_empty[s], 16); }
    for (int s = 0; s < kStagesA; ++s) { mbar_init(&C.a_full[s], 1); mbar_init(&C.a_empty[s], 1); }
    for (int s = 0; s < 2; ++s) { mbar_init(&C.b_full[s], 1); mbar_init(&C.b_empty[s], 1); }
    for (int s = 0; s < kAcc; ++s) { mbar_init(&C.t_full[s], 1); mbar_init(&C.t_empty[s], 128); }
    for (int s = 0; s < kStagesKV; ++s) { mbar_init(&C.kv_full[s], 32); mbar_init(&C.kv_empty[s], 1); }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&C.s_full[s], 1);
      mbar_init(&C.s_empty[s], 128);
      mbar_init(&C.p_full[s], 128);
      mbar_init(&C.p_empty[s], 1);
    }
    mbar_init(&C.q_full, 1);
    C.abort = 0;
    mbar_fence_init();
  }
  if (warp == kWarpMma) tmem_alloc(&C.tmem, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = C.tmem;
  if (warp == kWarpTma && lane == 0) {
    tma_prefetch_desc(&tm.ik);
    tma_prefetch_desc(&tm.qi);
    tma_prefetch_desc(&tm.q);
    tma_prefetch_desc(&tm.qh);
    tma_prefetch_desc(&tm.hk);
    tma_prefetch_desc(&tm.hv);
  }

  Counters K = {0, 0, 0, 0, 0};
  bool next_claimed = false;                     // TMA warp: the next item is already published
  int drain_from = 0;                            // TMA warp: stages not yet known to have landed
  bool b_pending[2] = {false, false};            // TMA warp: B loads not yet known to have landed

  // fail: this CTA drops the rest of its work and every CTA stops taking items
  auto fail = [&]() {
    *abort_flag = 1;
    raise_abort(a);
  };

  for (int seq = 0;; ++seq) {
    const int slot = seq % kRing;
    const uint32_t ring_ph = (uint32_t)((seq / kRing) & 1);
    // ---------------------------------------------------------- claim
    // claim and publish item seq (unless the previous SCORE item already did)
    auto publish = [&](int sq) {
      const int sl = sq % kRing;
      int4 itc = make_int4(kStop, 0, 0, 0);
      if (mbar_wait(&C.it_empty[sl], (uint32_t)(((sq / kRing) & 1) ^ 1), a.err)) {
        if (!*abort_flag && !aborted(a)) itc = claim_item(a);
      } else {
        fail();
      }
      C.ring[sl] = itc;
      mbar_arrive(&C.it_full[sl]);
    };
    if (warp == kWarpTma && lane == 0) {
      if (!next_claimed) publish(seq);
      next_claimed = false;
    }
    bool ok_slot = mbar_wait(&C.it_full[slot], ring_ph, a.err);
    ok_slot = __all_sync(0xffffffffu, ok_slot);
    const int4 it = ok_slot ? C.ring[slot] : make_int4(kStop, 0, 0, 0);
    __syncwarp();
    if (lane == 0) mbar_arrive(&C.it_empty[slot]);
    if (!ok_slot && lane == 0) fail();
    if (it.x == kStop) break;

    // ====================================================== SCORE item
    if (it.x == kScore) {
      const ScoreGeom G = score_geom(a, it.y, it.z);
      const int nt = G.t1 - G.t0;
      const bool live = nt > 0;
      const int sb = K.s_items & 1;
      const uint32_t b_ph = (uint32_t)((K.s_items >> 1) & 1);
      const int b = G.b;
      if (warp == kWarpTma) {
        if (lane == 0 && live && !*abort_flag) {
          bool ok = true;
          // blocks pooled this step: the stages holding their rows are loaded
          // only once POOL(b) is done; the stages before them do not wait
          const int fb_lo = __ldg(a.blk_lo + b), fb_hi = __ldg(a.blk_hi + b);
          bool pooled = false;
          ok = mbar_wait(&C.b_empty[sb], b_ph ^ 1, a.err);
          if (ok) {
            mbar_arrive_expect_tx(&C.b_full[sb], kBBytes);
            tma_load_2d(&tm.qi, &C.b_full[sb], sB + sb * kBBytes, 0, b * kHI);
            b_pending[sb] = true;
          }
          for (int t = G.t0; t < G.t1 && ok; t += kStageTiles) {
            const int u = K.stages + (t - G.t0) / kStageTiles;
            const int st = u % kStagesA;
            // halfway through this item's loads, take the next item: the
            // claim's memory round trips overlap the stream instead of
            // stalling it between items
            if (!next_claimed && 2 * (t - G.t0) >= G.t1 - G.t0) {
              publish(seq + 1);
              next_claimed = true;
            }
            if (!pooled && max(fb_lo, t * kTile) < min(fb_hi, (t + kStageTiles) * kTile)) {
              ok = wait_ge(a, ctr_of(a, kPoolDone, b), 1);
              asm volatile("fence.proxy.async;" ::: "memory");
              pooled = true;
              if (!ok) break;
            }
            if (!mbar_wait(&C.a_empty[st], (uint32_t)(((u / kStagesA) & 1) ^ 1), a.err)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&C.a_full[st], kABytes);
            tma_load_2d(&tm.ik, &C.a_full[st], sA + st * kABytes, 0,
                        (int32_t)((int64_t)b * a.N_cap + (int64_t)t * kTile));
          }
          if (!ok) fail();
        }
        __syncwarp();
      } else if (warp == kWarpMma) {
        if (lane == 0 && live && !*abort_flag) {
          constexpr uint32_t idesc = idesc_bf16(kTile, kHI);
          bool ok = mbar_wait(&C.b_full[sb], b_ph, a.err);
          const uint32_t b_base = smem_u32(sB + sb * kBBytes);
          for (int o = 0; o < nt && ok; ++o) {
            const int u = K.stages + o / kStageTiles, half = o % kStageTiles;
            const int st = u % kStagesA, og = K.tiles + o, acc = og % kAcc;
            if ((half == 0 && !mbar_wait(&C.a_full[st], (uint32_t)((u / kStagesA) & 1), a.err)) ||
                !mbar_wait(&C.t_empty[acc], (uint32_t)(((og / kAcc) & 1) ^ 1), a.err)) {
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
            if (half == kStageTiles - 1 || o == nt - 1) tc_commit(&C.a_empty[st]);
          }
          if (ok) tc_commit(&C.b_empty[sb]);
          else fail();
        }
        __syncwarp();
      } else if (warp >= kWarpEpi) {
        // epilogue warpgroup grp takes tiles og = grp (mod 3); warp w reads
        // TMEM lanes 32*(w%4)..
        const int grp = (warp - kWarpEpi) >> 2;
        const int gt = tid - (kWarpEpi + 4 * grp) * 32;          // 0..127 in the group
        const int quad = warp & 3;
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        if (live && gt < kHI) C.wgt[grp][gt] = __ldg(a.w + (int64_t)b * kHI + gt);
        named_bar_sync(2 + grp, 128);
        int nan_local = 0;

        const float4* w4 = reinterpret_cast<const float4*>(C.wgt[grp]);
        const int first = (grp - K.tiles % kEpiGroups + kEpiGroups) % kEpiGroups;
        for (int o = first; o < nt && live; o += kEpiGroups) {
          const int og = K.tiles + o, acc = og % kAcc;
          // warp-uniform: the TMEM loads below are warp-collective
          if (!__all_sync(0xffffffffu,
                          !*abort_flag &&
                              mbar_wait(&C.t_full[acc], (uint32_t)((og / kAcc) & 1), a.err))) {
            fail();
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
          const int j = (G.t0 + o) * kTile + quad * 32 + lane;
          if (j < G.n) {
            nan_local |= is_nan_bits(s);
            const uint32_t key = score_key(s);
            a.keys[(int64_t)b * key_stride(a.N_cap) + j] = key;
            // the row's 13-bit histogram, for its top-k (fire and forget)
            asm volatile("red.relaxed.gpu.global.add.s32 [%0], 1;" ::"l"(hist_of(a, b) +
                                                                           (key >> kFineShift))
                         : "memory");
          }
        }
        if (nan_local) atomicOr(ctr_of(a, kNan, b), 1);
        named_bar_sync(2 + grp, 128);            // the group's keys are written; weights free
        if (gt == 0) red_release_add(ctr_of(a, kScoreDone, b), 1);
      }
      if (live) {
        K.s_items += 1;
        K.stages += (nt + kStageTiles - 1) / kStageTiles;
        K.tiles += nt;
      }
      continue;
    }

    // ============================================ CTA-wide items
    // Every warp is past its earlier items: the score pipeline is empty (each
    // accumulator was read after its MMAs completed), so region X is free.
    if (warp == kWarpTma && lane == 0) {
      // no TMA copy may still be landing in region X (only after a failure
      // can one be outstanding)
      for (int u = max(drain_from, K.stages - kStagesA); u < K.stages; ++u)
        mbar_wait(&C.a_full[u % kStagesA], (uint32_t)((u / kStagesA) & 1), a.err);
      drain_from = K.stages;
      for (int s = 0; s < 2; ++s) {
        if (!b_pending[s]) continue;
        // the last B load into buffer s was use number K.s_items - 1 - ((K.s_items - 1 - s) & 1)
        const int use = (K.s_items - 1) - (((K.s_items - 1) & 1) != s ? 1 : 0);
        if (use >= 0) mbar_wait(&C.b_full[s], (uint32_t)((use >> 1) & 1), a.err);
        b_pending[s] = false;
      }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const int b = it.y;

    // --------------------------------------------------------- POOL
    if (it.x == kPool) {
      pool_item(a, C, X, b);
    }
    // -------------------------------------------------------- TOPKA / TOPKB
    else if (it.x == kTopkA) {
      topka_item(a, C, X, b, it.z);
    } else if (it.x == kTopkB) {
      topkb_item(a, C, X, b, it.z);
    }
    // --------------------------------------------------- CSA / HCA attention
    else {
      const int nt = att_item(tm, a, C, X, tmem, b, it.z, it.x == kCsa, K.att_tiles,
                              (uint32_t)(K.att_items & 1));
      if (nt > 0) K.att_items += 1;
      K.att_tiles += nt;
    }
    // the next items' TMA copies (the async proxy) may land where this item
    // wrote shared memory through the generic proxy
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }

  // no copy may still be landing when the CTA exits (only after a failure
  // can one be outstanding)
  if (warp == kWarpTma && lane == 0) {
    for (int u = max(drain_from, K.stages - kStagesA); u < K.stages; ++u)
      mbar_wait(&C.a_full[u % kStagesA], (uint32_t)((u / kStagesA) & 1), a.err);
    for (int s = 0; s < 2; ++s) {
      if (!b_pending[s]) continue;
      const int use = (K.s_items - 1) - (((K.s_items - 1) & 1) != s ? 1 : 0);
      if (use >= 0) mbar_wait(&C.b_full[s], (uint32_t)((use >> 1) & 1), a.err);
    }
  }
  tc_fence_before();
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

// bf16 matrix [rows, cols], box 64 columns x box_rows rows, 128-byte swizzle.
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

static size_t step_smem() {
  const size_t score = (size_t)kStagesA * kABytes + 2 * kBBytes;
  const size_t topk = 4 * (size_t)kKeyCap + sizeof(TopkSmem);
  const size_t att = kQBytes + (size_t)kStagesKV * kKVBytes + 2 * kPBytes +
                     4 * (size_t)kKeys * kStepMaxTilesPerPart;
  const size_t pool = 2 * (size_t)kMaxPool * 40 * 16 + 2 * 4 * 8 * 40 * 8;
  return round_up(sizeof(Ctl), 16) + 1024 + std::max(std::max(score, topk), std::max(att, pool));
}

constexpr size_t kSmemMax = 232448;              // 227 KB per block on sm_100-class parts

bool decode_step_plan(StepArgs& a, int num_sms) {
  if (a.B <= 0 || a.N_cap > kKeyCap || a.m > kMaxPool || a.m2 > kMaxPool || a.H > kHeads)
    return false;
  if (step_smem() > kSmemMax) return false;
  const int ntiles = (a.N_cap + kTile - 1) / kTile;
  a.tps = 32;
  a.ns = std::max(1, (ntiles + a.tps - 1) / a.tps);
  // attention shares: about 9 key tiles each, at most kMaxParts per row
  auto split = [](int ntl, int& parts, int& per) {
    parts = std::min(kMaxParts, std::max(1, (ntl + 8) / 9));
    per = std::max(1, (ntl + parts - 1) / parts);
  };
  const int ntl_a = ((std::min(a.k, a.N_cap) + 3) / 4 * 4 + a.W + kKeys - 1) / kKeys;
  const int ntl_h = ((a.N2_cap + 3) / 4 * 4 + a.W + kKeys - 1) / kKeys;
  split(ntl_a, a.na, a.tpa);
  split(ntl_h, a.nh, a.tph);
  if (a.tpa > kStepMaxTilesPerPart || a.tph > kStepMaxTilesPerPart) return false;
  a.grid = num_sms;
  return true;
}

size_t decode_step_counter_bytes(int B) {
  return round_up(4 * ((size_t)ctr_ints(B) + (size_t)B * (kFineBins + kInfo)), 256);
}

cudaError_t launch_decode_step(const StepArgs& a, cudaStream_t st) {
  TMaps tm;
  const bool no_keys = (uint64_t)a.B * a.N_cap == 0;
  if (!tmap_bf16(&tm.ik, no_keys ? a.q_idx : a.ik_c,
                 no_keys ? (uint64_t)a.B * kHI : (uint64_t)a.B * a.N_cap, kDI,
                 kStageTiles * kTile) ||
      !tmap_bf16(&tm.qi, a.q_idx, (uint64_t)a.B * kHI, kDI, kHI) ||
      !tmap_bf16(&tm.q, a.q, (uint64_t)a.B * a.H, kD, kHeads) ||
      !tmap_bf16(&tm.qh, a.q_hca, (uint64_t)a.B * a.H, kD, kHeads))
    return cudaErrorInvalidValue;
  // with no HCA rows the cache maps are never used: they then describe the
  // queries instead, so that they still encode
  const bool no_hca = (uint64_t)a.B * a.N2_cap == 0;
  if (!tmap_bf16(&tm.hk, no_hca ? a.q_hca : a.hk_c, no_hca ? (uint64_t)a.B * a.H : (uint64_t)a.B * a.N2_cap,
                 kD, kKeys) ||
      !tmap_bf16(&tm.hv, no_hca ? a.q_hca : a.hv_c, no_hca ? (uint64_t)a.B * a.H : (uint64_t)a.B * a.N2_cap,
                 kD, kKeys))
    return cudaErrorInvalidValue;
  const size_t smem = step_smem();
  cudaError_t e = cudaFuncSetAttribute(decode_step_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(a.ctr, 0, decode_step_counter_bytes(a.B), st);
  if (e != cudaSuccess) return e;
  decode_step_kernel<<<a.grid, kThreads, smem, st>>>(tm, a);
  return cudaGetLastError();
}

}  // namespace sa
