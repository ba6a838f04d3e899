// Multi-query attention over gathered compressed rows plus the sliding window
// on the 5th-generation tensor cores (bf16 in, fp32 accumulation in TMEM).
//
// Source: "오픈소스 LLM의 새 이정표: DeepSeek-V4 시리즈", section
// "압축 희소 어텐션(CSA)과 극압축 어텐션(HCA)" (CSA: top-k compressed entries plus a
// sliding-window branch; HCA: dense attention over all compressed entries),
// "DeepSeek-V4 논문 읽기: 백만 토큰 컨텍스트를 저렴하게", sections "Compressed Sparse
// Attention (CSA)" steps 3-4 and "Heavily Compressed Attention (HCA)", and
// "EP 95. DeepSeek-V4 논문 읽기 — 노정석", section IDEAS (one shared KV head).
//
// Work: an item is (query row, split of the row's key list); a persistent grid
// takes items as they come free.  Two shapes of the same pipeline:
//  * shallow (decode): two CTAs per SM, each with two K/V stages, one Q tile
//    and 256 TMEM columns -- two independent pipelines per SM hide the
//    set-up and drain of the short items of a decode step;
//  * deep (long key lists, prefill): one CTA per SM with six K/V stages and
//    four producer warps, so that up to four tiles are gathered while the
//    tensor core works on two.
// A row's key list is the
// compressed part (rows idx[r, i] for CSA, rows 0.. for HCA), padded to a
// multiple of 4 keys, then the window rows (ring slot u mod R); it is
// processed in tiles of 64 keys.
//
// Warp roles (P producer warps; 32 * (P + 6) threads):
//  * warp P, fetcher: takes the CTA's items one by one from a counter shared
//    by the grid (zeroed by the call before the launch) and passes them to
//    the other roles through a two-slot ring in shared memory.  CTAs that
//    start late -- behind another kernel that holds most SMs -- find the
//    work already taken, so the grid never waits for them.  Without a
//    counter it hands out items c, c+G, ...
//  * warps 0..P-1, producers: warp w issues the tiles with ordinal n = w (mod P).
//    Lane l finds the source rows of keys 2l and 2l+1; then each cp.async
//    instruction of the warp copies two whole 256-byte rows (half-warp per
//    key, one 16-byte chunk per lane) straight into the 128B-swizzled layout
//    the tensor core reads (keys past the list are zero-filled); the warp
//    waits for its copies, fences them to the async proxy and arrives on the
//    stage's mbarrier, so P tiles are in flight per CTA.  In dense mode
//    (HCA) a tile of 64 consecutive compressed rows comes instead by four TMA
//    boxes, the copy engine applying the same swizzle.
//    Warp 0 also brings the item's 64 query heads by one TMA tiled load per
//    64-column half into the Q tile.
//  * warp P+1, MMA: S(n) = Q . K(n)^T (M = 64 heads, N = 64 keys, K = 128) into
//    one of two TMEM S buffers, issued before PV(n-1) so that the softmax of
//    tile n overlaps the tensor core; O += P(n) . V(n) (M = 64, N = 128,
//    K = 64) into the TMEM O accumulator (freed by the softmax after each item).
//  * warps P+2..P+5, softmax (TMEM lane quarter = warp mod 4): the M = 64
//    accumulator puts rows 16q..16q+15 in
//    TMEM lanes 32q..32q+15; the 16x256b load shape spreads those 16 rows
//    over all 32 lanes (two heads and a quarter of the keys per lane), fp32
//    exp2 of the scaled logits, P to shared memory in bf16; the running max
//    is raised only when it grows by more than 32 (log2 units), and then O is
//    rescaled in TMEM.
//    At the end of an item it writes the normalised O and the LSE (or a
//    normalised split partial, merged by merge_splits_kernel).
// Mbarriers are waited by phase parity, which is sound only while a barrier is
// at most one phase away from the awaited one; every wait below is placed so
// that this holds.  Every wait is bounded; on a timeout the CTA records
// SA_ERR_DEVICE_TIMEOUT, stops and still frees its TMEM.
#include <cudaTypedefs.h>

#include "kernels.cuh"

namespace sa {

namespace {

constexpr int kMaxStages = 6;                  // K/V stages of the deepest shape

// One shape of the pipeline: CTAs per SM, K/V stages per CTA, producer warps.
// A producer's wait for stage n % S is sound by parity only while that
// barrier is at most one phase behind: the warp's own previous tile n - P
// waited for the release of tile n - P - S, which covers tile n - 2S as long
// as P <= S (releases come in tile order).
template <int kCtas, int kStg, int kProd>
struct AttnShape {
  static constexpr int kCtasPerSm = kCtas;
  static constexpr int kStages = kStg;
  static constexpr int kProducers = kProd;
  static constexpr int kFetchWarp = kProd;       // fills the item ring
  static constexpr int kMmaWarp = kProd + 1;     // MMA issuer and TMEM owner; softmax after it
  static constexpr int kThreads = 32 * (kProd + 6);
  // warps that read every item: the producers, the MMA warp, the 4 softmax warps
  static constexpr int kItemReaders = kProd + 1 + 4;
  static_assert(kProd <= kStg, "parity waits of the producers");
  static_assert(kStg <= kMaxStages, "stage barriers in Ctl");
};
using ShallowShape = AttnShape<2, 2, 2>;         // decode: two pipelines per SM
using DeepShape = AttnShape<1, 6, 4>;            // long key lists: one deep pipeline
// items per SM from which a launch takes the deep shape
constexpr int kAttnDeepItemsPerSm = 8;

constexpr int kKeys = 64;                      // keys per tile
constexpr int kQBufs = 1;                      // query tiles per CTA
constexpr int kOBufs = 1;                      // TMEM O accumulators per CTA
constexpr int kD = 128;                        // head dim
constexpr int kHeads = 64;                     // MMA M
constexpr int kHalf = kKeys * 128;             // 8 KB: a 64-dim half of a K or V tile
constexpr int kQBytes = kHeads * kD * 2;       // 16 KB: two 64-column halves
constexpr int kStageBytes = 4 * kHalf;         // K (2 halves) + V (2 halves) = 32 KB
constexpr int kPBytes = kHeads * kKeys * 2;    // 8 KB
constexpr int kTmemCols = 256;                 // S: 2 x 64 at 0; O: 128 at 128 (half of TMEM)
constexpr float kRescaleThreshold = 32.f;      // log2 units: P <= 2^32, far inside fp32 and bf16

struct Ctl {
  uint64_t full[kMaxStages], empty[kMaxStages];
  uint64_t q_full[kQBufs], q_empty[kQBufs];
  uint64_t s_full[2], s_empty[2];
  uint64_t p_full[2], p_empty[2];
  uint64_t o_empty[kOBufs];
  uint64_t it_full[2], it_empty[2];   // ring of the CTA's next items (fetched by the fetcher)
  int64_t it_slot[2];
  uint32_t tmem;
  int abort;
};

struct TMaps {
  CUtensorMap q;
  CUtensorMap k, v;        // dense mode: the compressed caches [B*N_cap, 128], box 64 x 64
  int dense_tma;           // 1: tiles wholly inside a row's compressed rows come by TMA
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

// Byte offset of 16-byte chunk `c` (0..7) of 128-byte row `r` inside a
// 128B-swizzled block whose base is 1024-aligned.
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}

struct Item {
  int64_t row;
  int split;
  int b, p;
  int64_t nvis, n_comp, n_comp_pad, n_win;
  int64_t t_begin;
  int nt;
};

__device__ __forceinline__ Item make_item(const AttnArgs& a, int64_t it) {
  Item I;
  I.row = it / a.nsplit;
  I.split = (int)(it % a.nsplit);
  I.b = (int)(I.row / a.T);
  I.p = __ldg(a.q_pos + I.row);
  I.nvis = I.p < 0 ? 0 : ((int64_t)I.p + 1) / a.m;
  if (I.nvis > a.N_cap) I.nvis = a.N_cap;
  I.n_comp = a.gather ? min64(a.k, I.nvis) : I.nvis;
  I.n_comp_pad = (I.n_comp + 3) & ~int64_t(3);
  I.n_win = I.p < 0 ? 0 : min64(a.W, (int64_t)I.p + 1);
  const int64_t nt_row = (I.n_comp_pad + I.n_win + kKeys - 1) / kKeys;
  I.t_begin = (int64_t)I.split * a.split_tiles;
  I.nt = (int)max64(0, min64(nt_row, I.t_begin + a.split_tiles) - I.t_begin);
  return I;
}

}  // namespace

template <class Sh>
__global__ void __launch_bounds__(Sh::kThreads, Sh::kCtasPerSm)
    attend_tc_kernel(const __grid_constant__ TMaps tm, AttnArgs a) {
  constexpr int kStages = Sh::kStages, kProducers = Sh::kProducers;
  constexpr int kFetchWarp = Sh::kFetchWarp, kMmaWarp = Sh::kMmaWarp;
  extern __shared__ unsigned char smem_raw[];
  Ctl& C = *reinterpret_cast<Ctl*>(smem_raw);
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + sizeof(Ctl) + 1023) & ~uintptr_t(1023));
  unsigned char* sQ = base;                          // [2][kQBytes]
  unsigned char* sKV = sQ + kQBufs * kQBytes;        // [kStages][kStageBytes]
  unsigned char* sP = sKV + kStages * kStageBytes;   // [2][kPBytes]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t n_items = (int64_t)a.B * a.T * a.nsplit;
  volatile int* abort_flag = &C.abort;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&C.full[s], 32);
      mbar_init(&C.empty[s], 1);
    }
    for (int s = 0; s < kQBufs; ++s) {
      mbar_init(&C.q_full[s], 1);
      mbar_init(&C.q_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&C.s_full[s], 1);
      mbar_init(&C.s_empty[s], 128);
      mbar_init(&C.p_full[s], 128);
      mbar_init(&C.p_empty[s], 1);
    }
    for (int s = 0; s < kOBufs; ++s) mbar_init(&C.o_empty[s], 128);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&C.it_full[s], 1);
      mbar_init(&C.it_empty[s], Sh::kItemReaders);
    }
    C.abort = 0;
    mbar_fence_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm.q);
    if (tm.dense_tma) {
      tma_prefetch_desc(&tm.k);
      tma_prefetch_desc(&tm.v);
    }
  }
  // the fetcher claims its first item now, so the round trip to the counter
  // overlaps the set-up
  int64_t first_item = -1;
  if (warp == kFetchWarp && lane == 0)
    first_item = a.item_counter ? (int64_t)atomicAdd(a.item_counter, 1u) : (int64_t)blockIdx.x;
  if (warp == kMmaWarp) tmem_alloc(&C.tmem, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = C.tmem;

  // The e-th item of this CTA (-1: none left), from the ring warp 3 fills;
  // lane 0 of each reading warp releases the slot once the warp has read it.
  auto next_item = [&](int64_t e, bool whole_warp) -> int64_t {
    const int slot = (int)(e & 1);
    if (!mbar_wait(&C.it_full[slot], (uint32_t)((e >> 1) & 1), a.err)) {
      *abort_flag = 1;
      return -1;
    }
    const int64_t it = *reinterpret_cast<volatile int64_t*>(&C.it_slot[slot]);
    if (whole_warp) __syncwarp();
    if (!whole_warp || lane == 0) mbar_arrive(&C.it_empty[slot]);
    return it;
  };

  if (warp == kFetchWarp) {
    // ======================================================= item fetcher
    // Items come from a counter shared by the grid (dynamic: CTAs that start
    // late, behind other kernels, find the work already taken), or c, c+G,
    // ... without one.
    if (lane == 0) {
      for (int64_t e = 0;; ++e) {
        const int slot = (int)(e & 1);
        int64_t it = -1;
        if (mbar_wait(&C.it_empty[slot], (uint32_t)(((e >> 1) & 1) ^ 1), a.err)) {
          it = e == 0 ? first_item
                      : a.item_counter ? (int64_t)atomicAdd(a.item_counter, 1u)
                                       : (int64_t)blockIdx.x + e * gridDim.x;
          if (it >= n_items || *abort_flag) it = -1;
        } else {
          *abort_flag = 1;
        }
        *reinterpret_cast<volatile int64_t*>(&C.it_slot[slot]) = it;
        mbar_arrive(&C.it_full[slot]);
        if (it < 0) break;
      }
    }
    __syncwarp();
  } else if (warp < kProducers) {
    // ============================================================ producer
    // warp w issues the tiles with ordinal n = w (mod kProducers): lane l gathers keys
    // 2l and 2l+1 (16 chunks of K and 16 of V each), waits for its copies,
    // fences them to the async proxy and arrives on the stage's barrier.
    const __nv_bfloat16* kc = static_cast<const __nv_bfloat16*>(a.kc);
    const __nv_bfloat16* vc = static_cast<const __nv_bfloat16*>(a.vc);
    const __nv_bfloat16* kr = static_cast<const __nv_bfloat16*>(a.kr);
    const __nv_bfloat16* vr = static_cast<const __nv_bfloat16*>(a.vr);
    int64_t n = 0, e = 0;
    bool ok = true;
    for (int64_t ei = 0; ok; ++ei) {
      const int64_t it = next_item(ei, true);
      if (it < 0) break;
      const Item I = make_item(a, it);
      if (I.nt == 0) continue;
      if (warp == 0) {            // the item's query heads, once the MMA warp has let go of the buffer
        const int qb = (int)(e % kQBufs);
        if (!mbar_wait(&C.q_empty[qb], (uint32_t)(((e / kQBufs) & 1) ^ 1), a.err)) { ok = false; break; }
        if (lane == 0) {
          mbar_arrive_expect_tx(&C.q_full[qb], kQBytes);
          const int32_t qrow = (int32_t)(I.row * a.H);
          tma_load_2d(&tm.q, &C.q_full[qb], sQ + qb * kQBytes, 0, qrow);
          tma_load_2d(&tm.q, &C.q_full[qb], sQ + qb * kQBytes + kHeads * 128, 64, qrow);
        }
      }
      for (int t = 0; t < I.nt; ++t, ++n) {
        if ((int)(n % kProducers) != warp) continue;
        if (*abort_flag) { ok = false; break; }
        const int st = (int)(n % kStages);
        if (!mbar_wait(&C.empty[st], (uint32_t)(((n / kStages) & 1) ^ 1), a.err)) {
          ok = false;
          break;
        }
        unsigned char* stage = sKV + st * kStageBytes;
        if (tm.dense_tma && (I.t_begin + t + 1) * kKeys <= I.n_comp) {
          // 64 consecutive compressed rows (dense mode): four TMA boxes; the
          // stage completes by byte count plus the warp's 32 arrivals
          if (lane == 0) {
            const int32_t y = (int32_t)((int64_t)I.b * a.N_cap + (I.t_begin + t) * kKeys);
            mbar_arrive_expect_tx(&C.full[st], kStageBytes);
            tma_load_2d(&tm.k, &C.full[st], stage, 0, y);
            tma_load_2d(&tm.k, &C.full[st], stage + kHalf, 64, y);
            tma_load_2d(&tm.v, &C.full[st], stage + 2 * kHalf, 0, y);
            tma_load_2d(&tm.v, &C.full[st], stage + 3 * kHalf, 64, y);
          } else {
            mbar_arrive(&C.full[st]);
          }
          continue;
        }
        // lane l resolves the source rows of keys 2l and 2l+1 as (row << 1 | raw),
        // -1 for a key with no row (masked: zero-filled)
        int64_t src2[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int64_t s = (I.t_begin + t) * kKeys + 2 * lane + q;
          int64_t code = -1;
          if (s < I.n_comp) {
            const int64_t j = a.gather ? (int64_t)__ldg(a.idx + I.row * a.k + s) : s;
            if (j >= 0 && j < I.nvis) code = ((int64_t)I.b * a.N_cap + j) << 1;
            else if (j != -1) set_err(a.err, SA_ERR_BOUNDS);
          } else if (s >= I.n_comp_pad && s < I.n_comp_pad + I.n_win) {
            const int64_t u = (int64_t)I.p - I.n_win + 1 + (s - I.n_comp_pad);
            code = (((int64_t)I.b * a.R + u % a.R) << 1) | 1;
          }
          src2[q] = code;
        }
        // then the warp copies two keys per instruction: half-warp h takes key
        // 2p + h of pair p, lane l its 16-byte chunk l % 16 -- each instruction
        // reads two whole 256-byte rows, so the memory system sees four full
        // lines instead of 32 scattered sectors
        const uint32_t kd = smem_u32(stage), vd = smem_u32(stage) + 2 * kHalf;
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
        mbar_arrive(&C.full[st]);
      }
      ++e;
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    if (!ok) *abort_flag = 1;
  } else if (warp == kMmaWarp) {
    // ================================================================= MMA
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16(kHeads, kKeys, 0, 0);
      constexpr uint32_t idO = idesc_bf16(kHeads, kD, 0, 1);
      int64_t n = 0, e = 0;
      bool ok = true;
      // PV of tile ordinal m (item-local t) into O buffer ob
      auto pv = [&](int64_t m, int t, int ob, int64_t e_item) -> bool {
        const int pb = (int)(m & 1);
        if (!mbar_wait(&C.p_full[pb], (uint32_t)((m >> 1) & 1), a.err)) return false;
        if (t == 0 &&
            !mbar_wait(&C.o_empty[ob], (uint32_t)(((e_item / kOBufs) & 1) ^ 1), a.err))
          return false;
        tc_fence_after();
        const uint32_t pa = smem_u32(sP + pb * kPBytes);
        const uint32_t va = smem_u32(sKV + (m % kStages) * kStageBytes) + 2 * kHalf;
        const uint32_t tO = tmem + 128 + ob * 128;
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk)
          tc_mma_f16(tO, sdesc_kmajor_sw128(pa + kk * 32),
                     sdesc_mnmajor_sw128(va + kk * 2048, kHalf, 1024), idO,
                     (t > 0 || kk > 0) ? 1u : 0u);
        tc_commit(&C.empty[m % kStages]);
        tc_commit(&C.p_empty[pb]);
        return true;
      };
      for (int64_t ei = 0; ok; ++ei) {
        const int64_t it = next_item(ei, false);
        if (it < 0) break;
        const Item I = make_item(a, it);
        if (I.nt == 0) continue;
        const int qb = (int)(e % kQBufs), ob = (int)(e % kOBufs);
        const uint32_t qa = smem_u32(sQ + qb * kQBytes);
        if (!mbar_wait(&C.q_full[qb], (uint32_t)((e / kQBufs) & 1), a.err)) { ok = false; break; }
        for (int t = 0; t < I.nt; ++t, ++n) {
          if (*abort_flag) { ok = false; break; }
          const int st = (int)(n % kStages), sb = (int)(n & 1);
          if (!mbar_wait(&C.full[st], (uint32_t)((n / kStages) & 1), a.err) ||
              !mbar_wait(&C.s_empty[sb], (uint32_t)(((n >> 1) & 1) ^ 1), a.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t ka = smem_u32(sKV + st * kStageBytes);
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk)
            tc_mma_f16(tmem + sb * 64,
                       sdesc_kmajor_sw128(qa + (kk >> 2) * (kHeads * 128) + (kk & 3) * 32),
                       sdesc_kmajor_sw128(ka + (kk >> 2) * kHalf + (kk & 3) * 32), idS,
                       kk > 0 ? 1u : 0u);
          tc_commit(&C.s_full[sb]);
          if (t == I.nt - 1) tc_commit(&C.q_empty[qb]);
          if (t > 0 && !pv(n - 1, t - 1, ob, e)) { ok = false; break; }
        }
        if (!ok) break;
        if (!pv(n - 1, I.nt - 1, ob, e)) { ok = false; break; }
        ++e;
      }
      if (!ok) *abort_flag = 1;
    }
    __syncwarp();
  } else {
    // ============================================================= softmax
    // S and O are read with the 16x256b TMEM shape: lane l holds heads
    // h0 = 16q + l/4 and h1 = h0 + 8 (q = this warp's TMEM quarter), keys
    // 8g + 2(l%4) and +1 of every 8-key group g.  The four lanes of a head
    // pair reduce the row max with two shuffles; each lane keeps a partial
    // row sum, reduced once at the end of the item.
    const int quad = warp & 3;
    const int l4 = lane & 3;
    const int h0 = quad * 16 + (lane >> 2), h1 = h0 + 8;
    const bool ok0 = h0 < a.H, ok1 = h1 < a.H;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const float c2 = a.sm_scale * 1.4426950408889634f;   // natural logits -> log2 units
    int64_t n = 0, e = 0;
    bool ok = true;
    for (int64_t ei = 0;; ++ei) {
      const int64_t it = next_item(ei, true);
      if (it < 0) break;
      const Item I = make_item(a, it);
      // a split partial (f32) or the row's output (f32 or bf16): element offset
      // `off` of the row's [H, d] block, two consecutive columns at a time
      const bool part = a.nsplit > 1;
      const bool o16 = !part && a.o_dtype == SA_BF16;
      float* out_o = part ? a.part_o + (I.row * a.nsplit + I.split) * a.H * kD
                          : static_cast<float*>(a.o) + I.row * a.H * kD;
      __nv_bfloat16* out_o16 = static_cast<__nv_bfloat16*>(a.o) + I.row * a.H * kD;
      auto put2 = [&](int off, float x, float y) {
        if (o16) *reinterpret_cast<__nv_bfloat162*>(out_o16 + off) = __floats2bfloat162_rn(x, y);
        else *reinterpret_cast<float2*>(out_o + off) = make_float2(x, y);
      };
      float* out_l = part ? a.part_lse + (I.row * a.nsplit + I.split) * a.H
                          : a.lse + I.row * a.H;
      if (I.nt == 0 || !ok) {                      // no keys (or stopped): empty result
#pragma unroll 4
        for (int g = 0; g < kD / 8; ++g) {
          const int col = 8 * g + 2 * l4;
          if (ok0) put2(h0 * kD + col, 0.f, 0.f);
          if (ok1) put2(h1 * kD + col, 0.f, 0.f);
        }
        if (l4 == 0 && ok0) out_l[h0] = -INFINITY;
        if (l4 == 0 && ok1) out_l[h1] = -INFINITY;
        continue;
      }
      const int ob = (int)(e % kOBufs);
      float m0 = -INFINITY, m1 = -INFINITY;        // running max (log2 units), per head
      float l0 = 0.f, l1 = 0.f;                    // this lane's share of the running sums
      for (int t = 0; t < I.nt && ok; ++t, ++n) {
        // (before the wait for S: the index loads overlap it) key i of the tile
        // is real iff it is a selected row naming a visible entry (a -1 or
        // out-of-range index is ignored: its zero-filled tile row must not
        // enter the softmax) or a window row.  Lane l tests keys 2l and 2l+1;
        // two ballots give the tile's even and odd keys, and this lane keeps
        // the bits of its keys 8g + 2(l%4) + j as bit 2g + j of keep16.
        const int64_t s0 = (I.t_begin + t) * kKeys;
        auto is_real = [&](int64_t sk) -> bool {
          if (sk < I.n_comp) {
            if (!a.gather) return true;
            const int64_t jj = __ldg(a.idx + I.row * a.k + sk);
            return jj >= 0 && jj < I.nvis;
          }
          return sk >= I.n_comp_pad && sk < I.n_comp_pad + I.n_win;
        };
        const uint32_t re = __ballot_sync(0xffffffffu, is_real(s0 + 2 * lane));
        const uint32_t ro = __ballot_sync(0xffffffffu, is_real(s0 + 2 * lane + 1));
        uint32_t keep16 = 0;
#pragma unroll
        for (int g = 0; g < 8; ++g)
          keep16 |= (((re >> (4 * g + l4)) & 1u) << (2 * g)) |
                    (((ro >> (4 * g + l4)) & 1u) << (2 * g + 1));
        const int sb = (int)(n & 1), pb = (int)(n & 1);
        ok = __all_sync(0xffffffffu, mbar_wait(&C.s_full[sb], (uint32_t)((n >> 1) & 1), a.err));
        if (!ok) break;
        tc_fence_after();
        float v[32];                               // group g: h0 keys k, k+1; h1 keys k, k+1
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
        float x0 = -INFINITY, x1 = -INFINITY;      // max of the raw logits (c2 > 0)
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
        auto raise = [&](float mt, float& m, float& al) {
          if (mt > m) {
            if (m == -INFINITY) {
              m = mt;                               // O of this item holds nothing yet
            } else if (mt > m + kRescaleThreshold) {
              al = fast_exp2(m - mt);
              m = mt;
              need = true;
            }
          }
        };
        raise(x0 * c2, m0, al0);
        raise(x1 * c2, m1, al1);
        if (__any_sync(0xffffffffu, need)) {
          // rescale O after PV(n-1), which signals p_empty of its P buffer (the
          // wait at tile n-1 already covered PV(n-3) on that barrier)
          ok = __all_sync(0xffffffffu, mbar_wait(&C.p_empty[(n - 1) & 1],
                                                 (uint32_t)(((n - 1) >> 1) & 1), a.err));
          if (!ok) break;
          tc_fence_after();
          const uint32_t tO = tmem + lane_base + 128 + ob * 128;
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
          // exp2(c2 * v - m): masked keys (-inf) give +0; with nothing real
          // so far m is -inf and every v is -inf
          unsigned char* prow = sP + pb * kPBytes + 4 * l4;
          const float r0 = m0 == -INFINITY ? 0.f : m0, r1 = m1 == -INFINITY ? 0.f : m1;
          float s0 = 0.f, s1 = 0.f;
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            const __nv_bfloat162 p0 = __floats2bfloat162_rn(fast_exp2(fmaf(v[4 * g], c2, -r0)),
                                                            fast_exp2(fmaf(v[4 * g + 1], c2, -r0)));
            const __nv_bfloat162 p1 = __floats2bfloat162_rn(fast_exp2(fmaf(v[4 * g + 2], c2, -r1)),
                                                            fast_exp2(fmaf(v[4 * g + 3], c2, -r1)));
            s0 += __low2float(p0) + __high2float(p0);
            s1 += __low2float(p1) + __high2float(p1);
            *reinterpret_cast<__nv_bfloat162*>(prow + swz(h0, g)) = p0;
            *reinterpret_cast<__nv_bfloat162*>(prow + swz(h1, g)) = p1;
          }
          l0 += s0;
          l1 += s1;
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&C.p_full[pb]);
      }
      // ---- end of item: O = all PVs of the item (PV(n-1) signals p_empty)
      if (ok)
        ok = __all_sync(0xffffffffu, mbar_wait(&C.p_empty[(n - 1) & 1],
                                               (uint32_t)(((n - 1) >> 1) & 1), a.err));
      tc_fence_after();
      l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
      l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
      l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
      l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
      const bool have0 = ok && l0 > 0.f, have1 = ok && l1 > 0.f;
      const float inv0 = have0 ? 1.f / l0 : 0.f, inv1 = have1 ? 1.f / l1 : 0.f;
      const uint32_t tO = tmem + lane_base + 128 + ob * 128;
#pragma unroll 1
      for (int c = 0; c < kD; c += 32) {
        float o[16];
        tmem_ld16x256b_x4(tO + c, o);
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const int col = c + 8 * g + 2 * l4;
          if (ok0) put2(h0 * kD + col, o[4 * g] * inv0, o[4 * g + 1] * inv0);
          if (ok1) put2(h1 * kD + col, o[4 * g + 2] * inv1, o[4 * g + 3] * inv1);
        }
      }
      if (l4 == 0 && ok0) out_l[h0] = have0 ? (m0 + log2f(l0)) * 0.6931471805599453f : -INFINITY;
      if (l4 == 0 && ok1) out_l[h1] = have1 ? (m1 + log2f(l1)) * 0.6931471805599453f : -INFINITY;
      tc_fence_before();
      mbar_arrive(&C.o_empty[ob]);
      ++e;
    }
    if (!ok) *abort_flag = 1;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
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

// bf16 matrix [rows, 128] (256-byte rows), box 64 columns x box_rows rows,
// 128-byte swizzle, zero fill out of range.
static bool tmap_rows128(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows) {
  auto enc = encode_fn();
  if (!enc || rows == 0) return false;
  cuuint64_t dims[2] = {128, rows};
  cuuint64_t strides[1] = {256};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool attend_tc_supported(const AttnArgs& a) {
  return a.dtype == SA_BF16 && a.d == kD && a.H >= 1 && a.H <= kHeads;
}

int attend_tc_items_per_sm() { return 2; }

template <class Sh>
static size_t attend_tc_smem() {
  return sizeof(Ctl) + 1024 + kQBufs * kQBytes + Sh::kStages * kStageBytes + 2 * kPBytes;
}
static_assert(sizeof(Ctl) + 1024 + kQBufs * kQBytes + DeepShape::kStages * kStageBytes +
                      2 * kPBytes <= 232448,
              "the deep pipeline fits the 227 KB of shared memory a block may have");
static_assert(2 * (sizeof(Ctl) + 1024 + kQBufs * kQBytes + ShallowShape::kStages * kStageBytes +
                   2 * kPBytes) <= 233472,
              "two shallow pipelines fit one SM");

template <class Sh>
static cudaError_t launch_shape(const TMaps& tm, const AttnArgs& a, int64_t items, int num_sms,
                                cudaStream_t st) {
  const size_t smem = attend_tc_smem<Sh>();
  cudaError_t e = cudaFuncSetAttribute(attend_tc_kernel<Sh>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int grid = (int)min64((int64_t)Sh::kCtasPerSm * num_sms, items);
  attend_tc_kernel<Sh><<<grid, Sh::kThreads, smem, st>>>(tm, a);
  return cudaGetLastError();
}

cudaError_t launch_attend_tc(const AttnArgs& a, int num_sms, cudaStream_t st) {
  const int64_t items = (int64_t)a.B * a.T * a.nsplit;
  if (items == 0) return cudaSuccess;
  if (a.split_tiles > kAttnTcMaxSplitTiles) return cudaErrorInvalidValue;
  TMaps tm;
  if (!tmap_rows128(&tm.q, a.q, (uint64_t)a.B * a.T * a.H, kHeads)) return cudaErrorInvalidValue;
  // dense mode reads runs of consecutive compressed rows: by TMA where the
  // caches admit a tensor map (16-byte aligned base)
  const uint64_t crow = (uint64_t)a.B * a.N_cap;
  tm.dense_tma = !a.gather && crow > 0 && tmap_rows128(&tm.k, a.kc, crow, kKeys) &&
                 tmap_rows128(&tm.v, a.vc, crow, kKeys);
  // many items (a prefill chunk): one deep pipeline per SM; a decode step's
  // few short items: two shallow ones
  return items >= kAttnDeepItemsPerSm * (int64_t)num_sms
             ? launch_shape<DeepShape>(tm, a, items, num_sms, st)
             : launch_shape<ShallowShape>(tm, a, items, num_sms, st);
}

}  // namespace sa
