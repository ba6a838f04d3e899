// Lightning-indexer scores on the 5th-generation tensor cores (bf16 inputs,
// fp32 accumulation in TMEM, fp32 ReLU-weighted head sum in the epilogue):
//     s[r, j] = sum_h w[r,h] * max(0, q_I[r,h,:] . Ik_c[b,j,:]),  j < n(r)
// Source: "EP 95. DeepSeek-V4 논문 읽기 — 노정석", section IDEAS (lightning indexer
// over the compressed cache) and "DeepSeek-V4 논문 읽기: 백만 토큰 컨텍스트를
// 저렴하게", section "Compressed Sparse Attention (CSA)" step 2.  The weighted ReLU
// head sum is the reading taken where the pages give no formula.
//
// The contraction is D[j, (q,h)] = Ik_c[j,:] . q_I[q,h,:] with M = 128 cache
// entries (A, streamed by TMA), N = QG*64 (the 64 indexer heads of QG queries;
// B, resident per query group) and K = 64.  Putting the heads on N keeps the
// head sum inside one TMEM lane: epilogue thread j reads its row of D and
// folds w and ReLU in fp32 -- no cross-thread reduction and no rounding of w
// into bf16 operands.
//
// Warp roles (320 threads): warp 0 = TMA producer, warp 1 = MMA issuer and
// TMEM owner, warps 2..9 = two epilogue warpgroups taking alternate tiles
// (warp w reads TMEM lanes 32*(w%4)..+31).  A stage is two consecutive tiles
// of one job, loaded by one 256-row TMA box (32 KB); decode keeps 6 stages
// (192 KB) in flight per SM: under load a copy takes microseconds to arrive,
// and the bytes in flight set the bandwidth.
// A ring of shared-memory stages holds the streamed Ik_c tiles; several TMEM
// accumulators let the epilogue of tile i overlap the MMAs of later tiles.
// Persistent grid of at most one CTA per SM; a job is (query group, chunk of
// entry tiles), and tiles past the group's causal limit are never loaded.
// With few query groups (decode) each CTA takes one contiguous run of jobs;
// with many (prefill) it takes every G-th job.
// Every wait is bounded; on a timeout the CTA records SA_ERR_DEVICE_TIMEOUT,
// drops its remaining work and still frees its TMEM.
#include <cudaTypedefs.h>

#include "kernels.cuh"
#include "score_jobs.cuh"

namespace sa {

constexpr int kScoreTcThreads = 320;
constexpr int kDI = kIdxDim;
constexpr int kHI = kIdxHeads;

template <int QG>
struct ScoreTcCfg {
  // a stage holds two consecutive tiles of one job, loaded by one TMA box of
  // 256 rows: the copy engine's cost is per request, so 32 KB requests stream
  // faster per SM than 16 KB ones
  static constexpr int kStageTiles = 2;
  static constexpr int kStages = QG == 1 ? 6 : 4;
  static constexpr int kAccCols = QG * kHI;
  static constexpr int kAccBufs = QG == 1 ? 4 : 2;
  static constexpr int kTmemCols = kAccBufs * kAccCols;       // 256 or 512
  static constexpr int kTileBytes = kTileEntries * kDI * 2;   // 16 KB
  static constexpr int kABytes = kStageTiles * kTileBytes;    // 32 KB
  static constexpr int kBBytes = QG * kHI * kDI * 2;          // 8 KB per query
  static constexpr int kWBytes = QG * kHI * 4;                // a group's head weights, f32
  static constexpr size_t kSmem = 1024 /*align slack*/ + kStages * kABytes + 2 * kBBytes +
                                  2 * kWBytes + 512 +
                                  kMaxJobsPerCta * sizeof(JobRec<QG>);
};

template <int QG>
__global__ void __launch_bounds__(kScoreTcThreads, 1)
    score_tc_kernel(const __grid_constant__ CUtensorMap tm_ik,
                    const __grid_constant__ CUtensorMap tm_q, ScoreJobs p) {
  using Cfg = ScoreTcCfg<QG>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* sA = smem;
  unsigned char* sB = sA + Cfg::kStages * Cfg::kABytes;
  // the head weights of each epilogue warpgroup's current query group
  float* sW = reinterpret_cast<float*>(sB + 2 * Cfg::kBBytes);         // [2][QG*64]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + 2 * Cfg::kBBytes + 2 * Cfg::kWBytes);
  uint64_t* full = bars;
  uint64_t* empty = full + Cfg::kStages;
  uint64_t* bfull = empty + Cfg::kStages;
  uint64_t* bempty = bfull + 2;
  uint64_t* tfull = bempty + 2;
  uint64_t* tempty = tfull + Cfg::kAccBufs;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(tempty + Cfg::kAccBufs);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
  JobRec<QG>* jobs = reinterpret_cast<JobRec<QG>*>(
      reinterpret_cast<unsigned char*>(bars) + 512);
  const int n_my = fill_job_table<QG>(p, jobs);

  const int warp = (int)warp_id(), lane = (int)lane_id();
  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::kStages; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bfull[s], 1);
      mbar_init(&bempty[s], 1);
    }
    for (int s = 0; s < Cfg::kAccBufs; ++s) {
      mbar_init(&tfull[s], 1);
      mbar_init(&tempty[s], 128);
    }
    *s_abort = 0;
    mbar_fence_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_ik);
    tma_prefetch_desc(&tm_q);
  }
  if (warp == 1) tmem_alloc(s_tmem, Cfg::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t ph = 0;
      int nsw = 0;
      int64_t prev_g = -1;
      for (int ji = 0; ji < n_my && !*s_abort; ++ji) {
        const JobRec<QG>& J = jobs[ji];
        if (J.t_lo >= J.t_hi) continue;
        if (J.g != prev_g) {
          const int slot = nsw & 1, u = nsw >> 1;
          if (!mbar_wait(&bempty[slot], (u & 1) ^ 1, p.err)) { *s_abort = 1; break; }
          mbar_arrive_expect_tx(&bfull[slot], Cfg::kBBytes);
          tma_load_2d(&tm_q, &bfull[slot], sB + slot * Cfg::kBBytes, 0,
                      (int32_t)(((int64_t)J.b * p.T + J.t0) * kHI));
          prev_g = J.g;
          ++nsw;
        }
        for (int t = J.t_lo; t < J.t_hi; t += Cfg::kStageTiles) {
          if (!mbar_wait(&empty[stage], ph ^ 1, p.err)) { *s_abort = 1; break; }
          mbar_arrive_expect_tx(&full[stage], Cfg::kABytes);
          tma_load_2d(&tm_ik, &full[stage], sA + stage * Cfg::kABytes, 0,
                      (int32_t)((int64_t)J.b * p.N_cap + (int64_t)t * kTileEntries));
          if (++stage == Cfg::kStages) { stage = 0; ph ^= 1; }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(128, Cfg::kAccCols);
      int stage = 0;
      uint32_t ph = 0;
      int acc = 0;
      uint32_t acc_ph = 0;
      int nsw = 0, slot = -1;
      int64_t prev_g = -1;
      for (int ji = 0; ji < n_my && !*s_abort; ++ji) {
        const JobRec<QG>& J = jobs[ji];
        if (J.t_lo >= J.t_hi) continue;
        if (J.g != prev_g) {
          if (slot >= 0) tc_commit(&bempty[slot]);
          slot = nsw & 1;
          const int u = nsw >> 1;
          if (!mbar_wait(&bfull[slot], u & 1, p.err)) { *s_abort = 1; break; }
          prev_g = J.g;
          ++nsw;
        }
        const uint32_t b_base = smem_u32(sB + slot * Cfg::kBBytes);
        for (int t = J.t_lo; t < J.t_hi; ++t) {
          const int half = (t - J.t_lo) % Cfg::kStageTiles;     // tile within its stage
          if (half == 0 && !mbar_wait(&full[stage], ph, p.err)) { *s_abort = 1; break; }
          if (!mbar_wait(&tempty[acc], acc_ph ^ 1, p.err)) { *s_abort = 1; break; }
          tc_fence_after();
          const uint32_t a_base = smem_u32(sA + stage * Cfg::kABytes + half * Cfg::kTileBytes);
#pragma unroll
          for (int kk = 0; kk < kDI / 16; ++kk)
            tc_mma_f16(tmem + acc * Cfg::kAccCols, sdesc_kmajor_sw128(a_base + kk * 32),
                       sdesc_kmajor_sw128(b_base + kk * 32), idesc, kk > 0 ? 1u : 0u);
          tc_commit(&tfull[acc]);
          if (half == Cfg::kStageTiles - 1 || t == J.t_hi - 1) {
            tc_commit(&empty[stage]);
            if (++stage == Cfg::kStages) { stage = 0; ph ^= 1; }
          }
          if (++acc == Cfg::kAccBufs) { acc = 0; acc_ph ^= 1; }
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    // Two warpgroups take alternate tiles (ordinal o of this CTA's tiles:
    // group o % 2, accumulator o % kAccBufs).  Each warpgroup copies the head
    // weights of a job's query group into its own shared-memory slot when the
    // group changes; the tile loop then reads them as broadcast float4s.
    const int grp = (warp - 2) >> 2;
    const int quad = warp & 3;
    const int row_in_tile = quad * 32 + lane;
    const int gtid = (warp - 2 - 4 * grp) * 32 + lane;        // 0..127 in the warpgroup
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    float* wg = sW + grp * QG * kHI;
    // Every thread walks every job, so that all 128 reach each named barrier;
    // once a wait gives up or the CTA aborts, the warp only skips its tiles.
    int64_t o = 0, prev_g = -1;
    bool stop = false;
    for (int ji = 0; ji < n_my; ++ji) {
      const JobRec<QG>& J = jobs[ji];
      if (J.t_lo >= J.t_hi) continue;
      if (J.g != prev_g) {
        named_bar_sync(1 + grp, 128);                         // the previous weights are read
        const float* wsrc = p.w + ((int64_t)J.b * p.T + J.t0) * kHI;
        for (int i = gtid; i < J.nq * kHI; i += 128) wg[i] = __ldg(wsrc + i);
        named_bar_sync(1 + grp, 128);
        prev_g = J.g;
      }
      for (int t = J.t_lo; t < J.t_hi; ++t, ++o) {
        if ((int)(o & 1) != grp) continue;
        stop = __any_sync(0xffffffffu, stop || *s_abort);
        if (stop) continue;
        const int acc = (int)(o % Cfg::kAccBufs);
        const uint32_t acc_ph = (uint32_t)((o / Cfg::kAccBufs) & 1);
        if (!__all_sync(0xffffffffu, mbar_wait(&tfull[acc], acc_ph, p.err))) {
          *s_abort = 1;
          stop = true;
          continue;
        }
        tc_fence_after();
        const int64_t j = (int64_t)t * kTileEntries + row_in_tile;
        const uint32_t tacc = tmem + lane_base + acc * Cfg::kAccCols;
#pragma unroll 1
        for (int q = 0; q < J.nq; ++q) {
          uint32_t v[64];
          tmem_ld32_async(tacc + q * kHI, v);
          tmem_ld32_async(tacc + q * kHI + 32, v + 32);
          tmem_wait_ld();
          const float4* w4 = reinterpret_cast<const float4*>(wg + q * kHI);
          float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float4 wv = w4[i];
            s0 = fmaf(wv.x, fmaxf(__uint_as_float(v[4 * i + 0]), 0.f), s0);
            s1 = fmaf(wv.y, fmaxf(__uint_as_float(v[4 * i + 1]), 0.f), s1);
            s2 = fmaf(wv.z, fmaxf(__uint_as_float(v[4 * i + 2]), 0.f), s2);
            s3 = fmaf(wv.w, fmaxf(__uint_as_float(v[4 * i + 3]), 0.f), s3);
          }
          const int64_t r = (int64_t)J.b * p.T + J.t0 + q;
          if (j < J.n[q]) p.scores[r * p.ld + j] = (s0 + s1) + (s2 + s3);
        }
        tc_fence_before();
        mbar_arrive(&tempty[acc]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::kTmemCols);
  }
}

// ---------------------------------------------------------------- host side

static PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
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

// 2-D bf16 tensor [rows, 64] (128-byte rows) with a {64, box_rows} box and the
// 128-byte swizzle expected by the K-major shared-memory descriptors.
bool make_tmap_bf16_rows64(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {64, rows};
  cuuint64_t strides[1] = {128};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool score_tc_supported(const ScoreArgs& a) {
  return a.dtype == SA_BF16 && a.HI == kHI && a.dI == kDI;
}

template <int QG>
static cudaError_t launch_qg(const ScoreArgs& a, int num_sms, cudaStream_t st) {
  using Cfg = ScoreTcCfg<QG>;
  CUtensorMap tm_ik, tm_q;
  if (!make_tmap_bf16_rows64(&tm_ik, a.ik, (uint64_t)a.B * a.N_cap,
                             Cfg::kStageTiles * kTileEntries) ||
      !make_tmap_bf16_rows64(&tm_q, a.q, (uint64_t)a.B * a.T * kHI, QG * kHI))
    return cudaErrorInvalidValue;
  ScoreJobs p{};
  p.w = a.w;
  p.q_pos = a.q_pos;
  p.B = a.B;
  p.T = a.T;
  p.m = a.m;
  p.N_cap = a.N_cap;
  p.scores = a.scores;
  p.ld = a.ld;
  p.err = a.err;
  const int grid = plan_score_jobs(p, QG, num_sms, Cfg::kStageTiles);
  if (grid == 0) return cudaSuccess;
  if (grid < 0) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(score_tc_kernel<QG>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)Cfg::kSmem);
  if (e != cudaSuccess) return e;
  score_tc_kernel<QG><<<grid, kScoreTcThreads, Cfg::kSmem, st>>>(tm_ik, tm_q, p);
  return cudaGetLastError();
}

cudaError_t launch_score_tc(const ScoreArgs& a, int num_sms, cudaStream_t st) {
  if (a.T >= 4) return launch_qg<4>(a, num_sms, st);
  return launch_qg<1>(a, num_sms, st);
}

}  // namespace sa
