// Lightning-indexer scores from MXFP4 indexer keys and queries, dequantised
// in-kernel to FP8 (e4m3) and contracted on the 5th-generation tensor cores
// (tcgen05 kind::f8f6f4, fp32 accumulation in TMEM).
//
// Source: "오픈소스 LLM의 새 이정표: DeepSeek-V4 시리즈", section "오픈소스 MoE
// 인프라: MegaMoE와 TileLang": the indexer QK path is stored in FP4 (MXFP4) and
// dequantised to FP8 without loss.  MXFP4 as in the OCP Microscaling Formats
// (MX) v1.0 specification: e2m1 elements, one e8m0 scale per 32 elements.
//
// Lossless FP4 -> FP8.  An element is c * 2^(e_b) with c on the e2m1 grid
// {0, .5, 1, 1.5, 2, 3, 4, 6} and e_b its block's exponent.  Each 64-wide row
// has two blocks; with e_row = max(e_0, e_1) the kernel stores
// c * 2^(e_b - e_row) in e4m3, which is exact while e_row - e_b <= 8 (e4m3's
// smallest subnormal is 2^-9), and applies 2^(e_row) in fp32 after the MMA:
//     q.k = 2^(e_row(q) + e_row(k)) * (q' . k')
// and, as 2^x > 0 commutes with ReLU,
//     s[r, j] = 2^(e_row(k_j)) * sum_h (w[r,h] * 2^(e_row(q_h))) * ReLU(q'_h . k'_j)
// (rows whose blocks differ by more than 8 exponents round the small block to
// the nearest e4m3 value).
//
// Work moves through the CTA in steps of kS consecutive 128-entry tiles of
// one job (kS = 4 for one query per group, 1 for four): one bulk load, one A
// stage, kS MMAs into one accumulator, one epilogue pass.  Every hand-off
// between roles costs a barrier round trip, so at decode, where a tile is only
// 4.3 KB of MXFP4, steps of four tiles spread those round trips over 17 KB
// (measured: 45 -> 33 us at the 128K decode shape).
//
// Warp roles (448 threads): warp 0 = bulk-copy producer (raw codes + scales
// of a step, 34 bytes per entry, into a ring of raw stages), warp 1 = MMA
// issuer and TMEM owner, then 12 worker warps:
//   converters -- one warpgroup at decode (a thread turns entry row c of each
//     tile of the step from e2m1 into e4m3), two warpgroups at prefill (each
//     takes one 32-element block of the row); the output is a K-major tile
//     with 64-byte swizzled rows; the row's factor 2^(e_row) goes to the
//     epilogue through a ring, so a raw stage is free as soon as it is
//     converted; together they also convert each query group's B tile;
//   epilogue -- two warpgroups at decode, taking alternate tiles of a step,
//     one at prefill: one entry row per thread, weighted ReLU head sum as in
//     the bf16 kernel; each warp keeps its query weights, with the row
//     exponents folded in, in shared memory.
// Every role takes the steps in order, so each ring slot's previous user is
// the same role one lap earlier and every parity wait is at most one phase
// away.  Every wait is bounded; on a timeout the CTA records
// SA_ERR_DEVICE_TIMEOUT, stops and still frees its TMEM.
#include <cuda_fp8.h>

#include "kernels.cuh"
#include "score_jobs.cuh"

namespace sa {

namespace {

constexpr int kMxThreads = 448;
constexpr int kCodeRowBytes = kIdxDim / 2;                       // 32
constexpr int kScaleRowBytes = kIdxDim / 32;                     // 2
constexpr int kARowBytes = 64;                                   // A: 64B-swizzled rows
constexpr int kABytes = kTileEntries * kARowBytes;               // 8 KB per tile
constexpr int kBRowBytes = 128;                                  // B: 128B-swizzled (64 used)

template <int QG>
struct MxCfg {
  static constexpr int kS = QG == 1 ? 4 : 1;                      // tiles per step
  // 12 worker warps: converters (whole rows with one warpgroup, one block of
  // each row per warpgroup with two) and epilogue warpgroups (each taking
  // every kEpiGroups-th tile of a step)
  static constexpr int kConvWarps = QG == 1 ? 4 : 8;
  static constexpr int kEpiWarps = 12 - kConvWarps;
  static constexpr int kStepEntries = kS * kTileEntries;
  static constexpr int kRawCodeBytes = kStepEntries * kCodeRowBytes;
  static constexpr int kRawBytes = kStepEntries * (kCodeRowBytes + kScaleRowBytes);
  static constexpr int kRawStages = QG == 1 ? 6 : 12;
  static constexpr int kAStages = QG == 1 ? 2 : 4;
  static constexpr int kAStepBytes = kS * kABytes;
  static constexpr int kAccCols = QG * kIdxHeads;                 // one tile's accumulator
  static constexpr int kAccBufs = 2;
  static constexpr int kTmemCols = kAccBufs * kS * kAccCols;      // 512
  // Key-row factors 2^(e_row) pass from the converters to the epilogue through
  // a ring of kKsSlots steps.  The converters reach step k only after the MMA
  // of step k - kAStages, which waited for the epilogue to finish step
  // k - kAStages - kAccBufs, so that many slots are never overwritten unread.
  static constexpr int kKsSlots = kAStages + kAccBufs;
  static constexpr int kBBytes = QG * kIdxHeads * kBRowBytes;    // 8 KB per query
  static constexpr size_t kWqBytes = kEpiWarps * QG * kIdxHeads * sizeof(float);
  static constexpr size_t kKsBytes = (size_t)kKsSlots * kStepEntries * sizeof(float);
  static constexpr size_t kSmem = 1024 + (size_t)kAStages * kAStepBytes + 2 * kBBytes +
                                  (size_t)kRawStages * kRawBytes + 1024 /* LUT + barriers */ +
                                  kMaxJobsPerCta * sizeof(JobRec<QG>) + kWqBytes + kKsBytes;
  static_assert(kRawBytes % 16 == 0 && kRawCodeBytes % 16 == 0, "bulk copies need 16 B");
  static_assert(kABytes % 512 == 0 && kBBytes % 1024 == 0, "swizzle atoms: 512 B (A), 1 KB (B)");
  static_assert(kTmemCols <= 512, "TMEM");
  static_assert(kSmem <= 227 * 1024, "shared memory per CTA");
};

struct MxPtrs {
  const uint8_t* q_codes;    // [B*T, 64, 32]
  const uint8_t* q_scales;   // [B*T, 64, 2]
  const uint8_t* k_codes;    // [B, N_cap, 32]
  const uint8_t* k_scales;   // [B, N_cap, 2]
};

// Shared-memory descriptor of a K-major operand with 64-byte swizzle: rows of
// 64 bytes (K = 64 8-bit values), the 16-byte chunk c of row r stored at chunk
// c ^ ((r >> 1) & 3), 8-row groups 512 B apart; the tile is 512-byte aligned.
__device__ __forceinline__ uint64_t sdesc_kmajor_sw64(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr >> 4) & 0x3FFFu);        // start address
  d |= (uint64_t)1u << 16;                        // leading byte offset (unused here)
  d |= (uint64_t)(512u >> 4) << 32;               // stride byte offset: 8 rows * 64 B
  d |= (uint64_t)1u << 46;                        // descriptor version (sm_100 family)
  d |= (uint64_t)4u << 61;                        // swizzle: 64 B
  return d;
}

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// e4m3 byte for e2m1 magnitude code c (0..7) times 2^-s, s = 0..15 (round to
// nearest even where the product is not an e4m3 value, i.e. only for s > 8).
__device__ __forceinline__ uint8_t e4m3_of(int c, int s) {
  const float mag[8] = {0.f, 0.5f, 1.f, 1.5f, 2.f, 3.f, 4.f, 6.f};
  return (uint8_t)__nv_cvt_float_to_fp8(ldexpf(mag[c], -s), __NV_SATFINITE, __NV_E4M3);
}

// Eight e2m1 codes (one 32-bit word, element 2i in the low nibble of byte i)
// -> eight e4m3 bytes, using an 8-entry magnitude table (lut_lo: codes 0-3,
// lut_hi: codes 4-7; every byte's top bit clear) for the block's shift.  The
// code's sign bit (bit 3 of its nibble) becomes a byte-permute selector, 0 or
// 4, into (0x00000000, 0x80808080): the e4m3 sign bit of that output byte.
__device__ __forceinline__ uint2 e2m1x8_to_e4m3(uint32_t w, uint32_t lut_lo, uint32_t lut_hi) {
  const uint32_t mag_lo = __byte_perm(lut_lo, lut_hi, w & 0x7777u);
  const uint32_t mag_hi = __byte_perm(lut_lo, lut_hi, (w >> 16) & 0x7777u);
  const uint32_t sg_lo = __byte_perm(0u, 0x80808080u, (w >> 1) & 0x4444u);
  const uint32_t sg_hi = __byte_perm(0u, 0x80808080u, (w >> 17) & 0x4444u);
  return make_uint2(mag_lo | sg_lo, mag_hi | sg_hi);
}

// Convert block h (elements 32h..32h+31, code bytes 16h..16h+15) of one
// 64-element MXFP4 row, given both of the row's scale bytes, into e4m3 bytes
// 32h..32h+31 of row r of a K-major tile with kRowBytes-byte swizzled rows
// (128: chunk c at c ^ (r & 7); 64: chunk c at c ^ ((r >> 1) & 3)); returns
// e_row.
template <int kRowBytes>
__device__ __forceinline__ int convert_half(uint4 cw, uint32_t sc0, uint32_t sc1, int h,
                                            const uint32_t* lut, unsigned char* tile, int r) {
  const int e0 = (int)sc0 - 127, e1 = (int)sc1 - 127;
  const int er = max(e0, e1);
  const int sh = min(er - (h ? e1 : e0), 15);
  const uint32_t la = lut[2 * sh], lb = lut[2 * sh + 1];
  const uint2 a0 = e2m1x8_to_e4m3(cw.x, la, lb), a1 = e2m1x8_to_e4m3(cw.y, la, lb);
  const uint2 a2 = e2m1x8_to_e4m3(cw.z, la, lb), a3 = e2m1x8_to_e4m3(cw.w, la, lb);
  unsigned char* row = tile + r * kRowBytes;
  const int x = kRowBytes == 128 ? (r & 7) : ((r >> 1) & 3);
  *reinterpret_cast<uint4*>(row + (((2 * h) ^ x) << 4)) = make_uint4(a0.x, a0.y, a1.x, a1.y);
  *reinterpret_cast<uint4*>(row + (((2 * h + 1) ^ x) << 4)) = make_uint4(a2.x, a2.y, a3.x, a3.y);
  return er;
}

// sum_i w[i] * ReLU(v[i]) over 32 columns of fp32 accumulators.
__device__ __forceinline__ float relu_dot32(const uint32_t* v, const float* w) {
  const float4* w4 = reinterpret_cast<const float4*>(w);
  float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 wv = w4[i];
    s0 = fmaf(wv.x, fmaxf(__uint_as_float(v[4 * i + 0]), 0.f), s0);
    s1 = fmaf(wv.y, fmaxf(__uint_as_float(v[4 * i + 1]), 0.f), s1);
    s2 = fmaf(wv.z, fmaxf(__uint_as_float(v[4 * i + 2]), 0.f), s2);
    s3 = fmaf(wv.w, fmaxf(__uint_as_float(v[4 * i + 3]), 0.f), s3);
  }
  return (s0 + s1) + (s2 + s3);
}

__device__ __forceinline__ float pow2i(int e) {
  e = max(-126, min(127, e));
  return __int_as_float((e + 127) << 23);
}

// Head weights of query row r with its per-head row exponents folded in,
// wq[h] = w[r,h] * 2^(max block exponent of q_I[r,h,:]), written by the 32
// lanes of a warp (two heads each) to that warp's 64 floats of shared memory.
__device__ __forceinline__ void store_wq(const ScoreJobs& p, const MxPtrs& x, int64_t r,
                                         float* dst) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int h = lane + 32 * u;
    const uint8_t* qs = x.q_scales + (r * kIdxHeads + h) * 2;
    dst[h] = __ldg(p.w + r * kIdxHeads + h) * pow2i(max((int)__ldg(qs), (int)__ldg(qs + 1)) - 127);
  }
  __syncwarp();
}

}  // namespace

template <int QG>
__global__ void __launch_bounds__(kMxThreads, 1) score_mx_kernel(ScoreJobs p, MxPtrs x) {
  using Cfg = MxCfg<QG>;
  constexpr int kS = Cfg::kS;
  constexpr int kRawStages = Cfg::kRawStages;
  constexpr int kAStages = Cfg::kAStages;
  constexpr int kAccBufs = Cfg::kAccBufs;
  constexpr int kKsSlots = Cfg::kKsSlots;
  constexpr int kConvWarps = Cfg::kConvWarps;
  constexpr int kConvThreads = 32 * kConvWarps;
  constexpr int kEpiThreads = 32 * Cfg::kEpiWarps;
  constexpr int kHalves = 8 / kConvWarps;                          // blocks per row per thread
  constexpr int kEpiGroups = Cfg::kEpiWarps / 4;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* sA = smem;                                        // [kAStages][kS][128][128]
  unsigned char* sB = sA + kAStages * Cfg::kAStepBytes;            // [2][QG*64][128]
  unsigned char* sRaw = sB + 2 * Cfg::kBBytes;                     // [kRawStages] codes, scales
  uint32_t* lut = reinterpret_cast<uint32_t*>(sRaw + kRawStages * Cfg::kRawBytes);   // [16][2]
  uint64_t* bars = reinterpret_cast<uint64_t*>(lut + 32);
  uint64_t* raw_full = bars;
  uint64_t* raw_empty = raw_full + kRawStages;
  uint64_t* a_full = raw_empty + kRawStages;
  uint64_t* a_empty = a_full + kAStages;
  uint64_t* b_full = a_empty + kAStages;
  uint64_t* b_empty = b_full + 2;
  uint64_t* t_full = b_empty + 2;
  uint64_t* t_empty = t_full + kAccBufs;
  uint64_t* ks_full = t_empty + kAccBufs;                          // [kKsSlots]
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(ks_full + kKsSlots);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
  JobRec<QG>* jobs = reinterpret_cast<JobRec<QG>*>(reinterpret_cast<unsigned char*>(lut) + 1024);
  float* s_wq = reinterpret_cast<float*>(jobs + kMaxJobsPerCta);   // [kEpiWarps][QG][64]
  float* s_ks = s_wq + Cfg::kEpiWarps * QG * kIdxHeads;             // [kKsSlots][kS*128]

  const int n_my = fill_job_table<QG>(p, jobs);
  const int warp = (int)warp_id(), lane = (int)lane_id();
  if (threadIdx.x < 128) {                  // magnitude tables for shifts 0..15
    const int s = threadIdx.x >> 3, c = threadIdx.x & 7;
    reinterpret_cast<uint8_t*>(lut)[s * 8 + c] = e4m3_of(c, s);
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kRawStages; ++s) {
      mbar_init(&raw_full[s], 1);
      mbar_init(&raw_empty[s], kConvThreads);
    }
    for (int s = 0; s < kKsSlots; ++s) mbar_init(&ks_full[s], kConvThreads);
    for (int s = 0; s < kAStages; ++s) {
      mbar_init(&a_full[s], kConvThreads);
      mbar_init(&a_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) { mbar_init(&b_full[s], kConvThreads); mbar_init(&b_empty[s], 1); }
    for (int s = 0; s < kAccBufs; ++s) { mbar_init(&t_full[s], 1); mbar_init(&t_empty[s], kEpiThreads); }
    *s_abort = 0;
    mbar_fence_init();
  }
  if (warp == 1) tmem_alloc(s_tmem, Cfg::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;

  // Every role walks the same steps: job by job, kS tiles at a time (fewer
  // at the end of a job).
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t ph = 0;
      for (int ji = 0; ji < n_my && !*s_abort; ++ji) {
        const JobRec<QG>& J = jobs[ji];
        for (int t = J.t_lo; t < J.t_hi; t += kS) {
          if (!mbar_wait(&raw_empty[stage], ph ^ 1, p.err)) { *s_abort = 1; break; }
          // the step's tiles are consecutive entries of sequence b; the last
          // tile of a sequence may be partial (N_cap is a multiple of 8, so
          // every copy stays a multiple of 16 bytes)
          const int nsub = min(kS, J.t_hi - t);
          const int64_t e0 = (int64_t)J.b * p.N_cap + (int64_t)t * kTileEntries;
          const uint32_t rows = (uint32_t)min64((int64_t)nsub * kTileEntries,
                                                (int64_t)p.N_cap - (int64_t)t * kTileEntries);
          unsigned char* dst = sRaw + stage * Cfg::kRawBytes;
          mbar_arrive_expect_tx(&raw_full[stage], rows * (kCodeRowBytes + kScaleRowBytes));
          bulk_g2s(dst, x.k_codes + e0 * kCodeRowBytes, rows * kCodeRowBytes, &raw_full[stage]);
          bulk_g2s(dst + Cfg::kRawCodeBytes, x.k_scales + e0 * kScaleRowBytes,
                   rows * kScaleRowBytes, &raw_full[stage]);
          if (++stage == kRawStages) { stage = 0; ph ^= 1; }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_e4m3(128, Cfg::kAccCols);
      int stage = 0, acc = 0, nsw = 0, slot = -1;
      uint32_t ph = 0, acc_ph = 0;
      int64_t prev_g = -1;
      for (int ji = 0; ji < n_my && !*s_abort; ++ji) {
        const JobRec<QG>& J = jobs[ji];
        if (J.t_lo >= J.t_hi) continue;
        if (J.g != prev_g) {
          if (slot >= 0) tc_commit(&b_empty[slot]);
          slot = nsw & 1;
          if (!mbar_wait(&b_full[slot], (nsw >> 1) & 1, p.err)) { *s_abort = 1; break; }
          prev_g = J.g;
          ++nsw;
        }
        const uint32_t b_base = smem_u32(sB + slot * Cfg::kBBytes);
        for (int t = J.t_lo; t < J.t_hi; t += kS) {
          const int nsub = min(kS, J.t_hi - t);
          if (!mbar_wait(&a_full[stage], ph, p.err)) { *s_abort = 1; break; }
          if (!mbar_wait(&t_empty[acc], acc_ph ^ 1, p.err)) { *s_abort = 1; break; }
          tc_fence_after();
          const uint32_t a_base = smem_u32(sA + stage * Cfg::kAStepBytes);
          const uint32_t d_base = tmem + (uint32_t)(acc * kS * Cfg::kAccCols);
#pragma unroll
          for (int s = 0; s < kS; ++s) {
            if (s >= nsub) break;
#pragma unroll
            for (int kk = 0; kk < 2; ++kk)        // K = 64 e4m3 = two MMAs of K = 32
              tc_mma_f8f6f4(d_base + (uint32_t)(s * Cfg::kAccCols),
                            sdesc_kmajor_sw64(a_base + s * kABytes + kk * 32),
                            sdesc_kmajor_sw128(b_base + kk * 32), idesc, kk > 0 ? 1u : 0u);
          }
          tc_commit(&a_empty[stage]);
          tc_commit(&t_full[acc]);
          if (++stage == kAStages) { stage = 0; ph ^= 1; }
          if (++acc == kAccBufs) { acc = 0; acc_ph ^= 1; }
        }
      }
    }
    __syncwarp();
  } else if (warp < 2 + kConvWarps) {
    // ---------------------------------------------------------- converters
    const int tc = (int)threadIdx.x - 64;       // 0 .. kConvThreads - 1
    const int c = tc & 127;                     // entry row within a tile
    const int h0 = tc >> 7;                     // first block of the row taken: 32*h0 ..
    int nsw = 0;
    int64_t k = 0;                              // step ordinal
    int64_t prev_g = -1;
    for (int ji = 0; ji < n_my && !*s_abort; ++ji) {
      const JobRec<QG>& J = jobs[ji];
      if (J.t_lo >= J.t_hi) continue;
      bool stop = false;
      if (J.g != prev_g) {
        // the query group's B tile: QG*64 rows (query q, head h), two blocks
        // each, zero past nq
        const int slot = nsw & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(&b_empty[slot], ((nsw >> 1) & 1) ^ 1, p.err))) {
          *s_abort = 1;
          break;
        }
        unsigned char* tile = sB + slot * Cfg::kBBytes;
        for (int it = tc; it < QG * kIdxHeads * 2; it += kConvThreads) {
          const int rr = it >> 1, hh = it & 1;
          const int q = rr / kIdxHeads;
          if (q < J.nq) {
            const int64_t qrow = ((int64_t)J.b * p.T + J.t0 + q) * kIdxHeads + (rr % kIdxHeads);
            const uint4* src = reinterpret_cast<const uint4*>(x.q_codes + qrow * kCodeRowBytes);
            convert_half<kBRowBytes>(__ldg(src + hh), x.q_scales[qrow * 2],
                                     x.q_scales[qrow * 2 + 1], hh, lut, tile, rr);
          } else {
            unsigned char* row = tile + rr * kBRowBytes;
            *reinterpret_cast<uint4*>(row + (((2 * hh) ^ (rr & 7)) << 4)) = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(row + (((2 * hh + 1) ^ (rr & 7)) << 4)) =
                make_uint4(0, 0, 0, 0);
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(&b_full[slot]);
        ++nsw;
        prev_g = J.g;
      }
      for (int t = J.t_lo; t < J.t_hi; t += kS, ++k) {
        const int nsub = min(kS, J.t_hi - t);
        const int rstage = (int)(k % kRawStages), astage = (int)(k % kAStages);
        const uint32_t rph = (uint32_t)((k / kRawStages) & 1), aph = (uint32_t)((k / kAStages) & 1);
        if (!__all_sync(0xffffffffu, mbar_wait(&raw_full[rstage], rph, p.err))) {
          *s_abort = 1;
          stop = true;
          break;
        }
        // all of the step's loads first, then the stage is released
        const unsigned char* raw = sRaw + rstage * Cfg::kRawBytes;
        uint4 cw[kS][kHalves];
        uint32_t sc0[kS], sc1[kS];
#pragma unroll
        for (int s = 0; s < kS; ++s) {
          if (s < nsub) {
            const int e = s * kTileEntries + c;
#pragma unroll
            for (int i = 0; i < kHalves; ++i)
              cw[s][i] = *reinterpret_cast<const uint4*>(raw + e * kCodeRowBytes + (h0 + i) * 16);
            sc0[s] = raw[Cfg::kRawCodeBytes + 2 * e];
            sc1[s] = raw[Cfg::kRawCodeBytes + 2 * e + 1];
          }
        }
        mbar_arrive(&raw_empty[rstage]);
        if (!__all_sync(0xffffffffu, mbar_wait(&a_empty[astage], aph ^ 1, p.err))) {
          *s_abort = 1;
          stop = true;
          break;
        }
        unsigned char* a = sA + astage * Cfg::kAStepBytes;
        float* ksd = s_ks + (int)(k % kKsSlots) * Cfg::kStepEntries;
#pragma unroll
        for (int s = 0; s < kS; ++s) {
          if (s < nsub) {
            int er = 0;
#pragma unroll
            for (int i = 0; i < kHalves; ++i)
              er = convert_half<kARowBytes>(cw[s][i], sc0[s], sc1[s], h0 + i, lut,
                                            a + s * kABytes, c);
            if (h0 == 0) ksd[s * kTileEntries + c] = pow2i(er);
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(&a_full[astage]);
        mbar_arrive(&ks_full[(int)(k % kKsSlots)]);
      }
      if (stop) break;
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // Step ordinal k uses accumulator k % kAccBufs: kS tile accumulators of
    // kAccCols columns each.
    const int quad = warp & 3;
    const int row_in_tile = quad * 32 + lane;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const int eg = (warp - 2 - kConvWarps) >> 2;                   // epilogue warpgroup
    float* wq = s_wq + (warp - 2 - kConvWarps) * QG * kIdxHeads;     // this warp's weights
    int64_t k = 0;                // step ordinal (factor slot k % kKsSlots)
    int64_t wq_g = -1;            // query group whose weights are in wq
    for (int ji = 0; ji < n_my && !*s_abort; ++ji) {
      const JobRec<QG>& J = jobs[ji];
      if (J.t_lo >= J.t_hi) continue;
      if (J.g != wq_g) {          // consecutive jobs of one group reuse its weights
        __syncwarp();                                    // previous group's weights are consumed
        for (int q = 0; q < J.nq; ++q)
          store_wq(p, x, (int64_t)J.b * p.T + J.t0 + q, wq + q * kIdxHeads);
        wq_g = J.g;
      }
      bool stop = false;
      for (int t = J.t_lo; t < J.t_hi; t += kS, ++k) {
        const int nsub = min(kS, J.t_hi - t);
        const int acc = (int)(k % kAccBufs);
        // warp-uniform waits: the TMEM loads below are warp-collective
        if (!__all_sync(0xffffffffu, mbar_wait(&t_full[acc], (uint32_t)((k / kAccBufs) & 1), p.err))) {
          *s_abort = 1;
          stop = true;
          break;
        }
        // this thread's entry rows' factors 2^(e_row), from the converters' ring
        const int ks = (int)(k % kKsSlots);
        if (!__all_sync(0xffffffffu, mbar_wait(&ks_full[ks], (uint32_t)((k / kKsSlots) & 1), p.err))) {
          *s_abort = 1;
          stop = true;
          break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int s = eg; s < nsub; s += kEpiGroups) {
          const float kscale = s_ks[ks * Cfg::kStepEntries + s * kTileEntries + row_in_tile];
          const int64_t j = (int64_t)(t + s) * kTileEntries + row_in_tile;
          const uint32_t col0 = (uint32_t)((acc * kS + s) * Cfg::kAccCols);
#pragma unroll 1
          for (int q = 0; q < J.nq; ++q) {
            const int64_t r = (int64_t)J.b * p.T + J.t0 + q;
            uint32_t v[64];
            tmem_ld32_async(tmem + lane_base + col0 + q * kIdxHeads, v);
            tmem_ld32_async(tmem + lane_base + col0 + q * kIdxHeads + 32, v + 32);
            tmem_wait_ld();
            const float d =
                relu_dot32(v, wq + q * kIdxHeads) + relu_dot32(v + 32, wq + q * kIdxHeads + 32);
            if (j < J.n[q]) p.scores[r * p.ld + j] = d * kscale;
          }
        }
        tc_fence_before();
        mbar_arrive(&t_empty[acc]);
      }
      if (stop) break;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::kTmemCols);
  }
}

bool score_mx_supported(const ScoreArgs& a) {
  return a.dtype == SA_MXFP4 && a.HI == kIdxHeads && a.dI == kIdxDim && a.N_cap % 8 == 0 &&
         a.q_scales != nullptr && a.ik_scales != nullptr &&
         ((reinterpret_cast<uintptr_t>(a.ik) | reinterpret_cast<uintptr_t>(a.ik_scales) |
           reinterpret_cast<uintptr_t>(a.q)) & 15u) == 0;
}

template <int QG>
static cudaError_t launch_mx_qg(const ScoreArgs& a, int num_sms, cudaStream_t st) {
  using Cfg = MxCfg<QG>;
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
  const int grid = plan_score_jobs(p, QG, num_sms, Cfg::kS);
  if (grid == 0) return cudaSuccess;
  if (grid < 0) return cudaErrorInvalidValue;
  MxPtrs x{static_cast<const uint8_t*>(a.q), static_cast<const uint8_t*>(a.q_scales),
           static_cast<const uint8_t*>(a.ik), static_cast<const uint8_t*>(a.ik_scales)};
  cudaError_t e = cudaFuncSetAttribute(score_mx_kernel<QG>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)Cfg::kSmem);
  if (e != cudaSuccess) return e;
  score_mx_kernel<QG><<<grid, kMxThreads, Cfg::kSmem, st>>>(p, x);
  return cudaGetLastError();
}

cudaError_t launch_score_mx(const ScoreArgs& a, int num_sms, cudaStream_t st) {
  if (a.T >= 4) return launch_mx_qg<4>(a, num_sms, st);
  return launch_mx_qg<1>(a, num_sms, st);
}

}  // namespace sa
