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
// Warp roles (448 threads): warp 0 = bulk-copy producer (raw codes + scales of
// 128 entries per tile, 4352 bytes, into a ring of raw stages), warp 1 = MMA
// issuer and TMEM owner, warps 2..9 = two converter warpgroups taking
// alternate tiles (one entry row per thread: e2m1 -> e4m3 into a
// 128B-swizzled K-major tile, the row's factor 2^(e_row) into a ring the
// epilogue reads, so a raw stage is free as soon as it is converted; the
// first group also converts each query group's B tile), warps 10..13 = the
// epilogue (weighted ReLU head sum as in the bf16 kernel; each warp keeps its
// query weights, with the row exponents folded in, in shared memory).
// Conversion is the longest per-tile chain, so it gets two warpgroups.  Every
// ring (16 raw stages, 4 A stages, 16 factor slots) has an even length: the
// previous user of a tile's slot is the tile of the same parity, handled by
// the same converter group, so each parity wait is at most one phase away.
// Every wait is bounded; on a timeout the CTA records SA_ERR_DEVICE_TIMEOUT,
// stops and still frees its TMEM.
#include <cuda_fp8.h>

#include "kernels.cuh"
#include "score_jobs.cuh"

namespace sa {

namespace {

constexpr int kMxThreads = 448;
constexpr int kMxConvWarps = 8;    // two converter warpgroups
constexpr int kMxEpiWarps = 4;     // one epilogue warpgroup
constexpr int kAStages = 4;
constexpr int kCodeRowBytes = kIdxDim / 2;                       // 32
constexpr int kScaleRowBytes = kIdxDim / 32;                     // 2
constexpr int kRawCodeBytes = kTileEntries * kCodeRowBytes;      // 4096
constexpr int kRawBytes = kTileEntries * (kCodeRowBytes + kScaleRowBytes);  // 4352
constexpr int kARowBytes = 128;                                  // swizzle row (64 used)
constexpr int kABytes = kTileEntries * kARowBytes;               // 16 KB

// Key-row factors 2^(e_row) pass from the converters to the epilogue through a
// ring of kKsSlots tiles.  A converter is at most kAStages + kAccBufs (<= 8)
// tiles ahead of the epilogue, so a slot is rewritten only after the epilogue
// has read it.
constexpr int kKsSlots = 16;

template <int QG>
struct MxCfg {
  static constexpr int kRawStages = QG == 1 ? 16 : 12;
  static constexpr int kAccCols = QG * kIdxHeads;
  static constexpr int kAccBufs = QG == 1 ? 4 : 2;
  static constexpr int kTmemCols = kAccBufs * kAccCols;          // 256 or 512
  static constexpr int kBBytes = QG * kIdxHeads * kARowBytes;    // 8 KB per query
  static constexpr size_t kWqBytes = kMxEpiWarps * QG * kIdxHeads * sizeof(float);
  static constexpr size_t kKsBytes = kKsSlots * kTileEntries * sizeof(float);
  static constexpr size_t kSmem = 1024 + kAStages * kABytes + 2 * kBBytes +
                                  kRawStages * kRawBytes + 1024 /* LUT + barriers */ +
                                  kMaxJobsPerCta * sizeof(JobRec<QG>) + kWqBytes + kKsBytes;
};

struct MxPtrs {
  const uint8_t* q_codes;    // [B*T, 64, 32]
  const uint8_t* q_scales;   // [B*T, 64, 2]
  const uint8_t* k_codes;    // [B, N_cap, 32]
  const uint8_t* k_scales;   // [B, N_cap, 2]
};

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
// lut_hi: codes 4-7) for the block's shift and the code's sign bit.
__device__ __forceinline__ uint2 e2m1x8_to_e4m3(uint32_t w, uint32_t lut_lo, uint32_t lut_hi) {
  const uint32_t mag_lo = __byte_perm(lut_lo, lut_hi, w & 0x7777u);
  const uint32_t mag_hi = __byte_perm(lut_lo, lut_hi, (w >> 16) & 0x7777u);
  const uint32_t sg = w & 0x88888888u;
  const uint32_t s_lo = ((sg & 0x8u) << 4) | ((sg & 0x80u) << 8) | ((sg & 0x800u) << 12) |
                        ((sg & 0x8000u) << 16);
  const uint32_t s_hi = ((sg >> 12) & 0x80u) | ((sg >> 8) & 0x8000u) | ((sg >> 4) & 0x800000u) |
                        (sg & 0x80000000u);
  return make_uint2(mag_lo | s_lo, mag_hi | s_hi);
}

// Convert one 64-element MXFP4 row (32 code bytes as two uint4, 2 scale bytes)
// into 64 e4m3 bytes at row `r` of a 128B-swizzled tile; returns e_row.
__device__ __forceinline__ int convert_row(uint4 c0, uint4 c1, uint32_t sc0, uint32_t sc1,
                                           const uint32_t* lut, unsigned char* tile, int r) {
  const int e0 = (int)sc0 - 127, e1 = (int)sc1 - 127;
  const int er = max(e0, e1);
  const int s0 = min(er - e0, 15), s1 = min(er - e1, 15);
  const uint32_t l0a = lut[2 * s0], l0b = lut[2 * s0 + 1];
  const uint32_t l1a = lut[2 * s1], l1b = lut[2 * s1 + 1];
  // block 0 = elements 0..31 = code bytes 0..15 = c0; block 1 = c1
  const uint2 a0 = e2m1x8_to_e4m3(c0.x, l0a, l0b), a1 = e2m1x8_to_e4m3(c0.y, l0a, l0b);
  const uint2 a2 = e2m1x8_to_e4m3(c0.z, l0a, l0b), a3 = e2m1x8_to_e4m3(c0.w, l0a, l0b);
  const uint2 b0 = e2m1x8_to_e4m3(c1.x, l1a, l1b), b1 = e2m1x8_to_e4m3(c1.y, l1a, l1b);
  const uint2 b2 = e2m1x8_to_e4m3(c1.z, l1a, l1b), b3 = e2m1x8_to_e4m3(c1.w, l1a, l1b);
  unsigned char* row = tile + r * kARowBytes;
  const int x = r & 7;
  *reinterpret_cast<uint4*>(row + ((0 ^ x) << 4)) = make_uint4(a0.x, a0.y, a1.x, a1.y);
  *reinterpret_cast<uint4*>(row + ((1 ^ x) << 4)) = make_uint4(a2.x, a2.y, a3.x, a3.y);
  *reinterpret_cast<uint4*>(row + ((2 ^ x) << 4)) = make_uint4(b0.x, b0.y, b1.x, b1.y);
  *reinterpret_cast<uint4*>(row + ((3 ^ x) << 4)) = make_uint4(b2.x, b2.y, b3.x, b3.y);
  return er;
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
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* sA = smem;
  unsigned char* sB = sA + kAStages * kABytes;
  unsigned char* sRaw = sB + 2 * Cfg::kBBytes;
  constexpr int kRawStages = Cfg::kRawStages;
  uint32_t* lut = reinterpret_cast<uint32_t*>(sRaw + kRawStages * kRawBytes);   // [16][2]
  uint64_t* bars = reinterpret_cast<uint64_t*>(lut + 32);
  uint64_t* raw_full = bars;
  uint64_t* raw_empty = raw_full + kRawStages;
  uint64_t* a_full = raw_empty + kRawStages;
  uint64_t* a_empty = a_full + kAStages;
  uint64_t* b_full = a_empty + kAStages;
  uint64_t* b_empty = b_full + 2;
  uint64_t* t_full = b_empty + 2;
  uint64_t* t_empty = t_full + Cfg::kAccBufs;
  uint64_t* ks_full = t_empty + Cfg::kAccBufs;                     // [kKsSlots]
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(ks_full + kKsSlots);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
  JobRec<QG>* jobs = reinterpret_cast<JobRec<QG>*>(reinterpret_cast<unsigned char*>(lut) + 1024);
  float* s_wq = reinterpret_cast<float*>(jobs + kMaxJobsPerCta);   // [kMxEpiWarps][QG][64]
  float* s_ks = s_wq + kMxEpiWarps * QG * kIdxHeads;                // [kKsSlots][128]

  const int n_my = fill_job_table<QG>(p, jobs);
  const int warp = (int)warp_id(), lane = (int)lane_id();
  if (threadIdx.x < 128) {                  // magnitude tables for shifts 0..15
    const int s = threadIdx.x >> 3, c = threadIdx.x & 7;
    reinterpret_cast<uint8_t*>(lut)[s * 8 + c] = e4m3_of(c, s);
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kRawStages; ++s) { mbar_init(&raw_full[s], 1); mbar_init(&raw_empty[s], 128); }
    for (int s = 0; s < kKsSlots; ++s) mbar_init(&ks_full[s], 128);
    for (int s = 0; s < kAStages; ++s) { mbar_init(&a_full[s], 128); mbar_init(&a_empty[s], 1); }
    for (int s = 0; s < 2; ++s) { mbar_init(&b_full[s], 128); mbar_init(&b_empty[s], 1); }
    for (int s = 0; s < Cfg::kAccBufs; ++s) { mbar_init(&t_full[s], 1); mbar_init(&t_empty[s], 128); }
    *s_abort = 0;
    mbar_fence_init();
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
      for (int ji = 0; ji < n_my && !*s_abort; ++ji) {
        const JobRec<QG>& J = jobs[ji];
        for (int t = J.t_lo; t < J.t_hi; ++t) {
          if (!mbar_wait(&raw_empty[stage], ph ^ 1, p.err)) { *s_abort = 1; break; }
          const int64_t e0 = (int64_t)J.b * p.N_cap + (int64_t)t * kTileEntries;
          const uint32_t rows = (uint32_t)min64(kTileEntries, (int64_t)p.N_cap - (int64_t)t * kTileEntries);
          unsigned char* dst = sRaw + stage * kRawBytes;
          mbar_arrive_expect_tx(&raw_full[stage], rows * (kCodeRowBytes + kScaleRowBytes));
          bulk_g2s(dst, x.k_codes + e0 * kCodeRowBytes, rows * kCodeRowBytes, &raw_full[stage]);
          bulk_g2s(dst + kRawCodeBytes, x.k_scales + e0 * kScaleRowBytes, rows * kScaleRowBytes,
                   &raw_full[stage]);
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
        for (int t = J.t_lo; t < J.t_hi; ++t) {
          if (!mbar_wait(&a_full[stage], ph, p.err)) { *s_abort = 1; break; }
          if (!mbar_wait(&t_empty[acc], acc_ph ^ 1, p.err)) { *s_abort = 1; break; }
          tc_fence_after();
          const uint32_t a_base = smem_u32(sA + stage * kABytes);
#pragma unroll
          for (int kk = 0; kk < 2; ++kk)          // K = 64 e4m3 = two MMAs of K = 32
            tc_mma_f8f6f4(tmem + acc * Cfg::kAccCols, sdesc_kmajor_sw128(a_base + kk * 32),
                          sdesc_kmajor_sw128(b_base + kk * 32), idesc, kk > 0 ? 1u : 0u);
          tc_commit(&a_empty[stage]);
          tc_commit(&t_full[acc]);
          if (++stage == kAStages) { stage = 0; ph ^= 1; }
          if (++acc == Cfg::kAccBufs) { acc = 0; acc_ph ^= 1; }
        }
      }
    }
    __syncwarp();
  } else if (warp < 2 + kMxConvWarps) {
    // ---------------------------------------------------------- converters
    const int cgrp = (warp - 2) >> 2;           // converts the tiles with ordinal parity cgrp
    const int c = ((int)threadIdx.x - 64) & 127;  // entry row of the tile, 0..127
    int nsw = 0;
    int64_t ko = 0;                             // tile ordinal: raw stage, A stage, factor slot
    int64_t prev_g = -1;
    for (int ji = 0; ji < n_my && !*s_abort; ++ji) {
      const JobRec<QG>& J = jobs[ji];
      if (J.t_lo >= J.t_hi) continue;
      bool stop = false;
      if (J.g != prev_g && cgrp == 0) {
        // the query group's B tile: QG*64 rows (query q, head h), zero past nq
        const int slot = nsw & 1;
        if (!mbar_wait(&b_empty[slot], ((nsw >> 1) & 1) ^ 1, p.err)) { *s_abort = 1; break; }
        unsigned char* tile = sB + slot * Cfg::kBBytes;
        for (int rr = c; rr < QG * kIdxHeads; rr += 128) {
          const int q = rr / kIdxHeads;
          if (q < J.nq) {
            const int64_t qrow = ((int64_t)J.b * p.T + J.t0 + q) * kIdxHeads + (rr % kIdxHeads);
            const uint4* src = reinterpret_cast<const uint4*>(x.q_codes + qrow * kCodeRowBytes);
            convert_row(__ldg(src), __ldg(src + 1), x.q_scales[qrow * 2], x.q_scales[qrow * 2 + 1],
                        lut, tile, rr);
          } else {
            unsigned char* row = tile + rr * kARowBytes;
#pragma unroll
            for (int ch = 0; ch < 4; ++ch)
              *reinterpret_cast<uint4*>(row + ((ch ^ (rr & 7)) << 4)) = make_uint4(0, 0, 0, 0);
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(&b_full[slot]);
        ++nsw;
      }
      prev_g = J.g;
      for (int t = J.t_lo; t < J.t_hi; ++t, ++ko) {
        if ((int)(ko & 1) != cgrp) continue;
        const int rstage = (int)(ko % kRawStages), astage = (int)(ko % kAStages);
        const uint32_t rph = (uint32_t)((ko / kRawStages) & 1), aph = (uint32_t)((ko / kAStages) & 1);
        if (!mbar_wait(&raw_full[rstage], rph, p.err)) { *s_abort = 1; stop = true; break; }
        const unsigned char* raw = sRaw + rstage * kRawBytes;
        const uint4 c0 = *reinterpret_cast<const uint4*>(raw + c * kCodeRowBytes);
        const uint4 c1 = *reinterpret_cast<const uint4*>(raw + c * kCodeRowBytes + 16);
        const uint32_t sc0 = raw[kRawCodeBytes + 2 * c], sc1 = raw[kRawCodeBytes + 2 * c + 1];
        mbar_arrive(&raw_empty[rstage]);
        if (!mbar_wait(&a_empty[astage], aph ^ 1, p.err)) { *s_abort = 1; stop = true; break; }
        const int er = convert_row(c0, c1, sc0, sc1, lut, sA + astage * kABytes, c);
        fence_proxy_async_smem();
        mbar_arrive(&a_full[astage]);
        const int ks = (int)(ko % kKsSlots);
        s_ks[ks * kTileEntries + c] = pow2i(er);
        mbar_arrive(&ks_full[ks]);
      }
      if (stop) break;
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // Tile ordinal o uses accumulator o % kAccBufs.
    const int quad = warp & 3;
    const int row_in_tile = quad * 32 + lane;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    float* wq = s_wq + (warp - 2 - kMxConvWarps) * QG * kIdxHeads;   // this warp's weights
    int64_t o = 0;                // tile ordinal (factor slot o % kKsSlots)
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
      for (int t = J.t_lo; t < J.t_hi; ++t, ++o) {
        const int acc = (int)(o % Cfg::kAccBufs);
        if (!mbar_wait(&t_full[acc], (uint32_t)((o / Cfg::kAccBufs) & 1), p.err)) {
          *s_abort = 1;
          stop = true;
          break;
        }
        // this entry row's factor 2^(e_row), from the converters' ring
        const int ks = (int)(o % kKsSlots);
        if (!mbar_wait(&ks_full[ks], (uint32_t)((o / kKsSlots) & 1), p.err)) {
          *s_abort = 1;
          stop = true;
          break;
        }
        const float kscale = s_ks[ks * kTileEntries + row_in_tile];
        tc_fence_after();
        const int64_t j = (int64_t)t * kTileEntries + row_in_tile;
#pragma unroll 1
        for (int q = 0; q < J.nq; ++q) {
          const int64_t r = (int64_t)J.b * p.T + J.t0 + q;
          uint32_t v[64];
          tmem_ld32_async(tmem + lane_base + acc * Cfg::kAccCols + q * kIdxHeads, v);
          tmem_ld32_async(tmem + lane_base + acc * Cfg::kAccCols + q * kIdxHeads + 32, v + 32);
          tmem_wait_ld();
          const float4* w4 = reinterpret_cast<const float4*>(wq + q * kIdxHeads);
          float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float4 wv = w4[i];
            s0 = fmaf(wv.x, fmaxf(__uint_as_float(v[4 * i + 0]), 0.f), s0);
            s1 = fmaf(wv.y, fmaxf(__uint_as_float(v[4 * i + 1]), 0.f), s1);
            s2 = fmaf(wv.z, fmaxf(__uint_as_float(v[4 * i + 2]), 0.f), s2);
            s3 = fmaf(wv.w, fmaxf(__uint_as_float(v[4 * i + 3]), 0.f), s3);
          }
          if (j < J.n[q]) p.scores[r * p.ld + j] = ((s0 + s1) + (s2 + s3)) * kscale;
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
  const int grid = plan_score_jobs(p, QG, num_sms);
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
