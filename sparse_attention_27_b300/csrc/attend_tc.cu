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
// One CTA per (query row, split of its key list), 128 threads.  Keys come in
// tiles of 64: the compressed part (rows idx[r, i] for CSA, rows 0.. for HCA)
// then the window rows (ring slot u mod R).  Every thread gathers 16-byte
// chunks of K and V rows with cp.async straight into the 128-byte-swizzled
// layout the tensor core reads (masked keys are zero-filled), four tiles in
// flight.  Per tile:
//   S[128 x 64]  = Q[128 x 128] . K_tile^T     (tcgen05, A = Q K-major, B = K K-major)
//   P            = exp2(S * scale*log2e - m)   (one thread per head row, fp32)
//   O[128 x 128] += P . V_tile                 (tcgen05, A = P K-major, B = V MN-major)
// The 64 query heads of the one query fill rows 32w..32w+15 of the M = 128
// MMA (16 heads per TMEM lane quadrant), so all four warps share the softmax.
// The running max is raised only when it grows by more than 8 (log2 units);
// then O is rescaled in TMEM.  The result is normalised (or written as a
// normalised split partial with its LSE for the merge kernel).
#include "kernels.cuh"

namespace sa {

namespace {

constexpr int kThreads = 128;
constexpr int kKeys = 64;                      // keys per tile
constexpr int kStages = 4;
constexpr int kD = 128;                        // head dim
constexpr int kQBytes = 128 * kD * 2;          // 32 KB: Q as two 64-column swizzled blocks
constexpr int kKVBlock = kKeys * 128;          // 8 KB: one 64-dim half of a K or V tile
constexpr int kStageBytes = 4 * kKVBlock;      // K (2 halves) + V (2 halves) = 32 KB
constexpr int kPBytes = 128 * kKeys * 2;       // 16 KB
constexpr int kTmemCols = 256;                 // S: 64 cols at 0; O: 128 cols at 128
constexpr float kRescaleThreshold = 8.f;       // log2 units

struct Smem {
  // 1024-aligned region follows: Q | stages | P
  uint64_t bar_s, bar_o;
  uint32_t tmem;
  int valid[kStages][kKeys];
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Byte offset of 16-byte chunk `c` (0..7) of 128-byte row `r` inside a
// 128B-swizzled block whose base is 1024-aligned.
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}

struct RowInfo {
  int64_t nvis, n_comp, n_win, n_keys;
  int p, b;
};

__device__ __forceinline__ RowInfo row_info(const AttnArgs& a, int64_t row) {
  RowInfo ri;
  ri.b = (int)(row / a.T);
  ri.p = __ldg(a.q_pos + row);
  ri.nvis = ri.p < 0 ? 0 : ((int64_t)ri.p + 1) / a.m;
  if (ri.nvis > a.N_cap) ri.nvis = a.N_cap;
  ri.n_comp = a.gather ? min64(a.k, ri.nvis) : ri.nvis;
  ri.n_win = ri.p < 0 ? 0 : min64(a.W, (int64_t)ri.p + 1);
  ri.n_keys = ri.n_comp + ri.n_win;
  return ri;
}

// Gather key tile `tile` (64 keys) of this row into stage `st`.  Thread t
// copies key (t >> 1), 64-dim half (t & 1): 8 chunks of K and 8 of V.
__device__ __forceinline__ void gather_tile(const AttnArgs& a, const RowInfo& ri, int64_t row,
                                            int64_t tile, unsigned char* stage, int* valid,
                                            int32_t* err) {
  const int t = threadIdx.x;
  const int key = t >> 1, half = t & 1;
  const int64_t s = tile * kKeys + key;
  const __nv_bfloat16* kp = static_cast<const __nv_bfloat16*>(a.kr);
  const __nv_bfloat16* vp = static_cast<const __nv_bfloat16*>(a.vr);
  int64_t src = -1;
  if (s < ri.n_keys) {
    if (s < ri.n_comp) {
      int64_t j = a.gather ? (int64_t)__ldg(a.idx + row * a.k + s) : s;
      if (j < -1 || j >= ri.nvis) {
        set_err(err, SA_ERR_BOUNDS);
        j = -1;
      }
      if (j >= 0) {
        src = (int64_t)ri.b * a.N_cap + j;
        kp = static_cast<const __nv_bfloat16*>(a.kc);
        vp = static_cast<const __nv_bfloat16*>(a.vc);
      }
    } else {
      const int64_t u = (int64_t)ri.p - ri.n_win + 1 + (s - ri.n_comp);
      src = (int64_t)ri.b * a.R + u % a.R;
    }
  }
  const uint32_t bytes = src >= 0 ? 16u : 0u;
  const int64_t off = (src >= 0 ? src : 0) * kD + half * 64;
  const uint32_t kdst = smem_u32(stage) + half * kKVBlock;
  const uint32_t vdst = smem_u32(stage) + 2 * kKVBlock + half * kKVBlock;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    cp_async16(kdst + swz(key, c), kp + off + c * 8, bytes);
    cp_async16(vdst + swz(key, c), vp + off + c * 8, bytes);
  }
  if (half == 0) valid[key] = src >= 0;
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 1) attend_tc_kernel(AttnArgs a) {
  extern __shared__ unsigned char smem_raw[];
  Smem& S = *reinterpret_cast<Smem*>(smem_raw);
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + sizeof(Smem) + 1023) & ~uintptr_t(1023));
  unsigned char* sQ = base;
  unsigned char* sKV = sQ + kQBytes;
  unsigned char* sP = sKV + kStages * kStageBytes;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t row = blockIdx.x / a.nsplit;
  const int split = blockIdx.x % a.nsplit;
  const RowInfo ri = row_info(a, row);
  const int64_t nt_row = (ri.n_keys + kKeys - 1) / kKeys;
  const int64_t t_begin = (int64_t)split * a.split_tiles;
  const int64_t t_end = min64(nt_row, t_begin + a.split_tiles);
  const int nt = (int)max64(0, t_end - t_begin);

  if (tid == 0) {
    mbar_init(&S.bar_s, 1);
    mbar_init(&S.bar_o, 1);
    mbar_fence_init();
  }
  if (warp == 0) tmem_alloc(&S.tmem, kTmemCols);

  // start the first gathers before staging Q
  for (int i = 0; i < kStages - 1; ++i) {
    if (i < nt) gather_tile(a, ri, row, t_begin + i, sKV + i * kStageBytes, S.valid[i], a.err);
    cp_async_commit();
  }
  // Q rows: head h -> row 32*(h/16) + h%16; all other rows zero.  P likewise.
  {
    uint4* q4 = reinterpret_cast<uint4*>(sQ);
    for (int i = tid; i < kQBytes / 16; i += kThreads) q4[i] = make_uint4(0, 0, 0, 0);
    uint4* p4 = reinterpret_cast<uint4*>(sP);
    for (int i = tid; i < kPBytes / 16; i += kThreads) p4[i] = make_uint4(0, 0, 0, 0);
  }
  __syncthreads();
  {
    const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q) + row * a.H * kD;
    for (int i = tid; i < a.H * 16; i += kThreads) {     // 16 chunks of 8 per head row
      const int h = i >> 4, c = i & 15;
      const int r = (h >> 4) * 32 + (h & 15);
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(q + h * kD + c * 8));
      *reinterpret_cast<uint4*>(sQ + (c >> 3) * (128 * 128) + swz(r, c & 7)) = v;
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem;
  const uint32_t tS = tmem, tO = tmem + 128;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
  const bool is_head = lane < 16 && (warp * 16 + lane) < a.H;
  const int my_row = warp * 32 + lane;

  constexpr uint32_t idS = idesc_bf16(128, kKeys, 0, 0);
  constexpr uint32_t idO = idesc_bf16(128, kD, 0, 1);
  const float c2 = a.sm_scale * 1.4426950408889634f;   // natural logits -> log2 units
  float m_run = -INFINITY, l_run = 0.f;
  bool ok = true;

  for (int j = 0; j < nt && ok; ++j) {
    const int st = j % kStages;
    unsigned char* stage = sKV + st * kStageBytes;
    // tile j landed (groups complete in order; kStages-1 younger groups may pend)
    cp_async_wait<kStages - 2>();
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      const uint32_t qa = smem_u32(sQ), ka = smem_u32(stage);
#pragma unroll
      for (int kk = 0; kk < kD / 16; ++kk)
        tc_mma_f16(tS, sdesc_kmajor_sw128(qa + (kk >> 2) * (128 * 128) + (kk & 3) * 32),
                   sdesc_kmajor_sw128(ka + (kk >> 2) * kKVBlock + (kk & 3) * 32), idS,
                   kk > 0 ? 1u : 0u);
      tc_commit(&S.bar_s);
    }
    ok = mbar_wait(&S.bar_s, j & 1, a.err);
    tc_fence_after();
    // PV of tile j-1 must be done before P and O are touched, and before its
    // stage is refilled.
    if (j > 0) ok = ok && mbar_wait(&S.bar_o, (j - 1) & 1, a.err);
    tc_fence_after();
    ok = __syncthreads_and(ok);          // CTA-uniform, so no thread is left at a barrier
    if (!ok) break;
    // refill the stage tile j-1 used with tile j+kStages-1
    {
      const int jn = j + kStages - 1;
      if (jn < nt) {
        const int sn = jn % kStages;
        gather_tile(a, ri, row, t_begin + jn, sKV + sn * kStageBytes, S.valid[sn], a.err);
      }
      cp_async_commit();
    }
    // ---- softmax of this tile's rows
    float v[64];
    tmem_ld32(tS + lane_base, v);
    tmem_ld32(tS + lane_base + 32, v + 32);
    float mt = -INFINITY;
#pragma unroll
    for (int i = 0; i < 64; ++i) {
      v[i] = S.valid[st][i] ? v[i] * c2 : -INFINITY;
      mt = fmaxf(mt, v[i]);
    }
    float alpha = 1.f;
    bool need = false;
    if (is_head && mt > m_run) {
      if (m_run == -INFINITY) {
        m_run = mt;                                 // O holds zeros so far
      } else if (mt > m_run + kRescaleThreshold) {
        alpha = exp2f(m_run - mt);
        m_run = mt;
        need = true;
      }
    }
    if (__any_sync(0xffffffffu, need) && j > 0) {
#pragma unroll 1
      for (int c = 0; c < kD; c += 32) {
        float o[32];
        tmem_ld32(tO + lane_base + c, o);
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] *= alpha;
        tmem_st32(tO + lane_base + c, o);
      }
      tmem_st_wait();
    }
    l_run *= alpha;
    if (is_head) {
      float psum = 0.f;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint32_t w4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float p0 = v[c * 8 + 2 * e] == -INFINITY ? 0.f : exp2f(v[c * 8 + 2 * e] - m_run);
          const float p1 =
              v[c * 8 + 2 * e + 1] == -INFINITY ? 0.f : exp2f(v[c * 8 + 2 * e + 1] - m_run);
          __nv_bfloat162 h2 = __floats2bfloat162_rn(p0, p1);
          psum += __low2float(h2) + __high2float(h2);
          w4[e] = *reinterpret_cast<uint32_t*>(&h2);
        }
        *reinterpret_cast<uint4*>(sP + swz(my_row, c)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
      }
      l_run += psum;
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      const uint32_t pa = smem_u32(sP), va = smem_u32(stage) + 2 * kKVBlock;
#pragma unroll
      for (int kk = 0; kk < kKeys / 16; ++kk)
        tc_mma_f16(tO, sdesc_kmajor_sw128(pa + kk * 32),
                   sdesc_mnmajor_sw128(va + kk * 2048, kKVBlock, 1024), idO,
                   (j > 0 || kk > 0) ? 1u : 0u);
      tc_commit(&S.bar_o);
    }
  }
  if (ok && nt > 0) ok = mbar_wait(&S.bar_o, (nt - 1) & 1, a.err);
  ok = __syncthreads_and(ok);
  cp_async_wait<0>();
  tc_fence_after();

  // ---- output: normalised O and LSE (or a split partial)
  float* out_o = a.nsplit > 1 ? a.part_o + (row * a.nsplit + split) * a.H * kD : a.o + row * a.H * kD;
  float* out_l = a.nsplit > 1 ? a.part_lse + (row * a.nsplit + split) * a.H : a.lse + row * a.H;
  const int h = warp * 16 + lane;
  const bool have = ok && nt > 0 && l_run > 0.f;
  const float inv = have ? 1.f / l_run : 0.f;
#pragma unroll 1
  for (int c = 0; c < kD; c += 32) {
    float o[32];
    if (nt > 0) tmem_ld32(tO + lane_base + c, o);
    if (is_head) {
      float4* dst = reinterpret_cast<float4*>(out_o + h * kD + c);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        dst[i] = have ? make_float4(o[4 * i] * inv, o[4 * i + 1] * inv, o[4 * i + 2] * inv,
                                    o[4 * i + 3] * inv)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  if (is_head) out_l[h] = have ? (m_run + log2f(l_run)) * 0.6931471805599453f : -INFINITY;
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

bool attend_tc_supported(const AttnArgs& a) {
  return a.dtype == SA_BF16 && a.d == kD && a.H >= 1 && a.H <= 64;
}

size_t attend_tc_smem() {
  return sizeof(Smem) + 1024 + kQBytes + kStages * kStageBytes + kPBytes;
}

cudaError_t launch_attend_tc(const AttnArgs& a, cudaStream_t st) {
  const int64_t rows = (int64_t)a.B * a.T;
  if (rows == 0) return cudaSuccess;
  const size_t smem = attend_tc_smem();
  cudaError_t e =
      cudaFuncSetAttribute(attend_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  attend_tc_kernel<<<(unsigned)(rows * a.nsplit), kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace sa
