// extern "C" entry points of libsa27 (declared and documented in include/sa.h):
// host-side argument validation, kernel choice by dtype and shape, workspace
// carving and launches.  Nothing here allocates, frees or synchronises.
#include <algorithm>
#include <mutex>

#include "kernels.cuh"

using namespace sa;

namespace {

int device_sms() {
  static std::mutex mu;
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  std::lock_guard<std::mutex> lk(mu);
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
int elem_bytes(int dt) { return dt == SA_F32 ? 4 : 2; }
bool plain_dtype(int dt) { return dt == SA_F32 || dt == SA_BF16; }
int status_of(cudaError_t e) {
  if (e == cudaSuccess) return SA_OK;
  cudaGetLastError();  // clear a sticky launch error for the caller's next call
  return e == cudaErrorNotSupported ? SA_ERR_UNSUPPORTED : SA_ERR_CUDA;
}
size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// Key-tile split of each query row's key list for the attention kernels.
struct Split {
  int nsplit, split_tiles;
};
// Splits per row: enough (row, split) items for `per_sm` items per SM, and
// no split longer than `cap` key tiles.
Split choose_split(int64_t rows, int max_tiles, int per_sm, int cap) {
  Split s{1, max_tiles > 0 ? max_tiles : 1};
  if (rows <= 0 || max_tiles <= 1) return s;
  const int64_t want = std::max<int64_t>(1, ((int64_t)per_sm * device_sms() + rows - 1) / rows);
  int ns = (int)std::min<int64_t>(want, max_tiles);
  ns = std::max(ns, (max_tiles + cap - 1) / cap);
  if (ns < 1) ns = 1;
  s.split_tiles = (max_tiles + ns - 1) / ns;
  s.nsplit = (max_tiles + s.split_tiles - 1) / s.split_tiles;
  return s;
}
size_t split_bytes(int64_t rows, int H, int d, const Split& s) {
  if (s.nsplit <= 1) return 0;
  return round256(sizeof(float) * (size_t)rows * s.nsplit * H * d) +
         round256(sizeof(float) * (size_t)rows * s.nsplit * H);
}
constexpr size_t kCounterBytes = 256;   // the attention's item counter, after the partials
int attn_tiles(int64_t n_comp_max, int W) {
  return (int)((n_comp_max + kAttnTile - 1) / kAttnTile + (W + kAttnTile - 1) / kAttnTile);
}

// Items per SM for an attention call: the tensor-core kernel is a persistent
// pipeline that takes about two items per SM; the CUDA-core kernel runs one
// CTA per item, at most one wave.
int attention_items_per_sm(int dtype, int H, int d) {
  AttnArgs probe{};
  probe.dtype = dtype; probe.H = H; probe.d = d;
  return attend_tc_supported(probe) ? attend_tc_items_per_sm() : 1;
}
int attention_split_cap(int dtype, int H, int d) {
  AttnArgs probe{};
  probe.dtype = dtype; probe.H = H; probe.d = d;
  return attend_tc_supported(probe) ? kAttnTcMaxSplitTiles : (1 << 30);
}
Split attention_split(int dtype, int64_t rows, int H, int d, int max_tiles) {
  return choose_split(rows, max_tiles, attention_items_per_sm(dtype, H, d),
                      attention_split_cap(dtype, H, d));
}

int run_attention(AttnArgs& a, void* ws, size_t ws_bytes, int max_tiles, cudaStream_t st) {
  const int64_t rows = (int64_t)a.B * a.T;
  const Split s = attention_split(a.dtype, rows, a.H, a.d, max_tiles);
  a.nsplit = s.nsplit;
  a.split_tiles = s.split_tiles;
  a.part_o = nullptr;
  a.part_lse = nullptr;
  a.item_counter = nullptr;
  const size_t need = split_bytes(rows, a.H, a.d, s);
  if (s.nsplit > 1) {
    if (ws == nullptr || ws_bytes < need || !al16(ws)) return SA_ERR_INVALID_ARG;
    a.part_o = static_cast<float*>(ws);
    a.part_lse = reinterpret_cast<float*>(static_cast<char*>(ws) +
                                          round256(sizeof(float) * (size_t)rows * s.nsplit * a.H * a.d));
  }
  const bool tc = attend_tc_supported(a);
  if (tc && ws != nullptr && ws_bytes >= need + kCounterBytes && al16(ws)) {
    // a workspace with room for the item counter: the tensor-core kernel takes
    // its items dynamically
    a.item_counter = reinterpret_cast<unsigned*>(static_cast<char*>(ws) + need);
    const cudaError_t z = cudaMemsetAsync(a.item_counter, 0, sizeof(unsigned), st);
    if (z != cudaSuccess) return status_of(z);
  }
  cudaError_t e = tc ? launch_attend_tc(a, device_sms(), st) : launch_attend_simt(a, st);
  if (e != cudaSuccess) return status_of(e);
  return status_of(launch_merge_splits(a, st));
}

}  // namespace

extern "C" {

const char* sa_status_string(int s) {
  switch (s) {
    case SA_OK: return "ok";
    case SA_ERR_INVALID_ARG: return "invalid argument";
    case SA_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case SA_ERR_CUDA: return "CUDA error";
    case SA_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case SA_ERR_BOUNDS: return "index or position out of range";
    case SA_ERR_NAN: return "NaN score";
    default: return "unknown status";
  }
}

int csa_compress(int dtype, int ik_dtype, int B, int d, int dI, int m, const void* k_raw,
                 const void* v_raw, const void* ik_raw, const float* z, int R,
                 const int32_t* blk_lo, const int32_t* blk_hi, int max_blocks, void* k_c,
                 void* v_c, void* ik_c, void* ik_c_scales, int N_cap, int32_t* err,
                 void* stream) {
  if (!plain_dtype(dtype) || B < 0 || d <= 0 || m < 1 || R < m || max_blocks < 0 || N_cap < 0)
    return SA_ERR_INVALID_ARG;
  const int vec = 16 / elem_bytes(dtype);
  if (d % vec || 2 * d / vec + (ik_raw && ik_dtype != SA_MXFP4 ? dI / vec : 0) > 256)
    return SA_ERR_UNSUPPORTED;
  if (!k_raw || !v_raw || !z || !blk_lo || !blk_hi || !k_c || !v_c) return SA_ERR_INVALID_ARG;
  if (!al16(k_raw) || !al16(v_raw) || !al16(k_c) || !al16(v_c)) return SA_ERR_INVALID_ARG;
  if (ik_raw) {
    if (!ik_c || !al16(ik_raw) || !al16(ik_c) || dI <= 0) return SA_ERR_INVALID_ARG;
    if (ik_dtype == SA_MXFP4) {
      if (dtype != SA_BF16 || dI % 32 || !ik_c_scales) return SA_ERR_UNSUPPORTED;
    } else if (ik_dtype != dtype || dI % vec) {
      return SA_ERR_UNSUPPORTED;
    }
  }
  if (B == 0 || max_blocks == 0) return SA_OK;
  CompressArgs a{dtype, ik_dtype, B, d, dI, m, k_raw, v_raw, ik_raw, z, R, blk_lo, blk_hi,
                 max_blocks, k_c, v_c, ik_c, ik_c_scales, N_cap, err};
  return status_of(launch_compress(a, static_cast<cudaStream_t>(stream)));
}

size_t csa_index_topk_workspace_bytes(int B, int T, int N_cap, int k) {
  (void)k;
  if (B <= 0 || T <= 0 || N_cap <= 0) return 0;
  return round256(sizeof(float) * (size_t)B * T * N_cap);
}

int csa_index_topk(int q_dtype, int B, int T, int HI, int dI, int m, int k, const void* q_idx,
                   const void* q_scales, const float* w, const void* ik_c,
                   const void* ik_scales, int N_cap, const int32_t* q_pos, int32_t* idx,
                   float* scores_out, const float* scores_in, void* ws, size_t ws_bytes,
                   int32_t* err, void* stream) {
  if (B < 0 || T < 0 || m < 1 || k < 0 || N_cap < 0 || !q_pos || (k > 0 && !idx))
    return SA_ERR_INVALID_ARG;
  if (!topk_supported(N_cap)) return SA_ERR_UNSUPPORTED;
  const int64_t rows = (int64_t)B * T;
  if (rows == 0 || (k == 0 && (scores_in || !scores_out))) return SA_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const float* sc = scores_in;
  if (!scores_in) {
    if (q_dtype != SA_F32 && q_dtype != SA_BF16 && q_dtype != SA_MXFP4) return SA_ERR_INVALID_ARG;
    if (HI <= 0 || dI <= 0 || !q_idx || !w || !ik_c) return SA_ERR_INVALID_ARG;
    if (!al16(q_idx) || !al16(w) || !al16(ik_c)) return SA_ERR_INVALID_ARG;
    float* dst = scores_out;
    if (!dst) {
      if (!ws || ws_bytes < csa_index_topk_workspace_bytes(B, T, N_cap, k) || !al16(ws))
        return SA_ERR_INVALID_ARG;
      dst = static_cast<float*>(ws);
    }
    ScoreArgs sa_{q_dtype, B, T, HI, dI, m, q_idx, q_scales, w, ik_c, ik_scales, N_cap,
                  q_pos, dst, (int64_t)N_cap, err};
    cudaError_t e;
    if (q_dtype == SA_MXFP4) {
      if (!score_mx_supported(sa_)) return SA_ERR_UNSUPPORTED;
      e = launch_score_mx(sa_, device_sms(), st);
    } else if (score_tc_supported(sa_)) {
      e = launch_score_tc(sa_, device_sms(), st);
    } else {
      if ((size_t)HI * dI + HI > 12 * 1024) return SA_ERR_UNSUPPORTED;
      e = launch_score_simt(sa_, st);
    }
    if (e != cudaSuccess) return status_of(e);
    sc = dst;
  }
  if (k == 0) return SA_OK;   // scores only
  TopkArgs ta{sc, (int64_t)N_cap, q_pos, (int)rows, m, N_cap, k, idx, err};
  return status_of(launch_topk(ta, device_sms(), st));
}

size_t csa_attend_workspace_bytes(int dtype, int B, int T, int H, int d, int k, int W) {
  const int64_t rows = (int64_t)B * T;
  if (rows <= 0 || H <= 0 || d <= 0) return 0;
  return split_bytes(rows, H, d, attention_split(dtype, rows, H, d, attn_tiles(k, W))) +
         kCounterBytes;
}

int csa_attend(int dtype, int B, int T, int H, int d, int m, int k, int W, float sm_scale,
               const void* q, const int32_t* q_pos, const void* k_c, const void* v_c,
               int N_cap, const int32_t* idx, const void* k_raw, const void* v_raw, int R,
               void* o, int o_dtype, float* lse, void* ws, size_t ws_bytes, int32_t* err,
               void* stream) {
  if (!plain_dtype(dtype) || !plain_dtype(o_dtype) || B < 0 || T < 0 || H <= 0 || d <= 0 ||
      d > 256 || m < 1 || k < 0 || W < 0 || N_cap < 0 || R < W || R < 1)
    return SA_ERR_INVALID_ARG;
  if (!q || !q_pos || !o || !lse || !k_raw || !v_raw || (k > 0 && (!idx || !k_c || !v_c)))
    return SA_ERR_INVALID_ARG;
  if (!al16(q) || !al16(o) || !al16(k_raw) || !al16(v_raw) || (k_c && !al16(k_c)) ||
      (v_c && !al16(v_c)))
    return SA_ERR_INVALID_ARG;
  if ((size_t)H * d > 16384 || d % 4) return SA_ERR_UNSUPPORTED;
  if ((int64_t)B * T == 0) return SA_OK;
  AttnArgs a{};
  a.dtype = dtype; a.B = B; a.T = T; a.H = H; a.d = d; a.sm_scale = sm_scale;
  a.q = q; a.q_pos = q_pos; a.kc = k_c; a.vc = v_c; a.N_cap = N_cap; a.idx = idx;
  a.k = k; a.m = m; a.kr = k_raw; a.vr = v_raw; a.R = R; a.W = W; a.o = o;
  a.o_dtype = o_dtype; a.lse = lse;
  a.err = err;
  a.gather = 1;
  return run_attention(a, ws, ws_bytes, attn_tiles(k, W), static_cast<cudaStream_t>(stream));
}

size_t hca_compress_attend_workspace_bytes(int dtype, int B, int T, int H, int d, int N2_cap,
                                           int W) {
  const int64_t rows = (int64_t)B * T;
  if (rows <= 0 || H <= 0 || d <= 0) return 0;
  return split_bytes(rows, H, d, attention_split(dtype, rows, H, d, attn_tiles(N2_cap, W))) +
         kCounterBytes;
}

int hca_compress_attend(int dtype, int B, int T, int H, int d, int m2, int W, float sm_scale,
                        const void* q, const int32_t* q_pos, const void* k_raw,
                        const void* v_raw, const float* z_hca, int R, const int32_t* blk_lo,
                        const int32_t* blk_hi, int max_blocks, void* hk_c, void* hv_c,
                        int N2_cap, void* o, int o_dtype, float* lse, void* ws,
                        size_t ws_bytes, int32_t* err, void* stream) {
  if (!plain_dtype(dtype) || !plain_dtype(o_dtype) || B < 0 || T < 0 || H <= 0 || d <= 0 ||
      d > 256 || m2 < 1 || W < 0 || N2_cap < 0 || R < W || R < 1 || max_blocks < 0)
    return SA_ERR_INVALID_ARG;
  if (!q || !q_pos || !o || !lse || !k_raw || !v_raw || (N2_cap > 0 && (!hk_c || !hv_c)))
    return SA_ERR_INVALID_ARG;
  if (!al16(q) || !al16(o) || !al16(k_raw) || !al16(v_raw) || (hk_c && !al16(hk_c)) ||
      (hv_c && !al16(hv_c)))
    return SA_ERR_INVALID_ARG;
  if ((size_t)H * d > 16384 || d % 4) return SA_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (max_blocks > 0 && B > 0) {
    if (!z_hca || !blk_lo || !blk_hi || R < m2) return SA_ERR_INVALID_ARG;
    const int vec = 16 / elem_bytes(dtype);
    if (d % vec || 2 * d / vec > 256) return SA_ERR_UNSUPPORTED;
    CompressArgs c{dtype, dtype, B, d, 0, m2, k_raw, v_raw, nullptr, z_hca, R, blk_lo, blk_hi,
                   max_blocks, hk_c, hv_c, nullptr, nullptr, N2_cap, err};
    const int s = status_of(launch_compress(c, st));
    if (s != SA_OK) return s;
  }
  if ((int64_t)B * T == 0) return SA_OK;
  AttnArgs a{};
  a.dtype = dtype; a.B = B; a.T = T; a.H = H; a.d = d; a.sm_scale = sm_scale;
  a.q = q; a.q_pos = q_pos; a.kc = hk_c; a.vc = hv_c; a.N_cap = N2_cap; a.idx = nullptr;
  a.gather = 0;
  a.k = 0; a.m = m2; a.kr = k_raw; a.vr = v_raw; a.R = R; a.W = W; a.o = o;
  a.o_dtype = o_dtype; a.lse = lse;
  a.err = err;
  return run_attention(a, ws, ws_bytes, attn_tiles(N2_cap, W), st);
}

int csa_decode(int B, int H, int d, int HI, int dI, int m, int k, int W, float sm_scale,
               const void* q, const void* q_idx, const float* w, const int32_t* q_pos,
               const void* k_raw, const void* v_raw, const void* ik_raw, const float* z, int R,
               const int32_t* blk_lo, const int32_t* blk_hi, int max_blocks, void* k_c,
               void* v_c, void* ik_c, int N_cap, int32_t* idx, void* o, int o_dtype,
               float* lse, int32_t* err, void* stream) {
  if (B < 0 || H < 1 || m < 1 || k < 0 || W < 0 || R < 1 || R < W || R < m || N_cap < 0 ||
      max_blocks < 0 || !plain_dtype(o_dtype))
    return SA_ERR_INVALID_ARG;
  if (d != 128 || HI != 64 || dI != 64 || H > 64 || m > 128) return SA_ERR_UNSUPPORTED;
  if (!q || !q_idx || !w || !q_pos || !k_raw || !v_raw || !ik_raw || !z || !blk_lo || !blk_hi ||
      !k_c || !v_c || !ik_c || !o || !lse || (k > 0 && !idx))
    return SA_ERR_INVALID_ARG;
  if (!al16(q) || !al16(q_idx) || !al16(w) || !al16(k_raw) || !al16(v_raw) || !al16(ik_raw) ||
      !al16(k_c) || !al16(v_c) || !al16(ik_c) || !al16(o))
    return SA_ERR_INVALID_ARG;
  if (B == 0) return SA_OK;
  FusedDecodeArgs a{};
  a.B = B; a.H = H; a.m = m; a.k = k; a.W = W; a.sm_scale = sm_scale;
  a.q = q; a.q_idx = q_idx; a.w = w; a.q_pos = q_pos;
  a.k_raw = k_raw; a.v_raw = v_raw; a.ik_raw = ik_raw; a.z = z; a.R = R;
  a.blk_lo = blk_lo; a.blk_hi = blk_hi; a.max_blocks = max_blocks;
  a.k_c = k_c; a.v_c = v_c; a.ik_c = ik_c; a.N_cap = N_cap;
  a.idx = idx; a.o = o; a.o_dtype = o_dtype; a.lse = lse; a.err = err;
  if (!fused_decode_plan(a, device_sms())) return SA_ERR_UNSUPPORTED;
  return status_of(launch_fused_decode(a, static_cast<cudaStream_t>(stream)));
}

int sa_compress_channels(int dtype, int B, int d, int m, const void* x_raw, const float* z, int R,
                         const int32_t* blk_lo, const int32_t* blk_hi, int max_blocks, void* x_c,
                         int N_cap, int32_t* err, void* stream) {
  if (!plain_dtype(dtype) || B < 0 || d < 1 || m < 1 || R < m || max_blocks < 0 || N_cap < 0)
    return SA_ERR_INVALID_ARG;
  if (!x_raw || !z || !blk_lo || !blk_hi || !x_c) return SA_ERR_INVALID_ARG;
  CompressChArgs a{};
  a.dtype = dtype; a.B = B; a.d = d; a.m = m; a.R = R; a.max_blocks = max_blocks; a.N_cap = N_cap;
  a.x_raw = x_raw; a.z = z; a.blk_lo = blk_lo; a.blk_hi = blk_hi; a.x_c = x_c; a.err = err;
  return status_of(launch_compress_channels(a, static_cast<cudaStream_t>(stream)));
}

int sa_ring_write(int B, int R, const int32_t* pos, int n, void* const* rings,
                  const void* const* rows, const int* row_bytes, int32_t* err, void* stream) {
  if (B < 0 || R < 1 || n < 1 || n > kRingMaxArrays || !pos || !rings || !rows || !row_bytes)
    return SA_ERR_INVALID_ARG;
  RingWriteArgs a{};
  a.B = B; a.R = R; a.n = n; a.pos = pos; a.err = err;
  for (int i = 0; i < n; ++i) {
    if (!rings[i] || !rows[i] || row_bytes[i] <= 0 || row_bytes[i] % 4 ||
        reinterpret_cast<uintptr_t>(rings[i]) % 4 || reinterpret_cast<uintptr_t>(rows[i]) % 4)
      return SA_ERR_INVALID_ARG;
    a.rings[i] = rings[i];
    a.rows[i] = rows[i];
    a.row_bytes[i] = row_bytes[i];
  }
  return status_of(launch_ring_write(a, static_cast<cudaStream_t>(stream)));
}

namespace {
// Workspace of sa_decode_step: counters, histograms and row info (zeroed by
// each call) | score keys [B, N_cap] | CSA partials | HCA partials | top-k
// candidate lists, each part 256-byte aligned.  Returns false when the step
// kernel does not take the shape.
bool step_layout(StepArgs& a, size_t* offs /* [7] */, size_t* total) {
  if (!decode_step_plan(a, device_sms())) return false;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  size_t o = 0;
  offs[0] = o; o += up(decode_step_counter_bytes(a.B));
  offs[1] = o; o += up(4 * (size_t)a.B * ((a.N_cap + 3) / 4 * 4));
  offs[2] = o; o += up(4 * (size_t)a.B * a.na * 64 * 128);
  offs[3] = o; o += up(4 * (size_t)a.B * a.na * 64);
  offs[4] = o; o += up(4 * (size_t)a.B * a.nh * 64 * 128);
  offs[5] = o; o += up(4 * (size_t)a.B * a.nh * 64);
  offs[6] = o; o += up(4 * (size_t)a.B * 4 * 4096);
  *total = o;
  return true;
}
}  // namespace

size_t sa_decode_step_workspace_bytes(int B, int H, int N_cap, int k, int W, int N2_cap) {
  if (B < 1 || H < 1 || N_cap < 0 || k < 0 || W < 0 || N2_cap < 0) return 0;
  StepArgs a{};
  a.B = B; a.H = H; a.N_cap = N_cap; a.k = k; a.W = W; a.N2_cap = N2_cap; a.m = 1; a.m2 = 1;
  size_t offs[7], total = 0;
  return step_layout(a, offs, &total) ? total : 0;
}

int sa_decode_step(int B, int H, int d, int HI, int dI, int m, int k, int W, int m2,
                   float sm_scale, const void* q, const void* q_idx, const float* w,
                   const void* q_hca, const int32_t* q_pos, const void* k_raw, const void* v_raw,
                   const void* ik_raw, const float* z, const void* hk_raw, const void* hv_raw,
                   const float* hz, int R, const int32_t* blk_lo, const int32_t* blk_hi,
                   int max_blocks, const int32_t* hblk_lo, const int32_t* hblk_hi,
                   int max_blocks2, void* k_c, void* v_c, void* ik_c, int N_cap, void* hk_c,
                   void* hv_c, int N2_cap, int32_t* idx, int o_dtype, void* o, float* lse,
                   void* ho, float* hlse, void* ws, size_t ws_bytes, int32_t* err,
                   void* stream) {
  if (B < 0 || H < 1 || m < 1 || m2 < 1 || k < 0 || W < 0 || R < 1 || R < W || R < m ||
      R < m2 || N_cap < 0 || N2_cap < 0 || max_blocks < 0 || max_blocks2 < 0 ||
      !plain_dtype(o_dtype))
    return SA_ERR_INVALID_ARG;
  if (d != 128 || HI != 64 || dI != 64 || H > 64 || m > 128 || m2 > 128)
    return SA_ERR_UNSUPPORTED;
  if (!q || !q_idx || !w || !q_hca || !q_pos || !k_raw || !v_raw || !ik_raw || !z || !hk_raw ||
      !hv_raw || !hz || !blk_lo || !blk_hi || !hblk_lo || !hblk_hi || !k_c || !v_c || !ik_c ||
      !hk_c || !hv_c || !o || !lse || !ho || !hlse || (k > 0 && !idx))
    return SA_ERR_INVALID_ARG;
  if (!al16(q) || !al16(q_idx) || !al16(w) || !al16(q_hca) || !al16(k_raw) || !al16(v_raw) ||
      !al16(ik_raw) || !al16(hk_raw) || !al16(hv_raw) || !al16(k_c) || !al16(v_c) ||
      !al16(ik_c) || !al16(hk_c) || !al16(hv_c) || !al16(o) || !al16(ho) || !al16(ws))
    return SA_ERR_INVALID_ARG;
  if (B == 0) return SA_OK;
  StepArgs a{};
  a.B = B; a.H = H; a.m = m; a.k = k; a.W = W; a.m2 = m2; a.sm_scale = sm_scale;
  a.q = q; a.q_idx = q_idx; a.w = w; a.q_hca = q_hca; a.q_pos = q_pos;
  a.k_raw = k_raw; a.v_raw = v_raw; a.ik_raw = ik_raw; a.z = z;
  a.hk_raw = hk_raw; a.hv_raw = hv_raw; a.hz = hz; a.R = R;
  a.blk_lo = blk_lo; a.blk_hi = blk_hi; a.max_blocks = max_blocks;
  a.hblk_lo = hblk_lo; a.hblk_hi = hblk_hi; a.max_blocks2 = max_blocks2;
  a.k_c = k_c; a.v_c = v_c; a.ik_c = ik_c; a.N_cap = N_cap;
  a.hk_c = hk_c; a.hv_c = hv_c; a.N2_cap = N2_cap;
  a.idx = idx; a.o_dtype = o_dtype; a.o = o; a.lse = lse; a.ho = ho; a.hlse = hlse; a.err = err;
  size_t offs[7], total = 0;
  if (!step_layout(a, offs, &total)) return SA_ERR_UNSUPPORTED;
  if (!ws || ws_bytes < total) return SA_ERR_INVALID_ARG;
  char* base = static_cast<char*>(ws);
  a.ctr = reinterpret_cast<int*>(base + offs[0]);
  a.keys = reinterpret_cast<uint32_t*>(base + offs[1]);
  a.part_o = reinterpret_cast<float*>(base + offs[2]);
  a.part_lse = reinterpret_cast<float*>(base + offs[3]);
  a.hpart_o = reinterpret_cast<float*>(base + offs[4]);
  a.hpart_lse = reinterpret_cast<float*>(base + offs[5]);
  a.tk_cand = reinterpret_cast<uint32_t*>(base + offs[6]);
  return status_of(launch_decode_step(a, static_cast<cudaStream_t>(stream)));
}

namespace {
// Shared checks and launch of the two attention backward calls.
int attention_backward(AttnBwdArgs& a, int64_t n_keys_max, cudaStream_t st) {
  if (!plain_dtype(a.dtype) || a.B < 0 || a.T < 0 || a.H <= 0 || a.d <= 0 || a.d > 256 ||
      a.d % 4 || a.m < 1 || a.k < 0 || a.W < 0 || a.N_cap < 0 || a.R < 1 || a.R < a.W)
    return SA_ERR_INVALID_ARG;
  if (!a.q || !a.q_pos || !a.kr || !a.vr || !a.o || !a.lse || !a.dout || !a.dq || !a.dkr ||
      !a.dvr || ((a.gather ? a.k > 0 : a.N_cap > 0) && (!a.kc || !a.vc || !a.dkc || !a.dvc)) ||
      (a.gather && a.k > 0 && !a.idx))
    return SA_ERR_INVALID_ARG;
  if (attend_backward_smem(a.H, a.d) > 227 * 1024) return SA_ERR_UNSUPPORTED;
  const int64_t rows = (int64_t)a.B * a.T;
  if (rows == 0) return SA_OK;
  const int tile = attend_backward_key_tile();
  const int tiles = (int)std::max<int64_t>(1, (n_keys_max + tile - 1) / tile);
  const int64_t want = std::max<int64_t>(1, (2 * (int64_t)device_sms() + rows - 1) / rows);
  const int ns = (int)std::min<int64_t>(want, tiles);
  a.split_tiles = (tiles + ns - 1) / ns;
  a.nsplit = (tiles + a.split_tiles - 1) / a.split_tiles;
  return status_of(launch_attend_backward(a, st));
}
}  // namespace

int csa_attend_backward(int dtype, int B, int T, int H, int d, int m, int k, int W,
                        float sm_scale, const void* q, const int32_t* q_pos, const void* k_c,
                        const void* v_c, int N_cap, const int32_t* idx, const void* k_raw,
                        const void* v_raw, int R, const float* o, const float* lse,
                        const float* dout, float* dq, float* dk_c, float* dv_c, float* dk_raw,
                        float* dv_raw, int32_t* err, void* stream) {
  AttnBwdArgs a{};
  a.dtype = dtype; a.B = B; a.T = T; a.H = H; a.d = d; a.sm_scale = sm_scale;
  a.q = q; a.q_pos = q_pos; a.kc = k_c; a.vc = v_c; a.N_cap = N_cap; a.idx = idx;
  a.gather = 1; a.k = k; a.m = m; a.kr = k_raw; a.vr = v_raw; a.R = R; a.W = W;
  a.o = o; a.lse = lse; a.dout = dout; a.dq = dq; a.dkc = dk_c; a.dvc = dv_c;
  a.dkr = dk_raw; a.dvr = dv_raw; a.err = err;
  return attention_backward(a, (int64_t)std::min(k, N_cap) + W, static_cast<cudaStream_t>(stream));
}

int hca_attend_backward(int dtype, int B, int T, int H, int d, int m2, int W, float sm_scale,
                        const void* q, const int32_t* q_pos, const void* hk_c, const void* hv_c,
                        int N2_cap, const void* k_raw, const void* v_raw, int R, const float* o,
                        const float* lse, const float* dout, float* dq, float* dhk_c,
                        float* dhv_c, float* dk_raw, float* dv_raw, int32_t* err,
                        void* stream) {
  AttnBwdArgs a{};
  a.dtype = dtype; a.B = B; a.T = T; a.H = H; a.d = d; a.sm_scale = sm_scale;
  a.q = q; a.q_pos = q_pos; a.kc = hk_c; a.vc = hv_c; a.N_cap = N2_cap; a.idx = nullptr;
  a.gather = 0; a.k = 0; a.m = m2; a.kr = k_raw; a.vr = v_raw; a.R = R; a.W = W;
  a.o = o; a.lse = lse; a.dout = dout; a.dq = dq; a.dkc = dhk_c; a.dvc = dhv_c;
  a.dkr = dk_raw; a.dvr = dv_raw; a.err = err;
  return attention_backward(a, (int64_t)N2_cap + W, static_cast<cudaStream_t>(stream));
}

int sa_compress_backward(int dtype, int B, int d, int m, const void* k_raw, const void* v_raw,
                         const float* z, int R, const int32_t* blk_lo, const int32_t* blk_hi,
                         int max_blocks, const float* dk_c, const float* dv_c, int N_cap,
                         float* dk_raw, float* dv_raw, float* dz, int32_t* err, void* stream) {
  if (!plain_dtype(dtype) || B < 0 || d <= 0 || m < 1 || R < m || max_blocks < 0 || N_cap < 0)
    return SA_ERR_INVALID_ARG;
  if (B == 0 || max_blocks == 0) return SA_OK;
  if (!k_raw || !v_raw || !z || !blk_lo || !blk_hi || !dk_c || !dv_c || !dk_raw || !dv_raw ||
      !dz)
    return SA_ERR_INVALID_ARG;
  if (2 * (size_t)m * sizeof(float) > 48 * 1024) return SA_ERR_UNSUPPORTED;
  CompressBwdArgs a{dtype, B, d, m, k_raw, v_raw, z, R, blk_lo, blk_hi, max_blocks, dk_c, dv_c,
                    N_cap, dk_raw, dv_raw, dz, err};
  return status_of(launch_compress_backward(a, static_cast<cudaStream_t>(stream)));
}

int sa_mxfp4_quantize(const void* x, int64_t nblk, void* codes, void* scales, void* stream) {
  if (nblk < 0 || (nblk > 0 && (!x || !codes || !scales))) return SA_ERR_INVALID_ARG;
  if (nblk == 0) return SA_OK;
  return status_of(launch_mxfp4_quantize(x, nblk, codes, scales, static_cast<cudaStream_t>(stream)));
}

int attn_merge(int n, const float* const* o_parts, const float* const* lse_parts, int64_t rows,
               int d, void* o, int o_dtype, float* lse, int32_t* err, void* stream) {
  (void)err;
  if (n < 1 || n > 8 || rows < 0 || d <= 0 || !o_parts || !lse_parts || !o || !lse ||
      !plain_dtype(o_dtype))
    return SA_ERR_INVALID_ARG;
  MergeArgs a{};
  a.n = n;
  for (int i = 0; i < n; ++i) {
    if (!o_parts[i] || !lse_parts[i]) return SA_ERR_INVALID_ARG;
    a.o_parts[i] = o_parts[i];
    a.lse_parts[i] = lse_parts[i];
  }
  a.rows = rows; a.d = d; a.o = o; a.o_dtype = o_dtype; a.lse = lse;
  return status_of(launch_merge(a, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
