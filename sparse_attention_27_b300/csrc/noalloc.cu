// csa_index_topk_noalloc: the indexer + top-k call for callers that cannot
// hand the library any scratch memory.  The fp32 score array that
// csa_index_topk keeps in the caller's workspace lives here instead, in a
// file-scope device array of fixed size that every GPU which loads the
// library holds until the process exits.
//
// Host code cannot pass g_noalloc_scores to a kernel by name: on the host
// that name is only a stand-in for the device variable, not a device
// address.  The device address is looked up once per device with
// cudaGetSymbolAddress (with that device current) and cached.
#include <mutex>

#include "kernels.cuh"

namespace sa {

// The score scratch: B * T * N_cap fp32 scores at most (8 MiB).
constexpr int64_t kNoAllocMaxScores = SA_NOALLOC_MAX_SCORES;
static __device__ __align__(256) float g_noalloc_scores[kNoAllocMaxScores];

namespace {

constexpr int kMaxDevices = 64;

struct DeviceScratch {
  float* scores = nullptr;
  int num_sms = 0;
};

// Device address of the scratch array and the SM count of the current
// device, looked up on the first call made with that device current.
int scratch_for_current_device(DeviceScratch* out) {
  static std::mutex mu;
  static DeviceScratch cache[kMaxDevices];
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return SA_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return SA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(mu);
  DeviceScratch& c = cache[dev];
  if (c.scores == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scores) != cudaSuccess || ptr == nullptr) {
      cudaGetLastError();
      return SA_ERR_CUDA;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      return SA_ERR_CUDA;
    }
    c.scores = static_cast<float*>(ptr);
    c.num_sms = n;
  }
  *out = c;
  return SA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int status_of(cudaError_t e) {
  if (e == cudaSuccess) return SA_OK;
  cudaGetLastError();
  return e == cudaErrorNotSupported ? SA_ERR_UNSUPPORTED : SA_ERR_CUDA;
}

}  // namespace
}  // namespace sa

using namespace sa;

extern "C" int csa_index_topk_noalloc(int q_dtype, int B, int T, int HI, int dI, int m, int k,
                                      const void* q_idx, const void* q_scales, const float* w,
                                      const void* ik_c, const void* ik_scales, int N_cap,
                                      const int32_t* q_pos, int32_t* idx, int32_t* err,
                                      void* stream) {
  if (B < 0 || T < 0 || m < 1 || k < 0 || N_cap < 0 || !q_pos || (k > 0 && !idx))
    return SA_ERR_INVALID_ARG;
  if ((int64_t)B * T * N_cap > kNoAllocMaxScores) return SA_ERR_UNSUPPORTED;
  if (!topk_supported(N_cap)) return SA_ERR_UNSUPPORTED;
  if (q_dtype == SA_MXFP4) return SA_ERR_UNSUPPORTED;
  if (q_dtype != SA_F32 && q_dtype != SA_BF16) return SA_ERR_INVALID_ARG;
  if (HI <= 0 || dI <= 0 || !q_idx || !w || !ik_c) return SA_ERR_INVALID_ARG;
  if (!aligned16(q_idx) || !aligned16(w) || !aligned16(ik_c)) return SA_ERR_INVALID_ARG;
  (void)q_scales;
  (void)ik_scales;
  const int64_t rows = (int64_t)B * T;
  if (rows == 0 || k == 0) return SA_OK;
  DeviceScratch s;
  const int st_setup = scratch_for_current_device(&s);
  if (st_setup != SA_OK) return st_setup;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // Every score the top-k reads (entries j < floor((q_pos+1)/m) of each row)
  // is written by the scoring kernel first, so the scratch needs no clearing.
  ScoreArgs sc{q_dtype, B, T, HI, dI, m, q_idx, nullptr, w, ik_c, nullptr, N_cap,
               q_pos, s.scores, (int64_t)N_cap, err};
  cudaError_t e;
  if (score_tc_supported(sc)) {
    e = launch_score_tc(sc, s.num_sms, st);
  } else {
    if ((size_t)HI * dI + HI > 12 * 1024) return SA_ERR_UNSUPPORTED;
    e = launch_score_simt(sc, st);
  }
  if (e != cudaSuccess) return status_of(e);
  TopkArgs ta{s.scores, (int64_t)N_cap, q_pos, (int)rows, m, N_cap, k, idx, err};
  return status_of(launch_topk(ta, s.num_sms, st));
}
