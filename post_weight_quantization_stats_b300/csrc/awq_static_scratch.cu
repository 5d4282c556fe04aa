// awq_search_scale_static: the alpha search for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc on the path where they run the search: code running under
// a strict memory budget that was fixed at start-up, plug-ins that receive a device but no
// allocator, or processes where another runtime owns all allocations. This entry point gives
// them the same search with its scratch taken from a fixed array compiled into this library.
//
// The scratch lives in a file-scope static __device__ array of AWQ_SEARCH_STATIC_SCRATCH_BYTES.
// Every GPU that loads this library holds that array until the process exits. In host code the
// array's name is only a host-side stand-in, so the device address is looked up once per device
// with cudaGetSymbolAddress and passed to the kernels.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/awq.h"

namespace awq {
size_t search_workspace_min_bytes(int64_t N, int64_t K, int64_t T, int32_t n_alpha,
                                  awq_qcfg_t cfg);
awq_status_t search_check_args(const void* W_f16, int64_t N, int64_t K, const void* X_f16,
                               int64_t T, const float* mean_abs, const float* alphas,
                               int32_t n_alpha, awq_qcfg_t cfg, const float* err_out,
                               const int32_t* best_idx, const float* s_out,
                               const float* inv_s_out);
}

namespace {

static __device__ __align__(256) unsigned char g_search_scratch[AWQ_SEARCH_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device; the first call on a device looks
// it up (this may load the library's device code on that device).
awq_status_t scratch_for_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return AWQ_ERR_NO_DEVICE;
  }
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    const cudaError_t rc = cudaGetSymbolAddress(&ptr, g_search_scratch);
    if (rc != cudaSuccess || ptr == nullptr) {
      cudaGetLastError();
      return AWQ_ERR_CUDA;
    }
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return AWQ_OK;
}

}  // namespace

extern "C" awq_status_t awq_search_scale_static(const void* W_f16, int64_t N, int64_t K,
                                                const void* X_f16, int64_t T,
                                                const float* mean_abs, const float* alphas,
                                                int32_t n_alpha, awq_qcfg_t cfg, float* err_out,
                                                int32_t* best_idx, float* s_out,
                                                float* inv_s_out, awq_stream_t stream) {
  // the workspace search's own argument checks first, so a bad pointer, size or alignment
  // gets the same error here as there; only valid inputs can be refused for their size
  const awq_status_t valid = awq::search_check_args(W_f16, N, K, X_f16, T, mean_abs, alphas,
                                                    n_alpha, cfg, err_out, best_idx, s_out,
                                                    inv_s_out);
  if (valid != AWQ_OK) return valid;
  // the smallest workspace the search runs with (one residual buffer, candidates in order)
  const size_t need = awq::search_workspace_min_bytes(N, K, T, n_alpha, cfg);
  if (need == 0 || need > static_cast<size_t>(AWQ_SEARCH_STATIC_SCRATCH_BYTES))
    return AWQ_ERR_WORKSPACE;
  void* scratch = nullptr;
  const awq_status_t st = scratch_for_current_device(&scratch);
  if (st != AWQ_OK) return st;
  return awq_search_scale(W_f16, N, K, X_f16, T, mean_abs, alphas, n_alpha, cfg, scratch,
                          static_cast<size_t>(AWQ_SEARCH_STATIC_SCRATCH_BYTES), err_out, best_idx,
                          s_out, inv_s_out, stream);
}
