// libawq: host side of the C ABI declared in include/awq.h.
//
// Every entry point validates its arguments on the host (no CUDA call is made for a rejected
// call), then enqueues its kernels on the caller's stream. The library allocates no device
// memory: the search's scratch is the caller's workspace, the device status word is a static
// __device__ variable.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/awq.h"
#include "awq_device.cuh"
#include "calib_stats.cuh"
#include "quant.cuh"
#include "score_gemm.cuh"
#include "w4a16_gemm_tc.cuh"
#include "w4a16_gemv.cuh"

namespace awq {

__device__ int g_status = 0;  // first device-side error of any kernel (AWQ_ERR_TIMEOUT)

namespace {

std::atomic<uint64_t> g_launches{0};
std::atomic<uint64_t> g_wait_limit_ns{2000000000ull};
constexpr int kMaxDevices = 64;
constexpr int kPartialStride = 1024;  // per-alpha slots for per-CTA partial sums

struct DeviceInfo {
  bool ready = false;
  bool ok = false;
  int sms = 0;
  int* status = nullptr;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

// Looks up the current device once: it must be an sm_103 part. Also resolves the device
// address of the status word and the driver's tensor-map encoder.
awq_status_t device_info(DeviceInfo** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return AWQ_ERR_NO_DEVICE;
  }
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    d.ready = true;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return AWQ_ERR_NO_DEVICE;
    }
    if (major != 10 || minor != 3) return AWQ_ERR_NO_DEVICE;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) {
      cudaGetLastError();
      return AWQ_ERR_CUDA;
    }
    d.status = static_cast<int*>(p);
    if (g_encode == nullptr) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult qr;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &qr) != cudaSuccess ||
          qr != cudaDriverEntryPointSuccess || fn == nullptr) {
        cudaGetLastError();
        return AWQ_ERR_CUDA;
      }
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    d.ok = true;
  }
  if (!d.ok) return AWQ_ERR_NO_DEVICE;
  *out = &d;
  return AWQ_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

awq_status_t check_cfg(awq_qcfg_t cfg) {
  if (cfg.group_size != 64 && cfg.group_size != 128) return AWQ_ERR_INVALID_ARG;
  if (cfg.symmetric != 0 && cfg.symmetric != 1) return AWQ_ERR_INVALID_ARG;
  return AWQ_OK;
}

constexpr int64_t kMaxElems = (int64_t{1} << 31) - 1;

awq_status_t check_nk(int64_t N, int64_t K, awq_qcfg_t cfg) {
  if (N < 1 || K < 1) return AWQ_ERR_INVALID_ARG;
  if (K % cfg.group_size != 0) return AWQ_ERR_UNSUPPORTED_SHAPE;
  if (N * K > kMaxElems) return AWQ_ERR_UNSUPPORTED_SHAPE;
  return AWQ_OK;
}

// ------------------------------------------------------------------ launch accounting
//
// Every launch goes through prof_start() / launched(): the launch counter is bumped and, while
// profiling is on, a CUDA event pair brackets the kernel on its own stream.

struct ProfPair {
  int kernel;
  cudaEvent_t start, stop;
};
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<ProfPair> g_prof_pool;  // events are created once and reused
size_t g_prof_used = 0;
cudaEvent_t g_prof_pending = nullptr;

void prof_start(int kernel, cudaStream_t st) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof_pending = nullptr;
  if (!g_prof_on) return;
  if (g_prof_used == g_prof_pool.size()) {
    ProfPair p{kernel, nullptr, nullptr};
    if (cudaEventCreate(&p.start) != cudaSuccess || cudaEventCreate(&p.stop) != cudaSuccess) {
      cudaGetLastError();
      return;
    }
    g_prof_pool.push_back(p);
  }
  ProfPair& p = g_prof_pool[g_prof_used];
  p.kernel = kernel;
  if (cudaEventRecord(p.start, st) != cudaSuccess) {
    cudaGetLastError();
    return;
  }
  g_prof_pending = p.stop;
  ++g_prof_used;
}

awq_status_t launched(int /*kernel*/, cudaStream_t st) {
  const cudaError_t e = cudaGetLastError();
  {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (g_prof_pending) {
      cudaEventRecord(g_prof_pending, st);
      g_prof_pending = nullptr;
    }
  }
  if (e != cudaSuccess) return AWQ_ERR_CUDA;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return AWQ_OK;
}

#define AWQ_TRY(x)                   \
  do {                               \
    const awq_status_t _s = (x);     \
    if (_s != AWQ_OK) return _s;     \
  } while (0)

// 2-D fp16 tensor map of a row-major [rows, cols] matrix (row stride `ld` elements), box
// [box_rows, 64 cols], 128-byte swizzle, out-of-range elements read as zero.
awq_status_t make_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int64_t ld,
                      int box_rows) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2u};
  const cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1u, 1u};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims,
                              strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? AWQ_OK : AWQ_ERR_CUDA;
}

// ------------------------------------------------------------------ launch helpers

awq_status_t launch_calib_stats(const __half* X, int64_t T, int64_t K, int64_t ldx, float* m,
                                cudaStream_t st) {
  dim3 grid(static_cast<unsigned>((K + stats::COLS - 1) / stats::COLS), stats::CLUSTER);
  prof_start(AWQ_K_CALIB_STATS, st);
  stats::calib_stats_kernel<<<grid, stats::THREADS, 0, st>>>(X, static_cast<int>(T),
                                                             static_cast<int>(K), ldx, m);
  return launched(AWQ_K_CALIB_STATS, st);
}

awq_status_t launch_quantize_pack(const __half* W, int64_t N, int64_t K, const float* s,
                                  awq_qcfg_t cfg, uint32_t* q, __half* scales, uint8_t* zeros,
                                  cudaStream_t st) {
  QuantArgs a{W, s, q, scales, cfg.symmetric ? nullptr : zeros, static_cast<int>(N),
              static_cast<int>(K), cfg.symmetric};
  const int64_t words = N * (K / 8);
  const unsigned grid = static_cast<unsigned>((words + 255) / 256);
  prof_start(AWQ_K_QUANTIZE_PACK, st);
  if (cfg.group_size == 128)
    quantize_pack_kernel<128><<<grid, 256, 0, st>>>(a);
  else
    quantize_pack_kernel<64><<<grid, 256, 0, st>>>(a);
  return launched(AWQ_K_QUANTIZE_PACK, st);
}

template <int BN, int G, bool INV>
awq_status_t launch_tc_t(const CUtensorMap& map, const w4tc::Args& a, cudaStream_t st) {
  auto kern = w4tc::w4a16_tc_kernel<BN, G, INV>;
  constexpr int smem = w4tc::Cfg<BN>::SMEM;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
    cudaGetLastError();
    return AWQ_ERR_CUDA;
  }
  dim3 grid(static_cast<unsigned>((a.N + w4tc::BM - 1) / w4tc::BM),
            static_cast<unsigned>((a.M + BN - 1) / BN));
  prof_start(AWQ_K_GEMM_TC, st);
  kern<<<grid, w4tc::THREADS, smem, st>>>(map, a);
  return launched(AWQ_K_GEMM_TC, st);
}

template <int BN>
awq_status_t launch_tc_bn(const __half* X, const w4tc::Args& a, int G, bool inv, cudaStream_t st) {
  CUtensorMap map;
  AWQ_TRY(make_map(&map, X, a.M, a.K, a.K, BN));
  if (G == 128)
    return inv ? launch_tc_t<BN, 128, true>(map, a, st) : launch_tc_t<BN, 128, false>(map, a, st);
  return inv ? launch_tc_t<BN, 64, true>(map, a, st) : launch_tc_t<BN, 64, false>(map, a, st);
}

template <int M>
awq_status_t launch_gemv_m(const gemv::Args& a0, int G, int sms, cudaStream_t st) {
  gemv::Args a = a0;
  const int64_t grid = std::min<int64_t>(2 * static_cast<int64_t>(sms),
                                         std::max<int64_t>(1, (a.N + gemv::R - 1) / gemv::R));
  a.rows_max = static_cast<int>((a.N + grid - 1) / grid) + 1;
  const int64_t ysum_bytes = static_cast<int64_t>(a.rows_max) * M * 4;
  const int64_t budget = 100 * 1024 - ysum_bytes;
  int64_t kc = (budget / (2 * M)) / gemv::STEP_K * gemv::STEP_K;
  const int64_t kpad = (a.K + gemv::STEP_K - 1) / gemv::STEP_K * gemv::STEP_K;
  if (kc > kpad) kc = kpad;
  if (kc < gemv::STEP_K) kc = gemv::STEP_K;
  a.kc = static_cast<int>(kc);
  const size_t smem = static_cast<size_t>(M) * kc * 2 + static_cast<size_t>(ysum_bytes);
  auto kern = (G == 128) ? gemv::gemv_kernel<M, 128> : gemv::gemv_kernel<M, 64>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess) {
    cudaGetLastError();
    return AWQ_ERR_CUDA;
  }
  prof_start(AWQ_K_GEMV, st);
  kern<<<static_cast<unsigned>(grid), gemv::THREADS, smem, st>>>(a);
  return launched(AWQ_K_GEMV, st);
}

// Sum of the per-CTA partials of every alpha in fixed order, the 2^-2p of the residual scale
// and the 1/(T N) of the mean; first minimiser in fp64; copy out s and 1/s of the winner.
__global__ void __launch_bounds__(256) finalize_kernel(const double* partial, int nparts,
                                                       int n_alpha, const unsigned int* absmax,
                                                       double tn, const float* s_grid,
                                                       const float* inv_grid, int K,
                                                       float* err_out, int* best_idx,
                                                       float* s_out, float* inv_s_out) {
  __shared__ double e[64];
  __shared__ int best;
  const int p2 = residual_exponent(*absmax);
  if (threadIdx.x < static_cast<unsigned>(n_alpha)) {
    double sum = 0.0;
    for (int c = 0; c < nparts; ++c) sum += partial[threadIdx.x * kPartialStride + c];
    const double v = ldexp(sum, -2 * p2) / tn;
    e[threadIdx.x] = v;
    err_out[threadIdx.x] = static_cast<float>(v);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int b = 0;
    for (int i = 1; i < n_alpha; ++i)
      if (e[i] < e[b]) b = i;
    best = b;
    *best_idx = b;
  }
  __syncthreads();
  const float* sb = s_grid + static_cast<long long>(best) * K;
  const float* ib = inv_grid + static_cast<long long>(best) * K;
  for (int k = threadIdx.x; k < K; k += blockDim.x) {
    if (s_out) s_out[k] = sb[k];
    if (inv_s_out) inv_s_out[k] = ib[k];
  }
}

struct SearchLayout {
  size_t m, s_grid, inv_grid, absmax, partial, D, total;
};

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

SearchLayout search_layout(int64_t N, int64_t K, int32_t n_alpha) {
  SearchLayout L{};
  size_t off = 0;
  L.m = off;        off = align256(off + sizeof(float) * K);
  L.s_grid = off;   off = align256(off + sizeof(float) * K * n_alpha);
  L.inv_grid = off; off = align256(off + sizeof(float) * K * n_alpha);
  L.absmax = off;   off = align256(off + sizeof(unsigned int));
  L.partial = off;  off = align256(off + sizeof(double) * kPartialStride * n_alpha);
  L.D = off;        off = align256(off + sizeof(__half) * N * K);
  L.total = off;
  return L;
}

}  // namespace
}  // namespace awq

using namespace awq;

extern "C" {

const char* awq_status_string(awq_status_t s) {
  switch (s) {
    case AWQ_OK: return "AWQ_OK";
    case AWQ_ERR_INVALID_ARG: return "AWQ_ERR_INVALID_ARG";
    case AWQ_ERR_UNSUPPORTED_SHAPE: return "AWQ_ERR_UNSUPPORTED_SHAPE";
    case AWQ_ERR_MISALIGNED: return "AWQ_ERR_MISALIGNED";
    case AWQ_ERR_WORKSPACE: return "AWQ_ERR_WORKSPACE";
    case AWQ_ERR_CUDA: return "AWQ_ERR_CUDA";
    case AWQ_ERR_TIMEOUT: return "AWQ_ERR_TIMEOUT";
    case AWQ_ERR_NO_DEVICE: return "AWQ_ERR_NO_DEVICE";
  }
  return "AWQ_ERR_UNKNOWN";
}

uint64_t awq_launch_count(void) { return g_launches.load(); }

uint64_t awq_set_wait_limit_ns(uint64_t limit_ns) { return g_wait_limit_ns.exchange(limit_ns); }

awq_status_t awq_profile_begin(void) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof_on = true;
  g_prof_used = 0;
  g_prof_pending = nullptr;
  return AWQ_OK;
}

awq_status_t awq_profile_end(double* total_ms, uint64_t* launches) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof_on = false;
  if (total_ms)
    for (int i = 0; i < AWQ_K_COUNT; ++i) total_ms[i] = 0.0;
  if (launches)
    for (int i = 0; i < AWQ_K_COUNT; ++i) launches[i] = 0;
  awq_status_t rc = AWQ_OK;
  for (size_t i = 0; i < g_prof_used; ++i) {
    const ProfPair& p = g_prof_pool[i];
    float ms = 0.f;
    if (cudaEventSynchronize(p.stop) != cudaSuccess ||
        cudaEventElapsedTime(&ms, p.start, p.stop) != cudaSuccess) {
      cudaGetLastError();
      rc = AWQ_ERR_CUDA;
      continue;
    }
    if (p.kernel >= 0 && p.kernel < AWQ_K_COUNT) {
      if (total_ms) total_ms[p.kernel] += ms;
      if (launches) launches[p.kernel] += 1;
    }
  }
  g_prof_used = 0;
  return rc;
}

awq_status_t awq_stream_status(awq_stream_t stream) {
  DeviceInfo* d = nullptr;
  AWQ_TRY(device_info(&d));
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return AWQ_ERR_CUDA;
  }
  int v = 0;
  const int zero = 0;
  if (cudaMemcpy(&v, d->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(d->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) {
    cudaGetLastError();
    return AWQ_ERR_CUDA;
  }
  return v == 0 ? AWQ_OK : static_cast<awq_status_t>(v);
}

awq_status_t awq_calib_stats(const void* X_f16, int64_t T, int64_t K, int64_t ldx,
                             float* mean_abs, awq_stream_t stream) {
  if (!X_f16 || !mean_abs || T < 1 || K < 1) return AWQ_ERR_INVALID_ARG;
  if (K % 8 != 0 || ldx < K || ldx % 8 != 0 || T * ldx > kMaxElems) return AWQ_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(X_f16) || !aligned16(mean_abs)) return AWQ_ERR_MISALIGNED;
  DeviceInfo* d = nullptr;
  AWQ_TRY(device_info(&d));
  return launch_calib_stats(static_cast<const __half*>(X_f16), T, K, ldx, mean_abs,
                            reinterpret_cast<cudaStream_t>(stream));
}

awq_status_t awq_quantize_pack(const void* W_f16, int64_t N, int64_t K, const float* s,
                               awq_qcfg_t cfg, uint32_t* qweight, void* scales_f16,
                               uint8_t* zeros, awq_stream_t stream) {
  AWQ_TRY(check_cfg(cfg));
  if (!W_f16 || !qweight || !scales_f16 || (!cfg.symmetric && !zeros)) return AWQ_ERR_INVALID_ARG;
  AWQ_TRY(check_nk(N, K, cfg));
  if (!aligned16(W_f16) || !aligned16(qweight) || !aligned16(scales_f16) ||
      (s && !aligned16(s)) || (zeros && !aligned16(zeros)))
    return AWQ_ERR_MISALIGNED;
  DeviceInfo* d = nullptr;
  AWQ_TRY(device_info(&d));
  return launch_quantize_pack(static_cast<const __half*>(W_f16), N, K, s, cfg, qweight,
                              static_cast<__half*>(scales_f16), zeros,
                              reinterpret_cast<cudaStream_t>(stream));
}

size_t awq_search_workspace_bytes(int64_t N, int64_t K, int64_t T, int32_t n_alpha,
                                  awq_qcfg_t cfg) {
  if (check_cfg(cfg) != AWQ_OK || check_nk(N, K, cfg) != AWQ_OK || T < 1 || n_alpha < 1 ||
      n_alpha > 64)
    return 0;
  return search_layout(N, K, n_alpha).total;
}

awq_status_t awq_search_scale(const void* W_f16, int64_t N, int64_t K, const void* X_f16,
                              int64_t T, const float* mean_abs, const float* alphas,
                              int32_t n_alpha, awq_qcfg_t cfg, void* workspace,
                              size_t ws_bytes, float* err_out, int32_t* best_idx,
                              float* s_out, float* inv_s_out, awq_stream_t stream) {
  AWQ_TRY(check_cfg(cfg));
  if (!W_f16 || !X_f16 || !alphas || !err_out || !best_idx || T < 1) return AWQ_ERR_INVALID_ARG;
  if (n_alpha < 1 || n_alpha > 64) return AWQ_ERR_INVALID_ARG;
  AWQ_TRY(check_nk(N, K, cfg));
  if (T * K > kMaxElems) return AWQ_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(W_f16) || !aligned16(X_f16) || (mean_abs && !aligned16(mean_abs)) ||
      !aligned4(err_out) || !aligned4(best_idx) || (s_out && !aligned16(s_out)) ||
      (inv_s_out && !aligned16(inv_s_out)) || !aligned16(workspace))
    return AWQ_ERR_MISALIGNED;
  const SearchLayout L = search_layout(N, K, n_alpha);
  if (!workspace || ws_bytes < L.total) return AWQ_ERR_WORKSPACE;
  DeviceInfo* d = nullptr;
  AWQ_TRY(device_info(&d));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* m = reinterpret_cast<float*>(ws + L.m);
  float* s_grid = reinterpret_cast<float*>(ws + L.s_grid);
  float* inv_grid = reinterpret_cast<float*>(ws + L.inv_grid);
  unsigned int* absmax = reinterpret_cast<unsigned int*>(ws + L.absmax);
  double* partial = reinterpret_cast<double*>(ws + L.partial);
  __half* D = reinterpret_cast<__half*>(ws + L.D);
  const __half* W = static_cast<const __half*>(W_f16);
  const __half* X = static_cast<const __half*>(X_f16);

  CUtensorMap mapX, mapD;
  AWQ_TRY(make_map(&mapX, X, T, K, K, score::BM));
  AWQ_TRY(make_map(&mapD, D, N, K, K, score::BN));

  // 1. statistic
  const float* mp = mean_abs;
  if (!mp) {
    AWQ_TRY(launch_calib_stats(X, T, K, K, m, st));
    mp = m;
  }
  // 2. scale grid
  GridArgs ga{};
  ga.m = mp;
  ga.s = s_grid;
  ga.inv_s = inv_grid;
  ga.K = static_cast<int>(K);
  ga.n_alpha = n_alpha;
  for (int i = 0; i < n_alpha; ++i) ga.alphas[i] = alphas[i];
  prof_start(AWQ_K_SCALE_GRID, st);
  scale_grid_kernel<<<static_cast<unsigned>((K * n_alpha + 255) / 256), 256, 0, st>>>(ga);
  AWQ_TRY(launched(AWQ_K_SCALE_GRID, st));
  // 3. max |W| for the residual's power-of-two scale
  if (cudaMemsetAsync(absmax, 0, sizeof(unsigned int), st) != cudaSuccess) {
    cudaGetLastError();
    return AWQ_ERR_CUDA;
  }
  const long long n8 = N * K / 8;
  const unsigned agrid = static_cast<unsigned>(std::min<long long>(4LL * d->sms, (n8 + 255) / 256));
  prof_start(AWQ_K_ABSMAX, st);
  absmax_kernel<<<agrid, 256, 0, st>>>(W, n8, absmax);
  AWQ_TRY(launched(AWQ_K_ABSMAX, st));
  // 4. per alpha: residual D = W - Q(W diag s) diag(s)^-1, then sum of squares of X D^T
  if (cudaFuncSetAttribute(score::score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           score::SMEM_BYTES) != cudaSuccess) {
    cudaGetLastError();
    return AWQ_ERR_CUDA;
  }
  score::Params sp{};
  sp.tiles_n = static_cast<int>((N + score::BN - 1) / score::BN);
  const int tiles_m = static_cast<int>((T + score::BM - 1) / score::BM);
  sp.num_tiles = tiles_m * sp.tiles_n;
  sp.num_kb = static_cast<int>((K + score::BK - 1) / score::BK);
  sp.status = d->status;
  sp.limit_ns = g_wait_limit_ns.load();
  const int sgrid = std::min(sp.num_tiles, std::min(d->sms, kPartialStride));
  const unsigned rgrid = static_cast<unsigned>((N * (K / 8) + 255) / 256);
  for (int i = 0; i < n_alpha; ++i) {
    ResidualArgs ra{W, s_grid + static_cast<size_t>(i) * K, inv_grid + static_cast<size_t>(i) * K,
                    absmax, D, static_cast<int>(N), static_cast<int>(K), cfg.symmetric};
    prof_start(AWQ_K_RESIDUAL, st);
    if (cfg.group_size == 128)
      residual_kernel<128><<<rgrid, 256, 0, st>>>(ra);
    else
      residual_kernel<64><<<rgrid, 256, 0, st>>>(ra);
    AWQ_TRY(launched(AWQ_K_RESIDUAL, st));
    sp.partial = partial + static_cast<size_t>(i) * kPartialStride;
    prof_start(AWQ_K_SCORE, st);
    score::score_kernel<<<sgrid, score::THREADS, score::SMEM_BYTES, st>>>(mapX, mapD, sp);
    AWQ_TRY(launched(AWQ_K_SCORE, st));
  }
  // 5. errors, argmin, winning scales
  prof_start(AWQ_K_FINALIZE, st);
  finalize_kernel<<<1, 256, 0, st>>>(partial, sgrid, n_alpha, absmax,
                                     static_cast<double>(T) * static_cast<double>(N), s_grid,
                                     inv_grid, static_cast<int>(K), err_out, best_idx, s_out,
                                     inv_s_out);
  return launched(AWQ_K_FINALIZE, st);
}

awq_status_t awq_w4a16_gemm(const void* X_f16, int64_t M, int64_t N, int64_t K,
                            const uint32_t* qweight, const void* scales_f16,
                            const uint8_t* zeros, const float* inv_s, awq_qcfg_t cfg,
                            void* Y_f16, awq_stream_t stream) {
  AWQ_TRY(check_cfg(cfg));
  if (!X_f16 || !qweight || !scales_f16 || !Y_f16 || (!cfg.symmetric && !zeros) || M < 1)
    return AWQ_ERR_INVALID_ARG;
  AWQ_TRY(check_nk(N, K, cfg));
  if (M * N > kMaxElems || M * K > kMaxElems) return AWQ_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(X_f16) || !aligned16(qweight) || !aligned16(scales_f16) || !aligned16(Y_f16) ||
      (zeros && !aligned16(zeros)) || (inv_s && !aligned16(inv_s)))
    return AWQ_ERR_MISALIGNED;
  DeviceInfo* d = nullptr;
  AWQ_TRY(device_info(&d));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const uint8_t* z = cfg.symmetric ? nullptr : zeros;
  const int G = cfg.group_size;
  if (M <= 8) {
    gemv::Args a{static_cast<const __half*>(X_f16), qweight, static_cast<const __half*>(scales_f16),
                 z, inv_s, static_cast<__half*>(Y_f16), static_cast<int>(M), static_cast<int>(N),
                 static_cast<int>(K), 0, 0};
    switch (M) {
      case 1: return launch_gemv_m<1>(a, G, d->sms, st);
      case 2: return launch_gemv_m<2>(a, G, d->sms, st);
      case 3: return launch_gemv_m<3>(a, G, d->sms, st);
      case 4: return launch_gemv_m<4>(a, G, d->sms, st);
      case 5: return launch_gemv_m<5>(a, G, d->sms, st);
      case 6: return launch_gemv_m<6>(a, G, d->sms, st);
      case 7: return launch_gemv_m<7>(a, G, d->sms, st);
      default: return launch_gemv_m<8>(a, G, d->sms, st);
    }
  }
  w4tc::Args a{qweight, static_cast<const __half*>(scales_f16), z, inv_s,
               static_cast<__half*>(Y_f16), static_cast<int>(M), static_cast<int>(N),
               static_cast<int>(K), static_cast<int>((K + w4tc::BK - 1) / w4tc::BK), d->status,
               g_wait_limit_ns.load()};
  const __half* X = static_cast<const __half*>(X_f16);
  const bool inv = inv_s != nullptr;
  if (M <= 16) return launch_tc_bn<16>(X, a, G, inv, st);
  if (M <= 32) return launch_tc_bn<32>(X, a, G, inv, st);
  if (M <= 64) return launch_tc_bn<64>(X, a, G, inv, st);
  if (M <= 128) return launch_tc_bn<128>(X, a, G, inv, st);
  return launch_tc_bn<256>(X, a, G, inv, st);
}

}  // extern "C"
