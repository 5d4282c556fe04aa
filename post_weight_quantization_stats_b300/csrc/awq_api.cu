// libawq: host side of the C ABI declared in include/awq.h.
//
// Every entry point validates its arguments on the host (no CUDA call is made for a rejected
// call), then enqueues its kernels on the caller's stream. The library allocates no device
// memory: the search's scratch is the caller's workspace, the device status word is a static
// __device__ variable.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <utility>
#include <vector>

#include "../../include/awq.h"
#include "awq_device.cuh"
#include "block_ops.cuh"
#include "calib_stats.cuh"
#include "gram_persistent.cuh"
#include "gram_score.cuh"
#include "quant.cuh"
#include "score_gemm.cuh"
#include "w4a16_gemm_tc.cuh"
#include "w4a16_gemv.cuh"

namespace awq {

__device__ int g_status = 0;  // first device-side error of any kernel (AWQ_ERR_TIMEOUT)

namespace {

std::atomic<uint64_t> g_launches{0};
std::atomic<uint64_t> g_wait_limit_ns{2000000000ull};
std::atomic<int> g_score_mode{AWQ_SCORE_AUTO};
constexpr int kMaxDevices = 64;
constexpr int kPartialStride = 1024;  // per-alpha slots for per-CTA partial sums

struct DeviceInfo {
  bool ready = false;
  bool ok = false;
  int sms = 0;
  int* status = nullptr;
  // the search's second stream (residuals run there, overlapping the scoring GEMM) and the
  // events that order the two streams; created once, on the first call on this device
  cudaStream_t side = nullptr;
  cudaEvent_t fork = nullptr, res_done[2] = {nullptr, nullptr}, score_done[2] = {nullptr, nullptr};
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
    if (cudaStreamCreateWithFlags(&d.side, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&d.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&d.res_done[0], cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&d.res_done[1], cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&d.score_done[0], cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&d.score_done[1], cudaEventDisableTiming) != cudaSuccess) {
      cudaGetLastError();
      return AWQ_ERR_CUDA;
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
  if (cfg.group_size != 32 && cfg.group_size != 64 && cfg.group_size != 128)
    return AWQ_ERR_INVALID_ARG;
  if (cfg.symmetric != 0 && cfg.symmetric != 1) return AWQ_ERR_INVALID_ARG;
  if (cfg.bits != 0 && cfg.bits != 2 && cfg.bits != 3 && cfg.bits != 4) return AWQ_ERR_INVALID_ARG;
  return AWQ_OK;
}

// Code width of a validated configuration (0 means the default, 4).
int cfg_bits(awq_qcfg_t cfg) { return cfg.bits == 0 ? 4 : cfg.bits; }

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

// Drops the event pair prof_start() opened for a launch that did not happen.
void prof_cancel() {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (g_prof_pending) {
    g_prof_pending = nullptr;
    --g_prof_used;
  }
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

// 2-D tensor map of a row-major [rows, cols] matrix of `elem_bytes`-byte elements (row stride
// `ld` elements), box [box_rows, box_cols], no swizzle unless asked, out-of-range elements read
// as zero.
awq_status_t make_map_plain(CUtensorMap* map, CUtensorMapDataType dt, int elem_bytes,
                            const void* base, int64_t rows, int64_t cols, int64_t ld, int box_cols,
                            int box_rows, CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_NONE) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * static_cast<cuuint64_t>(elem_bytes)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1u, 1u};
  const CUresult r = g_encode(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? AWQ_OK : AWQ_ERR_CUDA;
}

// Launch with a cluster of `cz` CTAs along grid z (cz = 1: a plain launch).
template <typename... P, typename... A>
awq_status_t launch_k(void (*kern)(P...), dim3 grid, int threads, size_t smem, int cz,
                      cudaStream_t st, A&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(static_cast<unsigned>(threads));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = static_cast<unsigned>(cz);
  cfg.attrs = attr;
  cfg.numAttrs = cz > 1 ? 1 : 0;
  if (cudaLaunchKernelEx(&cfg, kern, std::forward<A>(args)...) != cudaSuccess) return AWQ_ERR_CUDA;
  return AWQ_OK;
}

// ------------------------------------------------------------------ launch helpers

// squares = false: the statistic mean |x|; true: the channel energy sum x^2 (clipping search)
awq_status_t launch_calib_stats(const __half* X, int64_t T, int64_t K, int64_t ldx, float* m,
                                const DeviceInfo* d, cudaStream_t st, bool squares = false) {
  // boxes of 128 rows x 64 columns of X (row stride ldx); columns past K and rows past T read
  // as zero
  CUtensorMap map;
  AWQ_TRY(make_map_plain(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, X, T, K, ldx, stats::COLS,
                         stats::BOX_ROWS));
  dim3 grid(static_cast<unsigned>((K + stats::COLS - 1) / stats::COLS), stats::CLUSTER);
  prof_start(AWQ_K_CALIB_STATS, st);
  auto kern = squares ? stats::calib_stats_kernel<true> : stats::calib_stats_kernel<false>;
  kern<<<grid, stats::THREADS, 0, st>>>(map, static_cast<int>(T), static_cast<int>(K), m,
                                        d->status, g_wait_limit_ns.load());
  return launched(AWQ_K_CALIB_STATS, st);
}

// Grid of the run-per-thread kernels (quantize_pack_kernel, clip_search_kernel): row blocks on
// x, one group per block on y.
template <int MAXRUN>
dim3 run_grid(int64_t N, int64_t K, int G) {
  const int rows = G == 128 ? RunShape<128, MAXRUN>::ROWS
                            : (G == 64 ? RunShape<64, MAXRUN>::ROWS : RunShape<32, MAXRUN>::ROWS);
  return dim3(static_cast<unsigned>((N + rows - 1) / rows), static_cast<unsigned>(K / G));
}

awq_status_t launch_quantize_pack(const __half* W, int64_t N, int64_t K, const float* s,
                                  awq_qcfg_t cfg, uint32_t* q, __half* scales, uint8_t* zeros,
                                  cudaStream_t st, const float* clip = nullptr) {
  QuantArgs a{W, s, clip, q, scales, cfg.symmetric ? nullptr : zeros, static_cast<int>(N),
              static_cast<int>(K), cfg.symmetric, cfg_bits(cfg)};
  const dim3 grid = run_grid<PACK_RUN>(N, K, cfg.group_size);
  prof_start(AWQ_K_QUANTIZE_PACK, st);
  if (cfg.group_size == 128)
    quantize_pack_kernel<128><<<grid, 256, 0, st>>>(a);
  else if (cfg.group_size == 64)
    quantize_pack_kernel<64><<<grid, 256, 0, st>>>(a);
  else
    quantize_pack_kernel<32><<<grid, 256, 0, st>>>(a);
  return launched(AWQ_K_QUANTIZE_PACK, st);
}

// Tensor-core W4A16, grouped kernel (M <= 16): 120-row tiles, K split over a cluster of up
// to 8 CTAs (whole groups each) so the tiles fill two CTAs per SM.
awq_status_t launch_w4_grouped(const __half* X, const w4tc::Args& a0, int G, int sms,
                               cudaStream_t st) {
  namespace gk = w4tc::grouped;
  w4tc::Args a = a0;
  const int tiles = (a.N + gk::ROWS - 1) / gk::ROWS;
  const int nraw = (a.K + gk::RK - 1) / gk::RK;   // K splits are whole 256-channel raw stages
  int splits = 1;
  for (int sp = 1; sp <= 8; ++sp)
    if (tiles * sp <= 2 * sms && sp <= nraw) splits = sp;
  a.splits = splits;
  CUtensorMap mq, mx;
  const int mt = a.M <= 1 ? 1 : a.M <= 2 ? 2 : a.M <= 4 ? 4 : a.M <= 8 ? 8 : 16;
  AWQ_TRY(make_map_plain(&mq, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, a.Q, a.N, a.K / 8, a.K / 8,
                         gk::RK / 8, gk::ROWS, CU_TENSOR_MAP_SWIZZLE_128B));
  AWQ_TRY(make_map_plain(&mx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, X, a.M, a.K, a.K, gk::RK, mt));
  using KernT = void (*)(CUtensorMap, CUtensorMap, w4tc::Args);
  KernT kern;
  if (G == 128)
    kern = mt == 1 ? gk::grouped_kernel<128, 1> : mt == 2 ? gk::grouped_kernel<128, 2>
         : mt == 4 ? gk::grouped_kernel<128, 4> : mt == 8 ? gk::grouped_kernel<128, 8>
                   : gk::grouped_kernel<128, 16>;
  else
    kern = mt == 1 ? gk::grouped_kernel<64, 1> : mt == 2 ? gk::grouped_kernel<64, 2>
         : mt == 4 ? gk::grouped_kernel<64, 4> : mt == 8 ? gk::grouped_kernel<64, 8>
                   : gk::grouped_kernel<64, 16>;
  const int smem = gk::smem_bytes(mt);
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
    cudaGetLastError();
    return AWQ_ERR_CUDA;
  }
  prof_start(AWQ_K_GEMM_TC, st);
  const awq_status_t rc = launch_k(kern, dim3(static_cast<unsigned>(tiles), 1, static_cast<unsigned>(splits)),
                                   w4tc::THREADS, static_cast<size_t>(smem), splits, st, mq, mx, a);
  const awq_status_t rl = launched(AWQ_K_GEMM_TC, st);
  return rc != AWQ_OK ? rc : rl;
}

// Tensor-core W4A16, dequant kernel (any M; used above 16 tokens): token tile BN by M, K split
// over a cluster while the tiles alone leave SMs idle (each CTA keeps >= 2 stages).
template <int BN>
awq_status_t launch_w4_dequant_bn(const __half* X, const w4tc::Args& a0, int G, int sms,
                                  cudaStream_t st) {
  namespace dk = w4tc::dequant;
  using C = dk::Cfg<BN>;
  w4tc::Args a = a0;
  const int tiles_n = (a.N + w4tc::BM - 1) / w4tc::BM, tiles_m = (a.M + BN - 1) / BN;
  const int nkb = (a.K + dk::BK - 1) / dk::BK;
  int splits = 1;
  for (int sp = 1; sp <= 8; ++sp)
    if (tiles_n * tiles_m * sp <= sms && nkb >= 2 * sp) splits = sp;
  a.splits = splits;
  CUtensorMap mq, mx;
  AWQ_TRY(make_map_plain(&mq, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, a.Q, a.N, a.K / 8, a.K / 8,
                         dk::BK / 8, w4tc::BM));
  AWQ_TRY(make_map(&mx, X, a.M, a.K, a.K, BN));
  auto kern = G == 128 ? dk::dequant_kernel<BN, 128>
              : G == 64 ? dk::dequant_kernel<BN, 64> : dk::dequant_kernel<BN, 32>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess) {
    cudaGetLastError();
    return AWQ_ERR_CUDA;
  }
  prof_start(AWQ_K_GEMM_TC, st);
  const awq_status_t rc = launch_k(kern, dim3(static_cast<unsigned>(tiles_n), static_cast<unsigned>(tiles_m),
                                              static_cast<unsigned>(splits)),
                                   w4tc::THREADS, static_cast<size_t>(C::SMEM), splits, st, mq, mx, a);
  const awq_status_t rl = launched(AWQ_K_GEMM_TC, st);
  return rc != AWQ_OK ? rc : rl;
}

awq_status_t launch_w4_dequant(const __half* X, const w4tc::Args& a, int G, int sms, cudaStream_t st) {
  if (a.M <= 32) return launch_w4_dequant_bn<32>(X, a, G, sms, st);
  if (a.M <= 64) return launch_w4_dequant_bn<64>(X, a, G, sms, st);
  if (a.M <= 128) return launch_w4_dequant_bn<128>(X, a, G, sms, st);
  return launch_w4_dequant_bn<256>(X, a, G, sms, st);
}

// Launch shape of the decode GEMV: one CTA per SM (at most one per output row); the K parts
// follow from the items each lane holds; a stage holds at least one row per row group and about
// 32 KB; the ring is as deep as shared memory allows (at least 2 stages). Shapes that do not fit
// (K above 32 * 32 * IPL * CWARPS channels, or too many group parameters per CTA) return
// AWQ_ERR_UNSUPPORTED_SHAPE and go to the tensor-core kernel instead.
awq_status_t gemv_shape(gemv::Args& a, int G, int sms) {
  const int grid = static_cast<int>(std::min<int64_t>(sms, a.N));
  a.rows_max = (a.N + grid - 1) / grid;
  const int ipl = gemv::items_per_lane(a.M);
  const int items = a.K / gemv::ITEM_CH;
  a.parts = (items + 32 * ipl - 1) / (32 * ipl);
  if (a.parts > gemv::CWARPS) return AWQ_ERR_UNSUPPORTED_SHAPE;
  a.row_groups = gemv::CWARPS / a.parts;
  const int row_bytes = a.K / 2;
  a.pstride = a.K / G + 1;
  // Group parameters by TMA boxes where the arrays allow it: the rows of a CTA, its start
  // rounded down to 16, fit one box (at most 256 columns), and the row strides of the steps
  // (2 N bytes) and zero points (N bytes) are multiples of 16 bytes. The box width is 32 j + 16,
  // so the 8 groups a warp's lanes read per row fall on distinct banks for the zero points and
  // on two-way shared banks for the steps.
  const int ng = a.K / G;
  const int bc = (a.rows_max + 15 + 15) / 32 * 32 + 16;
  const bool box_ok = bc <= 256 && a.N % (a.zeros ? 16 : 8) == 0;
  // Rows per stage: about 32 KB, for M = 1 preferably a multiple of 2 RG (every consumer warp
  // then takes its rows two at a time; with more tokens the registers go to them instead), else
  // a multiple of RG. The ring is as deep as shared memory allows
  // (at least 2 stages, no more than the CTA's rows fill).
  auto fit = [&](int unit) {
    a.rows_stage = std::max(unit, (32768 / row_bytes + unit / 2) / unit * unit);
    a.stage_bytes = a.rows_stage * row_bytes;
    const int stages_needed = (a.rows_max + a.rows_stage - 1) / a.rows_stage;
    a.nstages = std::max(2, std::min(gemv::MAX_STAGES, stages_needed));
    while (a.nstages > 2 && gemv::smem_bytes(a) > static_cast<size_t>(gemv::SMEM_BUDGET)) --a.nstages;
    return gemv::smem_bytes(a) <= static_cast<size_t>(gemv::SMEM_BUDGET);
  };
  // Parameter boxes before plain parameter loads, paired rows before single rows.
  auto fit_any = [&](int direct) {
    a.x_direct = direct;
    for (int box = box_ok ? 1 : 0; box >= 0; --box) {
      a.pbox_cols = box ? bc : 0;
      a.pbox_groups = box ? std::min(ng, 256) : 0;
      if ((a.M == 1 && fit(2 * a.row_groups)) || fit(a.row_groups)) return true;
    }
    return false;
  };
  // Activation planes staged once per CTA, unless K is long enough that they leave fewer than
  // four ring stages: then, where at most two row groups share a lane's activations, each lane
  // converts its own (twice the conversion work at worst, but 2 M K bytes of shared memory go
  // to the weight ring), if that puts more weight bytes in flight.
  const bool staged = fit_any(0);
  if (staged && (a.nstages >= 4 || a.row_groups > 2)) return AWQ_OK;
  if (a.row_groups <= 2) {
    const gemv::Args keep = a;
    if (fit_any(1) && (!staged || a.nstages * a.stage_bytes > keep.nstages * keep.stage_bytes))
      return AWQ_OK;
    a = keep;
  }
  return staged ? AWQ_OK : AWQ_ERR_UNSUPPORTED_SHAPE;
}

template <int M>
awq_status_t launch_gemv_m(const gemv::Args& a, int G, cudaStream_t st) {
  const size_t smem = gemv::smem_bytes(a);
  // tensor maps of the group parameters [K/G, N] (unused when they are staged by plain loads)
  CUtensorMap tmS, tmZ;
  std::memset(&tmS, 0, sizeof(tmS));
  std::memset(&tmZ, 0, sizeof(tmZ));
  if (a.pbox_cols) {
    AWQ_TRY(make_map_plain(&tmS, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, a.scales, a.K / G, a.N, a.N,
                           a.pbox_cols, a.pbox_groups));
    if (a.zeros)
      AWQ_TRY(make_map_plain(&tmZ, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.zeros, a.K / G, a.N, a.N,
                             a.pbox_cols, a.pbox_groups));
  }
  auto kern = G == 128 ? gemv::gemv_kernel<M, 128>
              : G == 64 ? gemv::gemv_kernel<M, 64> : gemv::gemv_kernel<M, 32>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess) {
    cudaGetLastError();
    return AWQ_ERR_CUDA;
  }
  const unsigned grid = static_cast<unsigned>((a.N + a.rows_max - 1) / a.rows_max);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(gemv::THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see the kernel's header
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  prof_start(AWQ_K_GEMV, st);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, tmS, tmZ, a);
  const awq_status_t rl = launched(AWQ_K_GEMV, st);
  return e != cudaSuccess ? AWQ_ERR_CUDA : rl;
}

// Sum of the per-CTA partials of every alpha in a fixed order (one warp per alpha, 32 warps:
// lane l adds partials l, l + 32, ..., then a fixed butterfly), the 2^-2p of the residual scale
// and the 1/(T N) of the mean; first minimiser in fp64; copy out s and 1/s of the winner.
// With the Gram schedule (hmax != NULL) the partials hold 2^-h sum_n d^T H' d, i.e. half of
// 2^-h sum_n d^T H d: the factor 2^(1 + h) restores it.
__global__ void __launch_bounds__(1024) finalize_kernel(const double* partial, int nparts,
                                                       int n_alpha, const unsigned int* absmax,
                                                       const unsigned int* hmax,
                                                       double tn, const float* s_grid,
                                                       const float* inv_grid, int K,
                                                       float* err_out, int* best_idx,
                                                       float* s_out, float* inv_s_out) {
  __shared__ double e[64];
  __shared__ int best;
  const int p2 = residual_exponent(*absmax);
  const int h = hmax ? 1 + gram::gram_exponent(*hmax) : 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = warp; i < n_alpha; i += static_cast<int>(blockDim.x >> 5)) {
    double sum = 0.0;
    for (int c0 = lane; c0 < nparts; c0 += 8 * 32) {  // eight loads in flight, added in order
      double v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int c = c0 + 32 * u;
        v[u] = c < nparts ? partial[i * kPartialStride + c] : 0.0;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) sum += v[u];
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane == 0) {
      const double v = ldexp(sum, h - 2 * p2) / tn;
      e[i] = v;
      err_out[i] = static_cast<float>(v);
    }
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
  // K is a multiple of 64 and every buffer 16-byte aligned: copy float4s, four in flight
  const float4* sb = reinterpret_cast<const float4*>(s_grid + static_cast<long long>(best) * K);
  const float4* ib = reinterpret_cast<const float4*>(inv_grid + static_cast<long long>(best) * K);
  const int K4 = K / 4;
  for (int k0 = threadIdx.x; k0 < K4; k0 += 4 * blockDim.x) {
    float4 a[4], b[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int k = k0 + u * blockDim.x;
      if (k < K4) {
        a[u] = sb[k];
        b[u] = ib[k];
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int k = k0 + u * blockDim.x;
      if (k < K4) {
        if (s_out) reinterpret_cast<float4*>(s_out)[k] = a[u];
        if (inv_s_out) reinterpret_cast<float4*>(inv_s_out)[k] = b[u];
      }
    }
  }
}

struct SearchLayout {
  size_t m, s_grid, inv_grid, absmax, partial, D, D2, min_total, total;
  size_t hmax, colsq, xt, bmat, sync, gram_total;  // Gram schedule: H from X^T, its triangle
  int64_t Tp;
};

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

SearchLayout search_layout(int64_t N, int64_t K, int64_t T, int32_t n_alpha) {
  SearchLayout L{};
  size_t off = 0;
  L.m = off;        off = align256(off + sizeof(float) * K);
  L.s_grid = off;   off = align256(off + sizeof(float) * K * n_alpha);
  L.inv_grid = off; off = align256(off + sizeof(float) * K * n_alpha);
  L.absmax = off;   off = align256(off + sizeof(unsigned int));
  L.partial = off;  off = align256(off + sizeof(double) * kPartialStride * n_alpha);
  L.D = off;        off = align256(off + sizeof(__half) * N * K);
  L.min_total = off;   // one residual buffer: the alpha candidates run one after the other
  L.D2 = off;       off = align256(off + sizeof(__half) * N * K);
  L.total = off;       // two: the next candidate's residual overlaps this one's scoring
  L.Tp = (T + gram::TOK_BLOCK - 1) / gram::TOK_BLOCK * gram::TOK_BLOCK;
  L.hmax = off;     off = align256(off + sizeof(unsigned int));
  L.colsq = off;    off = align256(off + sizeof(float) * (L.Tp / gram::TOK_BLOCK) * K);
  L.xt = off;       off = align256(off + sizeof(__half) * K * L.Tp);
  L.bmat = off;     off = align256(off + sizeof(__half) * K * K);
  L.sync = off;     off = align256(off + sizeof(unsigned int) * (2 * n_alpha + 1));
  L.gram_total = off;  // Gram schedule (two residual buffers as well)
  return L;
}

// Shapes the Gram schedule handles: K a multiple of 64 (the transpose's channel blocks and the
// triangle's epilogue work in 64- and 32-channel pieces), 32-bit element offsets for X^T and H,
// a transpose grid within the launch limits.
bool gram_shape_ok(int64_t K, int64_t T) {
  const int64_t Tp = (T + gram::TOK_BLOCK - 1) / gram::TOK_BLOCK * gram::TOK_BLOCK;
  return K % 64 == 0 && K * Tp <= kMaxElems && K * K <= kMaxElems &&
         Tp / gram::TOK_BLOCK <= 65535;
}

// Tile counts of the Gram schedule's two kernel modes.
int gram_tiles(int64_t K) {  // GRAM mode: row tiles kt = 0..KT-1 take kt / 2 + 1 tiles each
  const int KT = static_cast<int>((K + gram::BM - 1) / gram::BM);
  int n = 0;
  for (int kt = 0; kt < KT; ++kt) n += kt / 2 + 1;
  return n;
}

// Whether scoring through H = X^T X takes fewer tensor-core tile steps (one 128 x 256 x 64
// MMA block each, counted on the most loaded of `sms` CTAs) than the direct X D^T, including
// forming H once and the transpose of X (converted at about 1.5 MB of traffic per step). The
// direct count is weighted by 1.2: its residuals run as separate kernels beside the scoring
// GEMM and slow it down, while the Gram launch builds them in its own spare warps (measured
// over layers from 256 x 512 to 28672 x 8192 with 64 to 8192 tokens: the weight picks the
// faster schedule on all but near-equal cases).
bool gram_pays(int64_t N, int64_t K, int64_t T, int32_t n_alpha, int sms) {
  const int64_t P = sms;
  const int64_t direct_tiles = ((T + 127) / 128) * ((N + 255) / 256);
  const double direct = static_cast<double>((direct_tiles + P - 1) / P) * ((K + 63) / 64);
  const int64_t RT = (N + gram::BM - 1) / gram::BM, CT = (K + gram::BN - 1) / gram::BN;
  std::vector<int64_t> load(static_cast<size_t>(P), 0);
  for (int64_t u = 0; u < RT * CT; ++u) {  // the kernel's serpentine deal, longest tiles first
    const int64_t ct = CT - 1 - u / RT, r = u / P, pos = u % P;
    const int64_t cta = (r & 1) ? P - 1 - pos : pos;
    load[static_cast<size_t>(cta)] += (std::min<int64_t>((ct + 1) * gram::BN, K) + 63) / 64;
  }
  int64_t per_alpha = 0;
  for (int64_t v : load) per_alpha = std::max(per_alpha, v);
  const int64_t Tp = (T + 63) / 64 * 64;
  const double once = static_cast<double>((gram_tiles(K) + P - 1) / P) * (Tp / 64) +
                      4.0 * static_cast<double>(T) * static_cast<double>(K) / 1.5e6;
  return static_cast<double>(n_alpha) * per_alpha + once < 1.2 * static_cast<double>(n_alpha) * direct;
}

// The persistent Gram-schedule search (gram_persistent.cuh): one cooperative launch, one CTA per
// SM, after the counters it synchronises on are zeroed. *done is false (and nothing is left
// pending) when the device refuses the cooperative launch; the caller then takes the
// one-launch-per-phase path.
awq_status_t launch_search_persistent(int G, DeviceInfo* d, const SearchLayout& L, uint8_t* ws,
                                      const __half* Xt, __half* Bm, const unsigned int* hmax,
                                      __half* const* Dbuf, const __half* W,
                                      const unsigned int* absmax, const float* s_grid,
                                      const float* inv_grid, double* partial, int64_t N,
                                      int64_t K, int n_alpha, int symmetric, int bits,
                                      bool* done, cudaStream_t st);

// The schedule a search with `ws_bytes` of workspace takes (ws_bytes = SIZE_MAX: the one the
// library prefers). Returns false if the workspace is too small.
enum class Sched { SERIAL, OVERLAP, GRAM };
bool pick_schedule(int64_t N, int64_t K, int64_t T, int32_t n_alpha, size_t ws_bytes, int sms,
                   const SearchLayout& L, Sched* out) {
  const int mode = g_score_mode.load();
  const bool gram_ok = gram_shape_ok(K, T);
  const bool forced = mode == AWQ_SCORE_GRAM || mode == AWQ_SCORE_GRAM_LAUNCHES;
  const bool want_gram = gram_ok && (forced ||
                                     (mode == AWQ_SCORE_AUTO && gram_pays(N, K, T, n_alpha, sms)));
  if (forced) {
    if (!gram_ok || ws_bytes < L.gram_total) return false;
    *out = Sched::GRAM;
    return true;
  }
  if (want_gram && ws_bytes >= L.gram_total) *out = Sched::GRAM;
  else if (ws_bytes >= L.total) *out = Sched::OVERLAP;
  else if (ws_bytes >= L.min_total) *out = Sched::SERIAL;
  else return false;
  return true;
}

awq_status_t launch_search_persistent(int G, DeviceInfo* d, const SearchLayout& L, uint8_t* ws,
                                      const __half* Xt, __half* Bm, const unsigned int* hmax,
                                      __half* const* Dbuf, const __half* W,
                                      const unsigned int* absmax, const float* s_grid,
                                      const float* inv_grid, double* partial, int64_t N,
                                      int64_t K, int n_alpha, int symmetric, int bits,
                                      bool* done, cudaStream_t st) {
  *done = false;
  CUtensorMap mXa, mXb, mD0, mD1, mB;
  AWQ_TRY(make_map(&mXa, Xt, K, L.Tp, L.Tp, gram::BM));
  AWQ_TRY(make_map(&mXb, Xt, K, L.Tp, L.Tp, gram::BN));
  AWQ_TRY(make_map(&mD0, Dbuf[0], N, K, K, gram::BM));
  AWQ_TRY(make_map(&mD1, Dbuf[1], N, K, K, gram::BM));
  AWQ_TRY(make_map(&mB, Bm, K, K, K, gram::BN));
  gram::SearchParams sp{};
  sp.K = static_cast<int>(K);
  sp.N = static_cast<int>(N);
  sp.n_alpha = n_alpha;
  sp.gram_tiles = gram_tiles(K);
  sp.gram_kb = static_cast<int>(L.Tp / gram::BK);
  sp.row_tiles = static_cast<int>((N + gram::BM - 1) / gram::BM);
  sp.col_tiles = static_cast<int>((K + gram::BN - 1) / gram::BN);
  sp.B = Bm;
  sp.hmax = hmax;
  sp.D[0] = Dbuf[0];
  sp.D[1] = Dbuf[1];
  sp.res = ResidualArgs{W, nullptr, nullptr, absmax, nullptr, static_cast<int>(N),
                        static_cast<int>(K), symmetric, bits};
  sp.s_grid = s_grid;
  sp.inv_grid = inv_grid;
  sp.partial = partial;
  sp.pstride = kPartialStride;
  sp.sync = reinterpret_cast<unsigned int*>(ws + L.sync);
  sp.status = d->status;
  sp.limit_ns = g_wait_limit_ns.load();
  auto kern = G == 128 ? gram::search_kernel<128>
              : G == 64 ? gram::search_kernel<64> : gram::search_kernel<32>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, gram::SMEM_BYTES) !=
      cudaSuccess) {
    cudaGetLastError();
    return AWQ_ERR_CUDA;
  }
  // every CTA must be resident at once: one per SM (the shared memory allows no second)
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, gram::THREADS,
                                                    gram::SMEM_BYTES) != cudaSuccess ||
      per_sm < 1) {
    cudaGetLastError();
    return AWQ_OK;  // not launchable cooperatively here: the caller falls back
  }
  if (cudaMemsetAsync(sp.sync, 0, sizeof(unsigned int) * (2 * n_alpha + 1), st) != cudaSuccess) {
    cudaGetLastError();
    return AWQ_ERR_CUDA;
  }
  const int grid = std::min(d->sms, kPartialStride);
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(gram::THREADS);
  cfg.dynamicSmemBytes = gram::SMEM_BYTES;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  prof_start(AWQ_K_GRAM_SEARCH, st);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, mXa, mXb, mD0, mD1, mB, sp);
  if (e == cudaErrorCooperativeLaunchTooLarge || e == cudaErrorNotSupported) {
    cudaGetLastError();
    prof_cancel();
    return AWQ_OK;  // the caller falls back
  }
  const awq_status_t rl = launched(AWQ_K_GRAM_SEARCH, st);
  if (e != cudaSuccess) return AWQ_ERR_CUDA;
  AWQ_TRY(rl);
  *done = true;
  return AWQ_OK;
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
  return launch_calib_stats(static_cast<const __half*>(X_f16), T, K, ldx, mean_abs, d,
                            reinterpret_cast<cudaStream_t>(stream));
}

awq_status_t awq_scale_rows(void* A_f16, int64_t rows, int64_t cols, int64_t lda,
                           const float* row_scale, awq_stream_t stream) {
  if (!A_f16 || !row_scale || rows < 1 || cols < 1 || lda < cols) return AWQ_ERR_INVALID_ARG;
  if (rows * lda > kMaxElems) return AWQ_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(A_f16) || !aligned4(row_scale)) return AWQ_ERR_MISALIGNED;
  DeviceInfo* d = nullptr;
  AWQ_TRY(device_info(&d));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int vec8 = (cols % 8 == 0 && lda % 8 == 0) ? 1 : 0;
  const long long work = vec8 ? rows * (cols / 8) : rows * cols;
  const unsigned grid = static_cast<unsigned>(std::min<long long>(4LL * d->sms, (work + 255) / 256));
  prof_start(AWQ_K_SCALE_ROWS, st);
  block::scale_rows_kernel<<<grid, 256, 0, st>>>(static_cast<__half*>(A_f16), rows, cols, lda,
                                                 row_scale, vec8);
  return launched(AWQ_K_SCALE_ROWS, st);
}

awq_status_t awq_rmsnorm(const void* X_f16, int64_t T, int64_t D, const void* gamma_f16,
                         float eps, void* Y_f16, awq_stream_t stream) {
  if (!X_f16 || !gamma_f16 || !Y_f16 || T < 1 || D < 1 || !(eps >= 0.0f))
    return AWQ_ERR_INVALID_ARG;
  if (D % 8 != 0 || T * D > kMaxElems || T > 0x7fffffffLL) return AWQ_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(X_f16) || !aligned16(gamma_f16) || !aligned16(Y_f16)) return AWQ_ERR_MISALIGNED;
  DeviceInfo* d = nullptr;
  AWQ_TRY(device_info(&d));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  prof_start(AWQ_K_RMSNORM, st);
  block::rmsnorm_kernel<<<static_cast<unsigned>(T), 256, 0, st>>>(
      static_cast<const __half*>(X_f16), static_cast<int>(D),
      static_cast<const __half*>(gamma_f16), eps, static_cast<__half*>(Y_f16));
  return launched(AWQ_K_RMSNORM, st);
}

awq_status_t awq_silu_mul(const void* G_f16, const void* U_f16, int64_t n, void* H_f16,
                          awq_stream_t stream) {
  if (!G_f16 || !U_f16 || !H_f16 || n < 1) return AWQ_ERR_INVALID_ARG;
  if (n % 8 != 0 || n > kMaxElems) return AWQ_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(G_f16) || !aligned16(U_f16) || !aligned16(H_f16)) return AWQ_ERR_MISALIGNED;
  DeviceInfo* d = nullptr;
  AWQ_TRY(device_info(&d));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const unsigned grid = static_cast<unsigned>(std::min<long long>(4LL * d->sms, (n / 8 + 255) / 256));
  prof_start(AWQ_K_SILU_MUL, st);
  block::silu_mul_kernel<<<grid, 256, 0, st>>>(static_cast<const __half*>(G_f16),
                                               static_cast<const __half*>(U_f16), n,
                                               static_cast<__half*>(H_f16));
  return launched(AWQ_K_SILU_MUL, st);
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

awq_status_t awq_quantize_pack_clip(const void* W_f16, int64_t N, int64_t K, const float* s,
                                    const float* clip, awq_qcfg_t cfg, uint32_t* qweight,
                                    void* scales_f16, uint8_t* zeros, awq_stream_t stream) {
  AWQ_TRY(check_cfg(cfg));
  if (!W_f16 || !clip || !qweight || !scales_f16 || (!cfg.symmetric && !zeros))
    return AWQ_ERR_INVALID_ARG;
  AWQ_TRY(check_nk(N, K, cfg));
  if (!aligned16(W_f16) || !aligned16(qweight) || !aligned16(scales_f16) || !aligned4(clip) ||
      (s && !aligned16(s)) || (zeros && !aligned16(zeros)))
    return AWQ_ERR_MISALIGNED;
  DeviceInfo* d = nullptr;
  AWQ_TRY(device_info(&d));
  return launch_quantize_pack(static_cast<const __half*>(W_f16), N, K, s, cfg, qweight,
                              static_cast<__half*>(scales_f16), zeros,
                              reinterpret_cast<cudaStream_t>(stream), clip);
}

awq_status_t awq_clip_search(const void* W_f16, int64_t N, int64_t K, const void* X_f16,
                             int64_t T, const float* s, const float* ratios, int32_t n_ratio,
                             awq_qcfg_t cfg, float* energy, float* clip_out,
                             awq_stream_t stream) {
  AWQ_TRY(check_cfg(cfg));
  if (!W_f16 || !X_f16 || !ratios || !energy || !clip_out || T < 1) return AWQ_ERR_INVALID_ARG;
  if (n_ratio < 1 || n_ratio > MAX_CLIP_RATIOS) return AWQ_ERR_INVALID_ARG;
  for (int j = 0; j < n_ratio; ++j)
    if (!(ratios[j] > 0.0f && ratios[j] <= 1.0f)) return AWQ_ERR_INVALID_ARG;
  AWQ_TRY(check_nk(N, K, cfg));
  if (T * K > kMaxElems) return AWQ_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(W_f16) || !aligned16(X_f16) || (s && !aligned16(s)) || !aligned16(energy) ||
      !aligned4(clip_out))
    return AWQ_ERR_MISALIGNED;
  DeviceInfo* d = nullptr;
  AWQ_TRY(device_info(&d));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // the channel energy sum_t x^2 (the statistic kernel, squares instead of magnitudes)
  AWQ_TRY(launch_calib_stats(static_cast<const __half*>(X_f16), T, K, K, energy, d, st, true));
  ClipArgs a{};
  a.W = static_cast<const __half*>(W_f16);
  a.s = s;
  a.energy = energy;
  a.clip = clip_out;
  a.N = static_cast<int>(N);
  a.K = static_cast<int>(K);
  a.symmetric = cfg.symmetric;
  a.bits = cfg_bits(cfg);
  a.n_ratio = n_ratio;
  for (int j = 0; j < n_ratio; ++j) a.ratios[j] = ratios[j];
  const dim3 grid = run_grid<CLIP_RUN>(N, K, cfg.group_size);
  prof_start(AWQ_K_CLIP_SEARCH, st);
  if (cfg.group_size == 128)
    clip_search_kernel<128><<<grid, 256, 0, st>>>(a);
  else if (cfg.group_size == 64)
    clip_search_kernel<64><<<grid, 256, 0, st>>>(a);
  else
    clip_search_kernel<32><<<grid, 256, 0, st>>>(a);
  return launched(AWQ_K_CLIP_SEARCH, st);
}

awq_status_t awq_quant_residual(const void* W_f16, int64_t N, int64_t K, const float* s,
                                const float* inv_s, awq_qcfg_t cfg, uint32_t* absmax_bits,
                                void* D_f16, awq_stream_t stream) {
  AWQ_TRY(check_cfg(cfg));
  if (!W_f16 || !s || !inv_s || !absmax_bits || !D_f16) return AWQ_ERR_INVALID_ARG;
  AWQ_TRY(check_nk(N, K, cfg));
  if (!aligned16(W_f16) || !aligned16(s) || !aligned16(inv_s) || !aligned16(D_f16) ||
      reinterpret_cast<uintptr_t>(absmax_bits) % 4 != 0)
    return AWQ_ERR_MISALIGNED;
  DeviceInfo* d = nullptr;
  AWQ_TRY(device_info(&d));
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const __half* W = static_cast<const __half*>(W_f16);
  if (cudaMemsetAsync(absmax_bits, 0, sizeof(uint32_t), st) != cudaSuccess) {
    cudaGetLastError();
    return AWQ_ERR_CUDA;
  }
  const long long n8 = N * K / 8;
  const unsigned agrid = static_cast<unsigned>(std::min<long long>(4LL * d->sms, (n8 + 255) / 256));
  prof_start(AWQ_K_ABSMAX, st);
  absmax_kernel<<<agrid, 256, 0, st>>>(W, n8, absmax_bits);
  AWQ_TRY(launched(AWQ_K_ABSMAX, st));
  const ResidualArgs ra{W, s, inv_s, absmax_bits, static_cast<__half*>(D_f16),
                        static_cast<int>(N), static_cast<int>(K), cfg.symmetric, cfg_bits(cfg)};
  const dim3 rgrid(static_cast<unsigned>((N + 8 * QROWS - 1) / (8 * QROWS)),
                   static_cast<unsigned>((K / 8 + 31) / 32));
  prof_start(AWQ_K_RESIDUAL, st);
  if (cfg.group_size == 128)
    residual_kernel<128><<<rgrid, 256, 0, st>>>(ra);
  else if (cfg.group_size == 64)
    residual_kernel<64><<<rgrid, 256, 0, st>>>(ra);
  else
    residual_kernel<32><<<rgrid, 256, 0, st>>>(ra);
  return launched(AWQ_K_RESIDUAL, st);
}

}  // extern "C"

namespace awq {
// Every argument check of the search except those on the workspace, in the order
// awq_search_scale makes them: configuration, NULL pointers and counts, sizes, alignment, and
// the shape a forced Gram score mode needs. Shared with the static-scratch search, so both
// report the same error for the same bad argument.
awq_status_t search_check_args(const void* W_f16, int64_t N, int64_t K, const void* X_f16,
                               int64_t T, const float* mean_abs, const float* alphas,
                               int32_t n_alpha, awq_qcfg_t cfg, const float* err_out,
                               const int32_t* best_idx, const float* s_out,
                               const float* inv_s_out) {
  AWQ_TRY(check_cfg(cfg));
  if (!W_f16 || !X_f16 || !alphas || !err_out || !best_idx || T < 1) return AWQ_ERR_INVALID_ARG;
  if (n_alpha < 1 || n_alpha > 64) return AWQ_ERR_INVALID_ARG;
  AWQ_TRY(check_nk(N, K, cfg));
  if (T * K > kMaxElems) return AWQ_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(W_f16) || !aligned16(X_f16) || (mean_abs && !aligned16(mean_abs)) ||
      !aligned4(err_out) || !aligned4(best_idx) || (s_out && !aligned16(s_out)) ||
      (inv_s_out && !aligned16(inv_s_out)))
    return AWQ_ERR_MISALIGNED;
  const int score_mode = g_score_mode.load();
  if ((score_mode == AWQ_SCORE_GRAM || score_mode == AWQ_SCORE_GRAM_LAUNCHES) &&
      !gram_shape_ok(K, T))
    return AWQ_ERR_UNSUPPORTED_SHAPE;
  return AWQ_OK;
}

// Smallest workspace awq_search_scale accepts (one residual buffer: candidates in order).
size_t search_workspace_min_bytes(int64_t N, int64_t K, int64_t T, int32_t n_alpha,
                                  awq_qcfg_t cfg) {
  if (check_cfg(cfg) != AWQ_OK || check_nk(N, K, cfg) != AWQ_OK || T < 1 || n_alpha < 1 ||
      n_alpha > 64)
    return 0;
  return search_layout(N, K, T, n_alpha).min_total;
}
}  // namespace awq

extern "C" {

size_t awq_search_workspace_bytes(int64_t N, int64_t K, int64_t T, int32_t n_alpha,
                                  awq_qcfg_t cfg) {
  if (check_cfg(cfg) != AWQ_OK || check_nk(N, K, cfg) != AWQ_OK || T < 1 || n_alpha < 1 ||
      n_alpha > 64)
    return 0;
  const SearchLayout L = search_layout(N, K, T, n_alpha);
  int sms = 148;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    sms = 148;
  }
  Sched sc;
  if (!pick_schedule(N, K, T, n_alpha, SIZE_MAX, sms, L, &sc)) return 0;
  return sc == Sched::GRAM ? L.gram_total : L.total;
}

awq_status_t awq_set_score_mode(awq_score_mode_t mode) {
  if (mode != AWQ_SCORE_AUTO && mode != AWQ_SCORE_DIRECT && mode != AWQ_SCORE_GRAM &&
      mode != AWQ_SCORE_GRAM_LAUNCHES)
    return AWQ_ERR_INVALID_ARG;
  g_score_mode.store(mode);
  return AWQ_OK;
}

awq_status_t awq_search_scale(const void* W_f16, int64_t N, int64_t K, const void* X_f16,
                              int64_t T, const float* mean_abs, const float* alphas,
                              int32_t n_alpha, awq_qcfg_t cfg, void* workspace,
                              size_t ws_bytes, float* err_out, int32_t* best_idx,
                              float* s_out, float* inv_s_out, awq_stream_t stream) {
  AWQ_TRY(search_check_args(W_f16, N, K, X_f16, T, mean_abs, alphas, n_alpha, cfg, err_out,
                            best_idx, s_out, inv_s_out));
  if (!aligned16(workspace)) return AWQ_ERR_MISALIGNED;
  const SearchLayout L = search_layout(N, K, T, n_alpha);
  const int score_mode = g_score_mode.load();
  if (!workspace || ws_bytes < L.min_total) return AWQ_ERR_WORKSPACE;
  DeviceInfo* d = nullptr;
  AWQ_TRY(device_info(&d));
  Sched sched;
  if (!pick_schedule(N, K, T, n_alpha, ws_bytes, d->sms, L, &sched)) return AWQ_ERR_WORKSPACE;
  const bool overlap = sched != Sched::SERIAL;
  const bool use_gram = sched == Sched::GRAM;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* m = reinterpret_cast<float*>(ws + L.m);
  float* s_grid = reinterpret_cast<float*>(ws + L.s_grid);
  float* inv_grid = reinterpret_cast<float*>(ws + L.inv_grid);
  unsigned int* absmax = reinterpret_cast<unsigned int*>(ws + L.absmax);
  double* partial = reinterpret_cast<double*>(ws + L.partial);
  __half* Dbuf[2] = {reinterpret_cast<__half*>(ws + L.D),
                     reinterpret_cast<__half*>(ws + (overlap ? L.D2 : L.D))};
  const __half* W = static_cast<const __half*>(W_f16);
  const __half* X = static_cast<const __half*>(X_f16);

  unsigned int* hmax = reinterpret_cast<unsigned int*>(ws + L.hmax);
  float* colsq = reinterpret_cast<float*>(ws + L.colsq);
  __half* Xt = reinterpret_cast<__half*>(ws + L.xt);
  __half* Bm = reinterpret_cast<__half*>(ws + L.bmat);

  // direct: A = X tiles, B = D tiles; Gram: A = D tiles, B = tiles of the scaled triangle of H
  CUtensorMap mapX, mapD[2], mapXa, mapXb, mapBm;
  if (use_gram) {
    AWQ_TRY(make_map(&mapXa, Xt, K, L.Tp, L.Tp, gram::BM));
    AWQ_TRY(make_map(&mapXb, Xt, K, L.Tp, L.Tp, gram::BN));
    AWQ_TRY(make_map(&mapBm, Bm, K, K, K, gram::BN));
    AWQ_TRY(make_map(&mapD[0], Dbuf[0], N, K, K, gram::BM));
    AWQ_TRY(make_map(&mapD[1], Dbuf[1], N, K, K, gram::BM));
  } else {
    AWQ_TRY(make_map(&mapX, X, T, K, K, score::BM));
    AWQ_TRY(make_map(&mapD[0], Dbuf[0], N, K, K, score::BN));
    AWQ_TRY(make_map(&mapD[1], Dbuf[1], N, K, K, score::BN));
  }

  // 1. statistic
  const float* mp = mean_abs;
  if (!mp) {
    AWQ_TRY(launch_calib_stats(X, T, K, K, m, d, st));
    mp = m;
  }
  // GRAM: the scale grid and max|W| (steps 2-3) run on the library's second stream while X^T
  // and its column sums are formed on the caller's (step 4); they join before the search
  cudaStream_t ps = st;
  if (use_gram) {
    if (cudaEventRecord(d->fork, st) != cudaSuccess || cudaStreamWaitEvent(d->side, d->fork, 0) != cudaSuccess) {
      cudaGetLastError();
      return AWQ_ERR_CUDA;
    }
    ps = d->side;
  }
  // 2. scale grid
  GridArgs ga{};
  ga.m = mp;
  ga.s = s_grid;
  ga.inv_s = inv_grid;
  ga.K = static_cast<int>(K);
  ga.n_alpha = n_alpha;
  for (int i = 0; i < n_alpha; ++i) ga.alphas[i] = alphas[i];
  prof_start(AWQ_K_SCALE_GRID, ps);
  scale_grid_kernel<<<dim3(static_cast<unsigned>((K + 127) / 128),
                           static_cast<unsigned>((n_alpha + GRID_ALPHAS - 1) / GRID_ALPHAS)),
                      128, 0, ps>>>(ga);
  AWQ_TRY(launched(AWQ_K_SCALE_GRID, ps));
  // 3. max |W| for the residual's power-of-two scale
  if (cudaMemsetAsync(absmax, 0, sizeof(unsigned int), ps) != cudaSuccess) {
    cudaGetLastError();
    return AWQ_ERR_CUDA;
  }
  const long long n8 = N * K / 8;
  const unsigned agrid = static_cast<unsigned>(std::min<long long>(4LL * d->sms, (n8 + 255) / 256));
  prof_start(AWQ_K_ABSMAX, ps);
  absmax_kernel<<<agrid, 256, 0, ps>>>(W, n8, absmax);
  AWQ_TRY(launched(AWQ_K_ABSMAX, ps));
  // 4. Gram schedule: X^T and its column sums of squares, max_k H[k][k], then the scaled lower
  //    triangle of H = X^T X (once per layer)
  auto smem_attr = [](const void* f, int bytes) -> awq_status_t {
    if (cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) == cudaSuccess)
      return AWQ_OK;
    cudaGetLastError();
    return AWQ_ERR_CUDA;
  };
  gram::Params gp{};
  int ggrid = 0;
  bool persistent = false;
  using TriKern = void (*)(CUtensorMap, CUtensorMap, gram::Params);
  const TriKern tri_gram = cfg.group_size == 128 ? gram::tri_kernel<gram::GRAM, 128>
                           : cfg.group_size == 64 ? gram::tri_kernel<gram::GRAM, 64>
                                                  : gram::tri_kernel<gram::GRAM, 32>;
  const TriKern tri_score = cfg.group_size == 128 ? gram::tri_kernel<gram::SCORE, 128>
                            : cfg.group_size == 64 ? gram::tri_kernel<gram::SCORE, 64>
                                                   : gram::tri_kernel<gram::SCORE, 32>;
  // the residual of candidate i into buffer i % 2
  auto res_args = [&](int i) {
    return ResidualArgs{W, s_grid + static_cast<size_t>(i) * K, inv_grid + static_cast<size_t>(i) * K,
                        absmax, Dbuf[i & 1], static_cast<int>(N), static_cast<int>(K), cfg.symmetric,
                        cfg_bits(cfg)};
  };
  if (use_gram) {
    if (cudaMemsetAsync(hmax, 0, sizeof(unsigned int), st) != cudaSuccess) {
      cudaGetLastError();
      return AWQ_ERR_CUDA;
    }
    const int nblk = static_cast<int>(L.Tp / gram::TOK_BLOCK);
    prof_start(AWQ_K_GRAM_PREP, st);
    gram::transpose_kernel<<<dim3(static_cast<unsigned>(K / 64), static_cast<unsigned>(nblk)), 256,
                             0, st>>>(X, static_cast<int>(T), static_cast<int>(K),
                                      static_cast<int>(L.Tp), Xt, colsq);
    AWQ_TRY(launched(AWQ_K_GRAM_PREP, st));
    prof_start(AWQ_K_GRAM_PREP, st);
    gram::colsq_max_kernel<<<static_cast<unsigned>((K + 31) / 32), 256, 0, st>>>(
        colsq, nblk, static_cast<int>(K), hmax);
    AWQ_TRY(launched(AWQ_K_GRAM_PREP, st));
    if (cudaEventRecord(d->score_done[0], ps) != cudaSuccess ||
        cudaStreamWaitEvent(st, d->score_done[0], 0) != cudaSuccess) {  // join
      cudaGetLastError();
      return AWQ_ERR_CUDA;
    }
    if (score_mode != AWQ_SCORE_GRAM_LAUNCHES) {
      AWQ_TRY(launch_search_persistent(cfg.group_size, d, L, ws, Xt, Bm, hmax, Dbuf, W, absmax,
                                       s_grid, inv_grid, partial, N, K, n_alpha, cfg.symmetric,
                                       cfg_bits(cfg), &persistent, st));
    }
  }
  if (use_gram && !persistent) {
    AWQ_TRY(smem_attr(reinterpret_cast<const void*>(tri_gram), gram::SMEM_BYTES));
    AWQ_TRY(smem_attr(reinterpret_cast<const void*>(tri_score), gram::SMEM_BYTES));
    gp.K = static_cast<int>(K);
    gp.N = static_cast<int>(N);
    gp.num_kb = static_cast<int>(L.Tp / gram::BK);  // TOK_BLOCK == BK
    gp.num_tiles = gram_tiles(K);
    gp.B = Bm;
    gp.hmax = hmax;
    gp.status = d->status;
    gp.limit_ns = g_wait_limit_ns.load();
    gp.res = res_args(0);  // candidate 0's residual is built alongside H
    gp.res_on = 1;
    prof_start(AWQ_K_GRAM, st);
    tri_gram<<<std::min(gp.num_tiles, d->sms), gram::THREADS, gram::SMEM_BYTES, st>>>(mapXa, mapXb,
                                                                                       gp);
    AWQ_TRY(launched(AWQ_K_GRAM, st));
    gp.row_tiles = static_cast<int>((N + gram::BM - 1) / gram::BM);
    gp.col_tiles = static_cast<int>((K + gram::BN - 1) / gram::BN);
    gp.num_tiles = gp.row_tiles * gp.col_tiles;
    gp.num_kb = 0;
    gp.B = nullptr;
    ggrid = std::min(gp.num_tiles, std::min(d->sms, kPartialStride));
  } else if (!use_gram) {
    AWQ_TRY(smem_attr(reinterpret_cast<const void*>(score::score_kernel), score::SMEM_BYTES));
  }
  if (persistent) ggrid = d->sms;
  // 5. per alpha: residual D = W - Q(W diag s) diag(s)^-1, then its error score
  score::Params sp{};
  sp.tiles_n = static_cast<int>((N + score::BN - 1) / score::BN);
  const int tiles_m = static_cast<int>((T + score::BM - 1) / score::BM);
  sp.num_tiles = tiles_m * sp.tiles_n;
  sp.num_kb = static_cast<int>((K + score::BK - 1) / score::BK);
  sp.status = d->status;
  sp.limit_ns = g_wait_limit_ns.load();
  const int sgrid = std::min(sp.num_tiles, std::min(d->sms, kPartialStride));
  const dim3 rgrid(static_cast<unsigned>((N + 8 * QROWS - 1) / (8 * QROWS)),
                   static_cast<unsigned>((K / 8 + 31) / 32));
  // Residual i goes to buffer i % 2. GRAM: the scoring launch of candidate i builds residual
  // i + 1 in its own extra warps. DIRECT with two buffers: the residual of candidate i + 1 runs
  // on the side stream while candidate i is scored (the scoring GEMM is tensor-bound and leaves
  // room on every SM for the memory-bound residual blocks); events order the two streams (the
  // side stream forks from and rejoins the caller's stream, so the sequence can be captured in
  // a graph). With one buffer everything runs in order on the caller's stream.
  auto residual = [&](int i, cudaStream_t rs) -> awq_status_t {
    const ResidualArgs ra = res_args(i);
    prof_start(AWQ_K_RESIDUAL, rs);
    if (cfg.group_size == 128)
      residual_kernel<128><<<rgrid, 256, 0, rs>>>(ra);
    else if (cfg.group_size == 64)
      residual_kernel<64><<<rgrid, 256, 0, rs>>>(ra);
    else
      residual_kernel<32><<<rgrid, 256, 0, rs>>>(ra);
    return launched(AWQ_K_RESIDUAL, rs);
  };
  auto ev = [](cudaError_t e) -> awq_status_t {
    if (e == cudaSuccess) return AWQ_OK;
    cudaGetLastError();
    return AWQ_ERR_CUDA;
  };
  if (persistent) {
    // the whole search ran in the persistent launch above
  } else if (use_gram) {
    // every launch on the caller's stream: each scoring launch also builds the next residual
    for (int i = 0; i < n_alpha; ++i) {
      gp.D = Dbuf[i & 1];
      gp.partial = partial + static_cast<size_t>(i) * kPartialStride;
      gp.res_on = i + 1 < n_alpha ? 1 : 0;
      if (gp.res_on) gp.res = res_args(i + 1);
      prof_start(AWQ_K_SCORE_GRAM, st);
      tri_score<<<ggrid, gram::THREADS, gram::SMEM_BYTES, st>>>(mapD[i & 1], mapBm, gp);
      AWQ_TRY(launched(AWQ_K_SCORE_GRAM, st));
    }
  } else {
    cudaStream_t rs = overlap ? d->side : st;
    if (overlap) {
      AWQ_TRY(ev(cudaEventRecord(d->fork, st)));
      AWQ_TRY(ev(cudaStreamWaitEvent(rs, d->fork, 0)));
    }
    AWQ_TRY(residual(0, rs));
    if (overlap) AWQ_TRY(ev(cudaEventRecord(d->res_done[0], rs)));
    for (int i = 0; i < n_alpha; ++i) {
      if (overlap) AWQ_TRY(ev(cudaStreamWaitEvent(st, d->res_done[i & 1], 0)));
      sp.partial = partial + static_cast<size_t>(i) * kPartialStride;
      prof_start(AWQ_K_SCORE, st);
      score::score_kernel<<<sgrid, score::THREADS, score::SMEM_BYTES, st>>>(mapX, mapD[i & 1], sp);
      AWQ_TRY(launched(AWQ_K_SCORE, st));
      if (i + 1 < n_alpha) {
        if (overlap) {
          AWQ_TRY(ev(cudaEventRecord(d->score_done[i & 1], st)));
          // buffer (i + 1) % 2 was last read by the scoring of candidate i - 1
          if (i >= 1) AWQ_TRY(ev(cudaStreamWaitEvent(rs, d->score_done[(i - 1) & 1], 0)));
        }
        AWQ_TRY(residual(i + 1, rs));
        if (overlap) AWQ_TRY(ev(cudaEventRecord(d->res_done[(i + 1) & 1], rs)));
      }
    }
  }
  // 6. errors, argmin, winning scales
  prof_start(AWQ_K_FINALIZE, st);
  finalize_kernel<<<1, 1024, 0, st>>>(partial, use_gram ? ggrid : sgrid, n_alpha, absmax,
                                     use_gram ? hmax : nullptr,
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
  if (M <= gemv::MAX_M) {
    gemv::Args a{};
    a.X = static_cast<const __half*>(X_f16);
    a.Q = qweight;
    a.scales = static_cast<const __half*>(scales_f16);
    a.zeros = z;
    a.inv_s = inv_s;
    a.Y = static_cast<__half*>(Y_f16);
    a.M = static_cast<int>(M);
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    a.status = d->status;
    a.limit_ns = g_wait_limit_ns.load();
    if (gemv_shape(a, G, d->sms) == AWQ_OK)
      return M == 1   ? launch_gemv_m<1>(a, G, st)
             : M == 2 ? launch_gemv_m<2>(a, G, st)
             : M == 3 ? launch_gemv_m<3>(a, G, st)
                      : launch_gemv_m<4>(a, G, st);
  }
  w4tc::Args a{};
  a.Q = qweight;
  a.scales = static_cast<const __half*>(scales_f16);
  a.zeros = z;
  a.inv_s = inv_s;
  a.Y = static_cast<__half*>(Y_f16);
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(N);
  a.K = static_cast<int>(K);
  a.splits = 1;
  a.status = d->status;
  a.limit_ns = g_wait_limit_ns.load();
  const __half* X = static_cast<const __half*>(X_f16);
  // the grouped kernel gives every group of 64 or more channels its own accumulator; G = 32
  // takes the dequant kernel at every M above the GEMV's
  if (M <= w4tc::grouped::BN && G >= 64) return launch_w4_grouped(X, a, G, d->sms, st);
  return launch_w4_dequant(X, a, G, d->sms, st);
}

}  // extern "C"
