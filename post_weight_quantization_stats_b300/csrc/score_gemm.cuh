// Output-error scoring of one alpha candidate on the tcgen05 tensor cores.
//
// "AWQ Math", "Searching the scale": for each alpha the layer is quantised, the calibration
// activations are run through it, and the mean-squared error against the original output is
// measured. Since W x - w_hat x = (W - w_hat) x, the error of one candidate is
//     E = 1/(T N) * sum_{t,n} ( sum_k X[t,k] D[n,k] )^2,   D = W - w_hat,
// a dense T x N x K contraction with a sum-of-squares epilogue. D arrives as fp16 scaled by
// 2^p (residual_kernel); the host removes 2^(2p) when it finalises E.
//
// Kernel shape (one CTA per SM, persistent over 128 x 256 output tiles):
//   warp 0     TMA producer: X tile [128 tok x 64 k] and D tile [256 out x 64 k] per stage,
//              128-byte swizzle, 4-stage ring of 48 KB stages.
//   warp 1     allocates 512 TMEM columns (two 128 x 256 fp32 accumulators) and issues
//              tcgen05.mma (M=128, N=256, K=16) from one thread; tcgen05.commit frees smem
//              stages and hands finished accumulators to the epilogue.
//   warps 2-5  epilogue: tcgen05.ld each accumulator lane (= token), square and sum, release
//              the accumulator; one fp64 partial per CTA at the end.
// Out-of-range tokens/outputs are zero-filled by TMA and add nothing.
#pragma once

#include "awq_device.cuh"

namespace awq {
namespace score {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int THREADS = 192;
constexpr uint32_t TMEM_COLS = 512;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;

struct Params {
  int tiles_n, num_tiles, num_kb;
  double* partial;  // [gridDim.x] sum of squares of this CTA's tiles
  int* status;
  unsigned long long limit_ns;
};

__global__ void __launch_bounds__(THREADS, 1)
    score_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmD,
                 Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + STAGES * B_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;   // [2]
  uint64_t* tempty = tfull + 2;       // [2]
  uint64_t* drain = tempty + 2;       // [1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  double* red = reinterpret_cast<double*>(tmem_slot + 4);  // [4]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tensormap(&tmX);
    prefetch_tensormap(&tmD);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const WaitCtx wc{p.limit_ns, abort_flag, p.status};

  if (warp == 0) {
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
        const int tm = tile / p.tiles_n, tn = tile - (tile / p.tiles_n) * p.tiles_n;
        for (int kb = 0; kb < p.num_kb; ++kb, ++it) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
          if (!wait_bounded(&empty[s], ph ^ 1u, wc)) { ok = false; break; }
          mbar_arrive_expect_tx(&full[s], STAGE_BYTES);
          tma_load_2d(sA + s * A_BYTES, &tmX, &full[s], kb * BK, tm * BM);
          tma_load_2d(sB + s * B_BYTES, &tmD, &full[s], kb * BK, tn * BN);
        }
      }
      {  // let the copies issued last land before the CTA exits (at once unless it gave up)
        const uint32_t first = it > STAGES ? it - STAGES : 0u;
        for (uint32_t j = first; j < it; ++j)
          wait_drain(&full[j % STAGES], (j / STAGES) & 1u, p.limit_ns);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16_f32(BM, BN);
      uint32_t it = 0, local = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x, ++local) {
        const uint32_t acc = local & 1u, use = local >> 1;
        if (!wait_bounded(&tempty[acc], (use & 1u) ^ 1u, wc)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < p.num_kb; ++kb, ++it) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
          if (!wait_bounded(&full[s], ph, wc)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + s * A_BYTES), b0 = smem_u32(sB + s * B_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            mma_f16(d_tmem, sw128_kmajor_desc(a0 + k * 32), sw128_kmajor_desc(b0 + k * 32), idesc,
                    (kb | k) != 0);
          mma_commit(&empty[s]);
        }
        if (!ok) break;
        mma_commit(&tfull[acc]);
      }
      mma_commit(drain);  // every MMA issued above has finished once this arrives
      wait_drain(drain, 0, p.limit_ns);
    }
  } else {
    const uint32_t q = static_cast<uint32_t>(warp & 3);  // TMEM lane quarter of this warp
    double total = 0.0;
    uint32_t local = 0;
    for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++local) {
      const uint32_t acc = local & 1u, use = local >> 1;
      const bool got = wait_bounded(&tfull[acc], use & 1u, wc);
      if (!__all_sync(0xffffffffu, got)) break;  // warp-uniform: tcgen05.ld is .sync.aligned
      tc_fence_after();
      float sum = 0.f;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        tmem_ld_x32(tmem_base + ((q * 32u) << 16) + acc * BN + c * 32, r);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float v = __uint_as_float(r[j]);
          sum = fmaf(v, v, sum);
        }
      }
      total += static_cast<double>(sum);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) total += __shfl_xor_sync(0xffffffffu, total, o);
    if (lane == 0) red[warp - 2] = total;
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) p.partial[blockIdx.x] = ((red[0] + red[1]) + red[2]) + red[3];
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

}  // namespace score
}  // namespace awq
