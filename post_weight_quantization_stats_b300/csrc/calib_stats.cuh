// Per-input-channel calibration statistic m_j = (1/T) sum_t |X[t, j]|.
//
// "AWQ Math", "Saliency is an activation property, not a weight property": input channels are
// ranked by the average |x_j| over the calibration set; the scale search raises this statistic
// to the power alpha ("Searching the scale").
//
// One read of X, HBM-bound. A cluster of 8 CTAs owns 64 columns; each CTA sums one eighth of
// the rows. Its rows stream through shared memory as TMA boxes of 128 rows x 64 columns (16 KB,
// a ring of 2), so every CTA keeps 32 KB of reads in flight without spending registers; the 256
// threads add a box with 16-byte reads (8 lanes x 8 fp16 per row, four rows per warp
// instruction, no bank conflicts), fold their 32 row slots in shared memory, and CTA rank 0
// adds the 8 CTA sums through distributed shared memory. Every sum runs in a fixed order, so
// the result is deterministic, and no global scratch is needed.
#pragma once

#include <cooperative_groups.h>

#include "awq_device.cuh"

namespace awq {
namespace stats {

constexpr int COLS = 64;       // columns per cluster (one TMA box wide)
constexpr int CLUSTER = 8;     // CTAs per cluster (row split)
constexpr int THREADS = 256;
constexpr int LANES_PER_ROW = COLS / 8;
constexpr int SLOTS = THREADS / LANES_PER_ROW;  // row slots per CTA read step
constexpr int BOX_ROWS = 128;  // rows per TMA box
constexpr int STAGES = 2;
constexpr int BOX_BYTES = BOX_ROWS * COLS * 2;

// SQ = false: |x| (the statistic); SQ = true: x^2 (the channel energy of the clipping search).
template <bool SQ>
__device__ __forceinline__ void add8(const uint4& raw, float (&acc)[8]) {
  const __half2* h2 = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (SQ) {
      const float2 f = __half22float2(h2[i]);
      acc[2 * i] = fmaf(f.x, f.x, acc[2 * i]);
      acc[2 * i + 1] = fmaf(f.y, f.y, acc[2 * i + 1]);
    } else {
      const float2 f = __half22float2(__habs2(h2[i]));
      acc[2 * i] += f.x;
      acc[2 * i + 1] += f.y;
    }
  }
}

// SQ = false: m_j = (1/T) sum_t |X[t, j]|. SQ = true: m_j = sum_t X[t, j]^2 (no division).
template <bool SQ>
__global__ void __cluster_dims__(1, CLUSTER, 1) __launch_bounds__(THREADS)
    calib_stats_kernel(const __grid_constant__ CUtensorMap tmX, int T, int K, float* __restrict__ m,
                       int* status, unsigned long long limit_ns) {
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  __shared__ __align__(128) uint8_t ring[STAGES][BOX_BYTES];
  __shared__ __align__(16) float part[SLOTS][COLS];
  __shared__ float cta_sum[COLS];
  __shared__ __align__(8) uint64_t full[STAGES];
  __shared__ int abort_flag;

  const int tid = threadIdx.x;
  const int slot = tid / LANES_PER_ROW;      // row slot 0..SLOTS-1
  const int cl = (tid % LANES_PER_ROW) * 8;  // column offset inside the block
  const int col0 = blockIdx.x * COLS;
  const int rank = static_cast<int>(cluster.block_rank());
  const int t0 = static_cast<int>(static_cast<long long>(T) * rank / CLUSTER);
  const int t1 = static_cast<int>(static_cast<long long>(T) * (rank + 1) / CLUSTER);
  const int nbox = (t1 - t0 + BOX_ROWS - 1) / BOX_ROWS;

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) mbar_init(&full[s], 1);
    abort_flag = 0;
    fence_mbar_init();
    prefetch_tensormap(&tmX);
    for (int j = 0; j < STAGES && j < nbox; ++j) {
      mbar_arrive_expect_tx(&full[j], BOX_BYTES);
      tma_load_2d(ring[j], &tmX, &full[j], col0, t0 + j * BOX_ROWS);
    }
  }
  __syncthreads();
  const WaitCtx wc{limit_ns, &abort_flag, status};

  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  bool ok = true;
  for (int j = 0; j < nbox; ++j) {
    const int s = j % STAGES;
    if (ok) ok = wait_bounded(&full[s], (j / STAGES) & 1u, wc);
    // rows of the box past the CTA's range belong to the next CTA (or lie past T): skip them;
    // columns past K read as zero
    const int rows = min(BOX_ROWS, t1 - t0 - j * BOX_ROWS);
    if (ok) {
#pragma unroll
      for (int r = slot; r < BOX_ROWS; r += SLOTS)
        if (r < rows) add8<SQ>(*reinterpret_cast<const uint4*>(ring[s] + r * COLS * 2 + cl * 2), acc);
    }
    __syncthreads();   // every thread is done with stage s
    if (tid == 0 && j + STAGES < nbox && !abort_flag) {
      mbar_arrive_expect_tx(&full[s], BOX_BYTES);
      tma_load_2d(ring[s], &tmX, &full[s], col0, t0 + (j + STAGES) * BOX_ROWS);
    }
  }
  if (tid == 0) {   // a CTA that gave up lets its copies in flight land before exiting
    for (int j = max(0, nbox - STAGES); j < nbox; ++j)
      wait_drain(&full[j % STAGES], (j / STAGES) & 1u, limit_ns);
  }
  float4* dst = reinterpret_cast<float4*>(&part[slot][cl]);
  dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
  dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  __syncthreads();
  if (tid < COLS) {
    float sum = 0.f;
#pragma unroll
    for (int r = 0; r < SLOTS; ++r) sum += part[r][tid];
    cta_sum[tid] = sum;
  }
  cluster.sync();
  if (rank == 0 && tid < COLS && !abort_flag) {
    float sum = 0.f;
#pragma unroll
    for (int r = 0; r < CLUSTER; ++r) sum += cluster.map_shared_rank(cta_sum, r)[tid];
    const int c = col0 + tid;
    if (c < K) m[c] = SQ ? sum : __fdiv_rn(sum, static_cast<float>(T));
  }
  cluster.sync();
}

}  // namespace stats
}  // namespace awq
