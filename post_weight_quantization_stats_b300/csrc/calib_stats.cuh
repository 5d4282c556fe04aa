// Per-input-channel calibration statistic m_j = (1/T) sum_t |X[t, j]|.
//
// "AWQ Math", "Saliency is an activation property, not a weight property": input channels are
// ranked by the average |x_j| over the calibration set; the scale search raises this statistic
// to the power alpha ("Searching the scale").
//
// One read of X, HBM-bound. A cluster of 8 CTAs owns 128 columns; each CTA sums one eighth of
// the rows with 16-byte loads (16 lanes x 8 fp16 per row, two rows per warp instruction, 8
// loads in flight per thread), folds its 16 row slots in shared memory, and CTA rank 0 adds
// the 8 CTA sums through distributed shared memory. Every sum runs in a fixed order, so the
// result is deterministic, and no global scratch is needed.
#pragma once

#include <cooperative_groups.h>

#include "awq_device.cuh"

namespace awq {
namespace stats {

constexpr int COLS = 128;      // columns per cluster
constexpr int CLUSTER = 8;     // CTAs per cluster (row split)
constexpr int THREADS = 256;
constexpr int SLOTS = THREADS / 16;  // row slots per CTA load step
constexpr int UNROLL = 8;

__device__ __forceinline__ void add_abs8(const uint4& raw, float (&acc)[8]) {
  const __half2* h2 = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __half22float2(__habs2(h2[i]));
    acc[2 * i] += f.x;
    acc[2 * i + 1] += f.y;
  }
}

__global__ void __cluster_dims__(1, CLUSTER, 1) __launch_bounds__(THREADS)
    calib_stats_kernel(const __half* __restrict__ X, int T, int K, long long ldx,
                       float* __restrict__ m) {
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  __shared__ __align__(16) float part[SLOTS][COLS];
  __shared__ float cta_sum[COLS];

  const int tid = threadIdx.x;
  const int slot = tid >> 4;              // row slot 0..15
  const int cl = (tid & 15) * 8;          // column offset inside the block
  const int col = blockIdx.x * COLS + cl;
  const int rank = static_cast<int>(cluster.block_rank());
  const int t0 = static_cast<int>(static_cast<long long>(T) * rank / CLUSTER);
  const int t1 = static_cast<int>(static_cast<long long>(T) * (rank + 1) / CLUSTER);

  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (col < K) {
    const __half* base = X + col;
    int t = t0 + slot;
    for (; t + (UNROLL - 1) * SLOTS < t1; t += UNROLL * SLOTS) {
      uint4 v[UNROLL];
#pragma unroll
      for (int u = 0; u < UNROLL; ++u)
        v[u] = __ldg(reinterpret_cast<const uint4*>(base + static_cast<long long>(t + u * SLOTS) * ldx));
#pragma unroll
      for (int u = 0; u < UNROLL; ++u) add_abs8(v[u], acc);
    }
    for (; t < t1; t += SLOTS)
      add_abs8(__ldg(reinterpret_cast<const uint4*>(base + static_cast<long long>(t) * ldx)), acc);
  }
  float4* dst = reinterpret_cast<float4*>(&part[slot][cl]);
  dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
  dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  __syncthreads();
  if (tid < COLS) {
    float s = 0.f;
#pragma unroll
    for (int r = 0; r < SLOTS; ++r) s += part[r][tid];
    cta_sum[tid] = s;
  }
  cluster.sync();
  if (rank == 0 && tid < COLS) {
    float s = 0.f;
#pragma unroll
    for (int r = 0; r < CLUSTER; ++r) s += cluster.map_shared_rank(cta_sum, r)[tid];
    const int c = blockIdx.x * COLS + tid;
    if (c < K) m[c] = __fdiv_rn(s, static_cast<float>(T));
  }
  cluster.sync();
}

}  // namespace stats
}  // namespace awq
