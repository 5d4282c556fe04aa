// W4A16 decode GEMV (M <= 2 tokens) on the CUDA cores.
//
// "AWQ > Benefits and Practical Considerations": decode is bound by reading the weights from
// HBM; the kernel unpacks the 4-bit integers, applies the group scale and zero point and,
// optionally, the per-channel inverse scale, fused with the product so no fp16 weight matrix is
// ever written.
//
// One CTA per SM, each owning a contiguous range of output rows. The packed codes of a row
// range are one contiguous byte range of qweight, so a single producer thread streams whole
// rows into a ring of shared-memory stages with 1-D bulk copies (cp.async.bulk, L2
// evict-first): every CTA keeps 100+ KB of weight reads in flight without spending registers.
//
// The consumers are P x RG warps: part p of K (IPL items of 32 channels per lane, 1024 * IPL
// channels per warp) times row group rg. A lane's activations never change: the CTA stages
// x~ = x * inv_s once in shared memory with coalesced loads, and each lane copies its K slice
// into registers; afterwards the only shared-memory traffic per code is the bulk copy's write
// and one 16-byte read per item. Per
// item and row:
//   * codes become exact (q - z) half2 pairs by the 0x6400 fp16 exponent trick (q + 1024 sits
//     in the mantissa of a half in [1024, 2048));
//   * HFMA2 multiplies them into x~ / 64 (a power of two: exact unless subnormal) in two
//     accumulators of 8 products per half, so partial sums stay below 120 |x~| / 64 and
//     cannot overflow for any |x~| below 34,000;
//   * the item sum is scaled by 64 * step and accumulated in fp32.
// Row partials are reduced with shuffles and written to shared memory per (row, part); the
// parts are added in a fixed order at the end, so the result is deterministic.
//
// Launched with programmatic dependent launch: the kernel lets the next W4A16 launch of the
// stream start right after its own set-up, and it streams its weights and stages its group
// parameters before waiting (griddepcontrol.wait) for the previous kernel, so back-to-back
// decode layers overlap one layer's weight prefetch with the previous layer's tail. The ring
// has only as many stages as the CTA's rows need, which keeps the next kernel's CTAs resident.
#pragma once

#include "awq_device.cuh"

namespace awq {
namespace gemv {

constexpr int CWARPS = 15;                // consumer warps (16 warps in all: 128 registers each)
constexpr int CTHREADS = CWARPS * 32;
constexpr int THREADS = CTHREADS + 32;    // + one producer warp
constexpr int ITEM_CH = 32;               // channels of one lane item (4 packed words)
constexpr int MAX_M = 2;
constexpr int MAX_STAGES = 8;
constexpr int SMEM_BUDGET = 220 * 1024;
constexpr float X_PRESCALE = 1.0f / 64.0f;

// Items per lane for M tokens: the registers holding x~ stay at 64 per thread.
__host__ __device__ constexpr int items_per_lane(int M) { return M == 1 ? 4 : 2; }

struct Args {
  const __half* X;        // [M, K]
  const uint32_t* Q;      // [N, K/8]
  const __half* scales;   // [K/G, N]
  const uint8_t* zeros;   // [K/G, N] (asymmetric only)
  const float* inv_s;     // [K] or nullptr
  __half* Y;              // [M, N]
  int M, N, K;
  int parts;              // K parts P = ceil((K / 32) / (32 * IPL))
  int row_groups;         // RG = CWARPS / P (warps beyond P * RG idle)
  int rows_stage;         // rows per stage RS (a multiple of RG)
  int stage_bytes;        // RS * K / 2
  int nstages;            // ring depth, 2..MAX_STAGES
  int rows_max;           // max output rows of one CTA
  int pstride;            // words per CTA row of staged group parameters: K / G + 1
  int* status;
  unsigned long long limit_ns;
};

// Shared-memory footprint for the given launch shape (the host sizes the launch with it).
__host__ __device__ inline int ysum_floats(const Args& a) {
  return (a.rows_max * a.parts * a.M + 3) & ~3;
}
__host__ __device__ inline int param_words(const Args& a) { return (a.rows_max * a.pstride + 3) & ~3; }
__host__ __device__ inline size_t xs_bytes(const Args& a) {
  return static_cast<size_t>(a.M) * static_cast<size_t>(a.K) * 2;
}
__host__ __device__ inline size_t smem_bytes(const Args& a) {
  return static_cast<size_t>(a.nstages) * a.stage_bytes + xs_bytes(a) +
         static_cast<size_t>(param_words(a)) * 4 + static_cast<size_t>(ysum_floats(a)) * 4 +
         2 * MAX_STAGES * 8 + 16;
}

// 8 codes of one word -> 4 exact half2 (q - z) pairs in the order (0,4), (1,5), (2,6), (3,7).
// zsub = 1024 + z (subtracted from the low-nibble lanes), zadd = -(64 + z) (added to the
// x/16 high-nibble lanes).
__device__ __forceinline__ void unpack_qz(uint32_t w, __half2 zsub, __half2 zadd, __half2 (&o)[4]) {
  const uint32_t t0 = lop3_and_or(w, 0x000F000Fu, 0x64006400u);        // 1024 + q0 | q4
  const uint32_t t1 = lop3_and_or(w, 0x00F000F0u, 0x64006400u);        // 1024 + 16 q1 | q5
  const uint32_t w8 = w >> 8;
  const uint32_t t2 = lop3_and_or(w8, 0x000F000Fu, 0x64006400u);       // 1024 + q2 | q6
  const uint32_t t3 = lop3_and_or(w8, 0x00F000F0u, 0x64006400u);       // 1024 + 16 q3 | q7
  const __half2 sixteenth = __float2half2_rn(0.0625f);
  o[0] = __hsub2(*reinterpret_cast<const __half2*>(&t0), zsub);
  o[1] = __hfma2(*reinterpret_cast<const __half2*>(&t1), sixteenth, zadd);
  o[2] = __hsub2(*reinterpret_cast<const __half2*>(&t2), zsub);
  o[3] = __hfma2(*reinterpret_cast<const __half2*>(&t3), sixteenth, zadd);
}

// Group parameters of every row of the CTA, as half2 (step, 1024 + z), row-major with a padded
// row stride (pstride = K / G + 1) so neither the staging writes nor the per-item reads
// conflict on banks.
template <int G>
__device__ __forceinline__ void stage_params(const Args& a, uint32_t* prm, int r0, int nrows) {
  const int ng = a.K / G;
  for (int idx = threadIdx.x; idx < ng * nrows; idx += CTHREADS) {
    const int g = idx / nrows, rl = idx - (idx / nrows) * nrows;
    const long long gi = static_cast<long long>(g) * a.N + r0 + rl;
    const __half st = a.scales[gi];
    const float z = a.zeros ? static_cast<float>(a.zeros[gi]) : 8.0f;
    const __half2 v = __halves2half2(st, __float2half_rn(1024.0f + z));
    prm[rl * a.pstride + g] = *reinterpret_cast<const uint32_t*>(&v);
  }
}

// x~ / 64 of every token, staged once per CTA with coalesced 16-byte loads: slot j (channels
// 8j .. 8j+7) of token m holds the pair order (x0,x4), (x1,x5), (x2,x6), (x3,x7). fp16(x * inv_s)
// is what the folded activation would be; the 2^-6 prescale is exact on it.
template <int M>
__device__ __forceinline__ void stage_x(const Args& a, uint4* xs) {
  const int slots = a.K / 8;
  for (int idx = threadIdx.x; idx < M * slots; idx += CTHREADS) {
    const int m = idx / slots, j = idx - (idx / slots) * slots;
    const int k = 8 * j;
    const uint4 raw = __ldg(reinterpret_cast<const uint4*>(a.X + static_cast<long long>(m) * a.K + k));
    const __half* xv = reinterpret_cast<const __half*>(&raw);
    float f[8];
    if (a.inv_s) {
      const float4 ia = __ldg(reinterpret_cast<const float4*>(a.inv_s + k));
      const float4 ib = __ldg(reinterpret_cast<const float4*>(a.inv_s + k) + 1);
      const float iv[8] = {ia.x, ia.y, ia.z, ia.w, ib.x, ib.y, ib.z, ib.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) f[e] = __half2float(xv[e]) * iv[e];
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) f[e] = __half2float(xv[e]);
    }
    __align__(16) __half2 pr[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      pr[e] = __halves2half2(__float2half_rn(__half2float(__float2half_rn(f[e])) * X_PRESCALE),
                             __float2half_rn(__half2float(__float2half_rn(f[e + 4])) * X_PRESCALE));
    xs[idx] = *reinterpret_cast<const uint4*>(pr);
  }
}

template <int M, int G>
__global__ void __launch_bounds__(THREADS, 1) gemv_kernel(Args a) {
  constexpr int IPL = items_per_lane(M);
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;
  uint4* xs = reinterpret_cast<uint4*>(smem + static_cast<size_t>(a.nstages) * a.stage_bytes);
  uint32_t* prm = reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(xs) + xs_bytes(a));
  float* ysum = reinterpret_cast<float*>(prm + param_words(a));
  uint64_t* full = reinterpret_cast<uint64_t*>(ysum + ysum_floats(a));
  uint64_t* empty = full + MAX_STAGES;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + MAX_STAGES);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = static_cast<int>(static_cast<long long>(a.N) * blockIdx.x / gridDim.x);
  const int r1 = static_cast<int>(static_cast<long long>(a.N) * (blockIdx.x + 1) / gridDim.x);
  const int nrows = r1 - r0;
  const int nstage_total = (nrows + a.rows_stage - 1) / a.rows_stage;
  const uint32_t row_bytes = static_cast<uint32_t>(a.K) / 2u;

  if (threadIdx.x == 0) {
    for (int s = 0; s < a.nstages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], CWARPS);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const WaitCtx wc{a.limit_ns, abort_flag, a.status};
  // The next W4A16 launch of the stream may start now: it only prefetches its own weights and
  // group parameters until its griddepcontrol.wait.
  if (threadIdx.x == 0) pdl_launch_dependents();

  if (warp == CWARPS) {
    // ------------------------------------------------------------ producer: code stream
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      int j = 0;
      bool ok = true;
      for (; j < nstage_total; ++j) {
        const int s = j % a.nstages;
        const uint32_t ph = (j / a.nstages) & 1u;
        if (!wait_bounded(&empty[s], ph ^ 1u, wc)) { ok = false; break; }
        const int row_lo = r0 + j * a.rows_stage;
        const uint32_t bytes = static_cast<uint32_t>(min(a.rows_stage, r1 - row_lo)) * row_bytes;
        mbar_arrive_expect_tx(&full[s], bytes);
        bulk_load(ring + static_cast<size_t>(s) * a.stage_bytes,
                  a.Q + static_cast<long long>(row_lo) * (a.K >> 3), bytes, &full[s], pol);
      }
      {  // let the copies issued last land before the CTA exits (at once unless it gave up)
        for (int jj = (j > a.nstages ? j - a.nstages : 0); jj < j; ++jj)
          wait_drain(&full[jj % a.nstages], (jj / a.nstages) & 1u, a.limit_ns);
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const bool active = warp < a.parts * a.row_groups;
  const int part = warp % a.parts, rg = warp / a.parts;
  const int items = a.K / ITEM_CH;
  stage_params<G>(a, prm, r0, nrows);
  // Activations (and the output) may belong to the previous kernel of the stream: everything
  // below waits for it. The weight stream and the group parameters above do not.
  pdl_wait();
  stage_x<M>(a, xs);
  named_bar_sync(1, CTHREADS);
  // each lane's x~ slice: 4 consecutive 16-byte slots per item (conflict-free: a warp reads
  // 32 consecutive items' slots in four passes)
  __half2 xr[M][IPL][16];
  if (active) {
#pragma unroll
    for (int u = 0; u < IPL; ++u) {
      const int it = part * IPL * 32 + lane + 32 * u;
#pragma unroll
      for (int m = 0; m < M; ++m) {
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const uint4 q = it < items ? xs[m * (a.K / 8) + it * 4 + v] : make_uint4(0, 0, 0, 0);
          const __half2* h2 = reinterpret_cast<const __half2*>(&q);
#pragma unroll
          for (int e = 0; e < 4; ++e) xr[m][u][v * 4 + e] = h2[e];
        }
      }
    }
  }

  const __half2 c960 = __float2half2_rn(960.0f);
  bool ok = true;
  for (int j = 0; j < nstage_total; ++j) {
    const int s = j % a.nstages;
    const uint32_t ph = (j / a.nstages) & 1u;
    if (ok) ok = wait_bounded(&full[s], ph, wc);
    ok = __all_sync(0xffffffffu, ok);
    const int row_lo = j * a.rows_stage;               // CTA-local
    const int nr = min(a.rows_stage, nrows - row_lo);
    if (ok && active) {
      const uint8_t* stage = ring + static_cast<size_t>(s) * a.stage_bytes;
      for (int r = rg; r < nr; r += a.row_groups) {
        const int rl = row_lo + r;
        const uint8_t* codes = stage + static_cast<size_t>(r) * row_bytes;
        const uint32_t* prow = prm + rl * a.pstride;
        float acc[M];
#pragma unroll
        for (int m = 0; m < M; ++m) acc[m] = 0.f;
#pragma unroll
        for (int u = 0; u < IPL; ++u) {
          const int it = part * IPL * 32 + lane + 32 * u;
          if (it < items) {
            const uint4 qv = *reinterpret_cast<const uint4*>(codes + it * 16);
            const uint32_t pw = prow[(it * ITEM_CH) / G];
            const __half2 pv = *reinterpret_cast<const __half2*>(&pw);
            const __half2 zsub = __high2half2(pv);                     // 1024 + z
            const __half2 zadd = __hsub2(c960, zsub);             // -(64 + z), exact
            const float step64 = __low2float(pv) * 64.0f;
            const uint32_t wq[4] = {qv.x, qv.y, qv.z, qv.w};
            __half2 qz[16];
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              __half2 o[4];
              unpack_qz(wq[v], zsub, zadd, o);
#pragma unroll
              for (int e = 0; e < 4; ++e) qz[v * 4 + e] = o[e];
            }
#pragma unroll
            for (int m = 0; m < M; ++m) {
              __half2 h0 = __float2half2_rn(0.f), h1 = h0;
#pragma unroll
              for (int e = 0; e < 16; e += 2) {
                h0 = __hfma2(qz[e], xr[m][u][e], h0);
                h1 = __hfma2(qz[e + 1], xr[m][u][e + 1], h1);
              }
              const float2 f0 = __half22float2(h0), f1 = __half22float2(h1);
              acc[m] = fmaf((f0.x + f0.y) + (f1.x + f1.y), step64, acc[m]);
            }
          }
        }
#pragma unroll
        for (int m = 0; m < M; ++m) {
          float v = acc[m];
#pragma unroll
          for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          if (lane == 0) ysum[(rl * a.parts + part) * M + m] = v;
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
  named_bar_sync(1, CTHREADS);
  if (!ok) return;
  for (int i = threadIdx.x; i < nrows * M; i += CTHREADS) {
    const int m = i / nrows, r = i - (i / nrows) * nrows;
    float y = 0.f;
    for (int p = 0; p < a.parts; ++p) y += ysum[(r * a.parts + p) * M + m];
    a.Y[static_cast<long long>(m) * a.N + r0 + r] = __float2half_rn(y);
  }
}

}  // namespace gemv
}  // namespace awq
