// W4A16 decode GEMV (M <= 8 tokens) on the CUDA cores.
//
// "AWQ > Benefits and Practical Considerations": decode is bound by reading the weights from
// HBM; the kernel unpacks the 4-bit integers, applies the group scale and zero point and,
// optionally, the per-channel inverse scale, fused with the product so no fp16 weight matrix is
// ever written.
//
// Layout of the work:
//   * each CTA owns a contiguous range of output rows (balanced to within one row), so the
//     per-group scale/zero sectors it reads are shared by its warps through L1;
//   * the activations x~ = x * inv_s (fp32 product, rounded to fp16) are staged once per CTA in
//     shared memory, in the pair order the nibble unpacking produces ((x0,x4), (x1,x5), ...);
//   * a warp takes R rows at a time; per 1024-channel step each lane reads 16 bytes (32 codes)
//     of each row and the matching x~ from shared memory (laid out so the 32 lanes read 32
//     consecutive 16-byte slots: no bank conflicts);
//   * codes are unpacked with the 0x6400 fp16 exponent trick into exact (q - z) half2 pairs,
//     multiplied by x~ with HFMA2 over the lane's 32 channels, then converted to fp32 and scaled
//     by the group step: y += step * sum (q - z) x~;
//   * lane partials are reduced with warp shuffles into per-row fp32 sums in shared memory.
#pragma once

#include "awq_device.cuh"

namespace awq {
namespace gemv {

constexpr int THREADS = 256;
constexpr int WARPS = THREADS / 32;
constexpr int R = 2;            // rows per warp pass
constexpr int STEP_K = 1024;    // channels per warp step (32 lanes x 32)

struct Args {
  const __half* X;        // [M, K]
  const uint32_t* Q;      // [N, K/8]
  const __half* scales;   // [K/G, N]
  const uint8_t* zeros;   // [K/G, N] (asymmetric only)
  const float* inv_s;     // [K] or nullptr
  __half* Y;              // [M, N]
  int M, N, K;
  int kc;                 // channels staged per chunk (multiple of STEP_K)
  int rows_max;           // max rows of any CTA (size of the per-row sums)
};

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));  // (a & b) | c
  return d;
}

// 8 codes of one word -> 4 exact half2 (q - z) pairs in the order (0,4), (1,5), (2,6), (3,7).
__device__ __forceinline__ void unpack_qz(uint32_t w, __half2 zlo, __half2 zhi, __half2 (&o)[4]) {
  const uint32_t t0 = lop3_and_or(w, 0x000F000Fu, 0x64006400u);        // 1024 + q0 | q4
  const uint32_t t1 = lop3_and_or(w, 0x00F000F0u, 0x64006400u);        // 1024 + 16 q1 | q5
  const uint32_t w8 = w >> 8;
  const uint32_t t2 = lop3_and_or(w8, 0x000F000Fu, 0x64006400u);       // 1024 + q2 | q6
  const uint32_t t3 = lop3_and_or(w8, 0x00F000F0u, 0x64006400u);       // 1024 + 16 q3 | q7
  const __half2 sixteenth = __float2half2_rn(0.0625f);
  o[0] = __hsub2(*reinterpret_cast<const __half2*>(&t0), zlo);          // - (1024 + z)
  o[1] = __hfma2(*reinterpret_cast<const __half2*>(&t1), sixteenth, zhi);  // /16 - (64 + z)
  o[2] = __hsub2(*reinterpret_cast<const __half2*>(&t2), zlo);
  o[3] = __hfma2(*reinterpret_cast<const __half2*>(&t3), sixteenth, zhi);
}

template <int M, int G>
__global__ void __launch_bounds__(THREADS, 2) gemv_kernel(Args a) {
  extern __shared__ uint4 smem4[];
  // x~ staging: [M][kc/8] 16-byte slots; per-row sums after it: [rows_max][M] fp32
  uint4* xs = smem4;
  float* ysum = reinterpret_cast<float*>(smem4 + static_cast<size_t>(M) * (a.kc / 8));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = static_cast<int>(static_cast<long long>(a.N) * blockIdx.x / gridDim.x);
  const int r1 = static_cast<int>(static_cast<long long>(a.N) * (blockIdx.x + 1) / gridDim.x);
  const int nrows = r1 - r0;
  const int kw = a.K >> 3;
  const bool sym = a.zeros == nullptr;

  for (int i = threadIdx.x; i < nrows * M; i += THREADS) ysum[i] = 0.f;

  for (int kbeg = 0; kbeg < a.K; kbeg += a.kc) {
    const int klen = min(a.kc, a.K - kbeg);
    const int nslots = a.kc / 8;
    __syncthreads();
    // ---- stage x~ for this chunk in the lane-interleaved pair order
    for (int idx = threadIdx.x; idx < M * nslots; idx += THREADS) {
      const int m = idx / nslots, j = idx - (idx / nslots) * nslots;   // logical slot j
      const int k = kbeg + 8 * j;
      __align__(16) __half h[8];
      if (8 * j < klen) {
        const uint4 raw = __ldg(reinterpret_cast<const uint4*>(a.X + static_cast<long long>(m) * a.K + k));
        const __half* xv = reinterpret_cast<const __half*>(&raw);
        if (a.inv_s) {
          const float4 ia = __ldg(reinterpret_cast<const float4*>(a.inv_s + k));
          const float4 ib = __ldg(reinterpret_cast<const float4*>(a.inv_s + k) + 1);
          const float iv[8] = {ia.x, ia.y, ia.z, ia.w, ib.x, ib.y, ib.z, ib.w};
#pragma unroll
          for (int e = 0; e < 8; ++e) h[e] = __float2half_rn(__half2float(xv[e]) * iv[e]);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) h[e] = xv[e];
        }
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) h[e] = __float2half_rn(0.f);
      }
      __align__(16) __half2 pr[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) pr[e] = __halves2half2(h[e], h[e + 4]);
      const int step = j >> 7, rr = j & 127, l = rr >> 2, u = rr & 3;
      xs[m * nslots + step * 128 + u * 32 + l] = *reinterpret_cast<const uint4*>(pr);
    }
    __syncthreads();

    // ---- rows of this CTA, R at a time per warp
    const int nsteps = (klen + STEP_K - 1) / STEP_K;
    for (int rb = warp * R; rb < nrows; rb += WARPS * R) {
      float acc[R][M];
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < M; ++m) acc[r][m] = 0.f;

      for (int st = 0; st < nsteps; ++st) {
        const int w0 = (kbeg >> 3) + st * 128 + lane * 4;   // first word of this lane
        const bool lane_ok = w0 < kw;
        const int g = (w0 * 8) / G;
        uint4 qv[R];
        float step[R];
        __half2 zlo[R], zhi[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const int row = r0 + rb + r;
          const bool ok = lane_ok && (rb + r) < nrows;
          qv[r] = ok ? __ldg(reinterpret_cast<const uint4*>(a.Q + static_cast<long long>(row) * kw + w0))
                     : make_uint4(0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u);
          const long long gi = static_cast<long long>(g) * a.N + row;
          step[r] = ok ? __half2float(a.scales[gi]) : 0.f;
          const float z = sym ? 8.f : (ok ? static_cast<float>(a.zeros[gi]) : 8.f);
          zlo[r] = __float2half2_rn(1024.f + z);
          zhi[r] = __float2half2_rn(-(64.f + z));
        }
        __half2 qz[R][16];
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const uint32_t wq[4] = {qv[r].x, qv[r].y, qv[r].z, qv[r].w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            __half2 o[4];
            unpack_qz(wq[u], zlo[r], zhi[r], o);
#pragma unroll
            for (int e = 0; e < 4; ++e) qz[r][u * 4 + e] = o[e];
          }
        }
        const int slot0 = st * 128 + lane;
#pragma unroll
        for (int m = 0; m < M; ++m) {
          const uint4* xm = xs + m * nslots + slot0;
          __half2 hacc[R];
#pragma unroll
          for (int r = 0; r < R; ++r) hacc[r] = __float2half2_rn(0.f);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint4 xv = xm[u * 32];
            const __half2* x2 = reinterpret_cast<const __half2*>(&xv);
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
              for (int e = 0; e < 4; ++e) hacc[r] = __hfma2(qz[r][u * 4 + e], x2[e], hacc[r]);
          }
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const float2 f = __half22float2(hacc[r]);
            acc[r][m] = fmaf(step[r], f.x + f.y, acc[r][m]);
          }
        }
      }
      // ---- reduce lane partials, add into the per-row sums
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < M; ++m) {
          float v = acc[r][m];
#pragma unroll
          for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          if (lane == 0 && rb + r < nrows) ysum[(rb + r) * M + m] += v;
        }
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < nrows * M; i += THREADS) {
    const int m = i / nrows, r = i - (i / nrows) * nrows;
    a.Y[static_cast<long long>(m) * a.N + r0 + r] = __float2half_rn(ysum[r * M + m]);
  }
}

}  // namespace gemv
}  // namespace awq
