// W4A16 GEMM for batches above the GEMV range, on the tcgen05 tensor cores.
//
// Y [M, N] = X [M, K] (dequant(Q) diag(inv_s))^T with the dequantisation fused into the
// operand staging ("AWQ > Benefits and Practical Considerations": unpack the 4-bit integers,
// apply the group scale and zero point and optionally the inverse scale, fused with the matmul
// so the fp16 weight matrix is never materialised).
//
// Operand roles are swapped so that the weight rows fill the 128-row MMA dimension and the
// (possibly small) token count is the MMA N dimension (16..256): D[n, t] = sum_k Wh[n, k] X[t, k].
//
// CTA = one 128-row x BN-token output tile, full K, 10 warps:
//   warps 0-7  dequantisers: thread (row r, half h) turns 64 codes of its row into fp16
//              (q - z) * step (* inv_s) and writes them into the 128B-swizzled K-major A tile;
//              warps 0-3 then run the epilogue (TMEM -> fp16 Y, coalesced along n).
//   warp 8     TMA loads of the X tile (two 64-channel boxes per 128-channel stage).
//   warp 9     TMEM allocation and tcgen05.mma issue (M=128, N=BN, K=16), one thread.
// A stage is 128 channels = one group of 128 (or two of 64), so each thread reads one step and
// one zero point per stage.
#pragma once

#include "awq_device.cuh"
#include "w4a16_gemv.cuh"  // lop3_and_or

namespace awq {
namespace w4tc {

constexpr int BM = 128;
constexpr int BK = 128;
constexpr int THREADS = 320;
constexpr int A_SUB = BM * 64 * 2;   // one 64-channel swizzled sub-tile: 16 KB
constexpr int A_STAGE = 2 * A_SUB;

template <int BN>
struct Cfg {
  static constexpr int B_SUB = BN * 128;
  static constexpr int B_STAGE = 2 * B_SUB;
  static constexpr int STAGES = (BN <= 64) ? 4 : (BN == 128 ? 3 : 2);
  static constexpr int SMEM = STAGES * (A_STAGE + B_STAGE) + 1024 + 256;
  static constexpr uint32_t TMEM_COLS = BN < 32 ? 32u : static_cast<uint32_t>(BN);
};

struct Args {
  const uint32_t* Q;      // [N, K/8]
  const __half* scales;   // [K/G, N]
  const uint8_t* zeros;   // [K/G, N] (asymmetric only)
  const float* inv_s;     // [K] or nullptr
  __half* Y;              // [M, N]
  int M, N, K, num_kb;
  int* status;
  unsigned long long limit_ns;
};

// 8 codes (channels 8w..8w+7 in natural order) -> 8 fp16 (q - z) * step in natural order.
__device__ __forceinline__ uint4 dequant8_f16(uint32_t w, __half2 zlo, __half2 zhi, __half2 st2) {
  const uint32_t t0 = gemv::lop3_and_or(w, 0x000F000Fu, 0x64006400u);   // q0 | q4
  const uint32_t t1 = gemv::lop3_and_or(w, 0x00F000F0u, 0x64006400u);   // 16 q1 | 16 q5
  const uint32_t w8 = w >> 8;
  const uint32_t t2 = gemv::lop3_and_or(w8, 0x000F000Fu, 0x64006400u);  // q2 | q6
  const uint32_t t3 = gemv::lop3_and_or(w8, 0x00F000F0u, 0x64006400u);  // 16 q3 | 16 q7
  // natural pairs, each mixing an unscaled (low) and a x16 (high) half
  const uint32_t p01 = __byte_perm(t0, t1, 0x5410);
  const uint32_t p23 = __byte_perm(t2, t3, 0x5410);
  const uint32_t p45 = __byte_perm(t0, t1, 0x7632);
  const uint32_t p67 = __byte_perm(t2, t3, 0x7632);
  const __half2 mul = __halves2half2(__float2half_rn(1.0f), __float2half_rn(0.0625f));
  const __half2 add = __halves2half2(__low2half(zlo), __low2half(zhi));  // -(1024+z), -(64+z)
  uint4 out;
  __half2 v;
  v = __hmul2(__hfma2(*reinterpret_cast<const __half2*>(&p01), mul, add), st2);
  out.x = *reinterpret_cast<uint32_t*>(&v);
  v = __hmul2(__hfma2(*reinterpret_cast<const __half2*>(&p23), mul, add), st2);
  out.y = *reinterpret_cast<uint32_t*>(&v);
  v = __hmul2(__hfma2(*reinterpret_cast<const __half2*>(&p45), mul, add), st2);
  out.z = *reinterpret_cast<uint32_t*>(&v);
  v = __hmul2(__hfma2(*reinterpret_cast<const __half2*>(&p67), mul, add), st2);
  out.w = *reinterpret_cast<uint32_t*>(&v);
  return out;
}

// Same with the per-channel inverse scale, in fp32: fp16((q - z) * step * inv_s_k).
__device__ __forceinline__ uint4 dequant8_f32(uint32_t w, float z, float step,
                                             const float (&inv)[8]) {
  uint4 out;
  uint32_t* o = reinterpret_cast<uint32_t*>(&out);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float a = (static_cast<float>((w >> (8 * e)) & 0xFu) - z) * step;
    const float b = (static_cast<float>((w >> (8 * e + 4)) & 0xFu) - z) * step;
    __half2 h = __floats2half2_rn(a * inv[2 * e], b * inv[2 * e + 1]);
    o[e] = *reinterpret_cast<uint32_t*>(&h);
  }
  return out;
}

template <int BN, int G, bool HAS_INV_S>
__global__ void __launch_bounds__(THREADS, 1)
    w4a16_tc_kernel(const __grid_constant__ CUtensorMap tmX, Args a) {
  using C = Cfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + C::STAGES * A_STAGE;
  uint64_t* full_a = reinterpret_cast<uint64_t*>(sB + C::STAGES * C::B_STAGE);
  uint64_t* full_b = full_a + C::STAGES;
  uint64_t* empty = full_b + C::STAGES;
  uint64_t* tfull = empty + C::STAGES;
  uint64_t* drain = tfull + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * BM, m0 = blockIdx.y * BN;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full_a[s], 256);
      mbar_init(&full_b[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tensormap(&tmX);
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const WaitCtx wc{a.limit_ns, abort_flag, a.status};
  const int kw = a.K >> 3;

  if (warp < 8) {
    // ------------------------------------------------------------ dequantise A tiles
    const int r = threadIdx.x & 127, h = threadIdx.x >> 7;
    const int row = n0 + r;
    const bool row_ok = row < a.N;
    const bool sym = a.zeros == nullptr;
    bool ok = true;
    for (int kb = 0; kb < a.num_kb; ++kb) {
      const uint32_t s = kb % C::STAGES, ph = (kb / C::STAGES) & 1u;
      const int kbase = kb * BK + h * 64;
      const bool live = row_ok && kbase < a.K;
      uint4 q0 = make_uint4(0, 0, 0, 0), q1 = q0;
      float step = 0.f, z = 0.f;
      if (live) {
        const uint4* src = reinterpret_cast<const uint4*>(a.Q + static_cast<long long>(row) * kw + (kbase >> 3));
        q0 = __ldg(src);
        q1 = __ldg(src + 1);
        const long long gi = static_cast<long long>(kbase / G) * a.N + row;
        step = __half2float(a.scales[gi]);
        z = sym ? 8.f : static_cast<float>(a.zeros[gi]);
      }
      if (!wait_bounded(&empty[s], ph ^ 1u, wc)) { ok = false; break; }
      uint8_t* dst = sA + s * A_STAGE + h * A_SUB;
      const uint32_t wq[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
      if (!live) {
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4*>(dst + sw128_offset(r, c)) = make_uint4(0, 0, 0, 0);
      } else if (HAS_INV_S) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const float4 ia = __ldg(reinterpret_cast<const float4*>(a.inv_s + kbase + 8 * c));
          const float4 ib = __ldg(reinterpret_cast<const float4*>(a.inv_s + kbase + 8 * c) + 1);
          const float inv[8] = {ia.x, ia.y, ia.z, ia.w, ib.x, ib.y, ib.z, ib.w};
          *reinterpret_cast<uint4*>(dst + sw128_offset(r, c)) = dequant8_f32(wq[c], z, step, inv);
        }
      } else {
        const __half2 zlo = __float2half2_rn(-(1024.f + z));
        const __half2 zhi = __float2half2_rn(-(64.f + z));
        const __half2 st2 = __float2half2_rn(step);
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4*>(dst + sw128_offset(r, c)) = dequant8_f16(wq[c], zlo, zhi, st2);
      }
      fence_proxy_async_smem();
      mbar_arrive(&full_a[s]);
    }
    if (warp < 4) {
      // ---------------------------------------------------------- epilogue: TMEM -> Y
      const bool got = ok && wait_bounded(tfull, 0, wc);
      if (__all_sync(0xffffffffu, got)) {  // warp-uniform: tcgen05.ld is .sync.aligned
        tc_fence_after();
        const uint32_t q = static_cast<uint32_t>(warp);
        const int orow = n0 + static_cast<int>(q) * 32 + lane;
        if constexpr (BN == 16) {
          uint32_t v[16];
          tmem_ld_x16(tmem_base + ((q * 32u) << 16), v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int t = m0 + j;
            if (t < a.M && orow < a.N)
              a.Y[static_cast<long long>(t) * a.N + orow] = __float2half_rn(__uint_as_float(v[j]));
          }
        } else {
#pragma unroll 1
          for (int c = 0; c < BN / 32; ++c) {
            uint32_t v[32];
            tmem_ld_x32(tmem_base + ((q * 32u) << 16) + c * 32, v);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int t = m0 + c * 32 + j;
              if (t < a.M && orow < a.N)
                a.Y[static_cast<long long>(t) * a.N + orow] = __float2half_rn(__uint_as_float(v[j]));
            }
          }
        }
      }
    }
  } else if (warp == 8) {
    // ------------------------------------------------------------ TMA: X tiles
    if (lane == 0) {
      int issued = 0;
      for (int kb = 0; kb < a.num_kb; ++kb) {
        const uint32_t s = kb % C::STAGES, ph = (kb / C::STAGES) & 1u;
        if (!wait_bounded(&empty[s], ph ^ 1u, wc)) break;
        mbar_arrive_expect_tx(&full_b[s], C::B_STAGE);
        tma_load_2d(sB + s * C::B_STAGE, &tmX, &full_b[s], kb * BK, m0);
        tma_load_2d(sB + s * C::B_STAGE + C::B_SUB, &tmX, &full_b[s], kb * BK + 64, m0);
        ++issued;
      }
      if (issued < a.num_kb) {  // gave up: let the copies already issued land
        const int first = issued > C::STAGES ? issued - C::STAGES : 0;
        for (int j = first; j < issued; ++j)
          wait_drain(&full_b[j % C::STAGES], (j / C::STAGES) & 1u, a.limit_ns);
      }
    }
  } else {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16_f32(BM, BN);
      bool ok = true;
      for (int kb = 0; kb < a.num_kb; ++kb) {
        const uint32_t s = kb % C::STAGES, ph = (kb / C::STAGES) & 1u;
        if (!wait_bounded(&full_a[s], ph, wc) || !wait_bounded(&full_b[s], ph, wc)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = smem_u32(sA + s * A_STAGE), b0 = smem_u32(sB + s * C::B_STAGE);
#pragma unroll
        for (int sub = 0; sub < 2; ++sub)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_f16(tmem_base, sw128_kmajor_desc(a0 + sub * A_SUB + k * 32),
                    sw128_kmajor_desc(b0 + sub * C::B_SUB + k * 32), idesc, (kb | sub | k) != 0);
        mma_commit(&empty[s]);
      }
      if (ok) mma_commit(tfull);
      mma_commit(drain);
      wait_drain(drain, 0, a.limit_ns);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

}  // namespace w4tc
}  // namespace awq
