// Group-wise 4-bit quantiser of W diag(s) and the kernels built on it.
//
// "AWQ Math", "Weight-only quantization and where it breaks": Q(w) = step * round(w / step)
// with step = max|w| / 2^(N-1) (the symmetric variant, codes clamped to [-8, 7] so 4 bits
// hold them). "Shapes, granularity, and complexity" and "AWQ > Benefits and Practical
// Considerations": one step and one zero point per group of input channels (asymmetric
// variant: the group range widened to hold 0, step = (hi - lo) / 15, z = rint(-lo / step)).
//
// Every operation that decides a code is an IEEE fp32 operation written as an intrinsic
// (__fmul_rn, __fsub_rn, __fdiv_rn, rintf), so nothing is contracted into an FMA and the codes
// are reproducible bit for bit.
//
// Thread layout shared by the kernels here: thread i of the grid owns packed word i of the
// [N, K/8] code matrix, i.e. 8 consecutive input channels of one row; the G/8 threads of a
// group are consecutive lanes of one warp and reduce the group's min/max with shuffles.
#pragma once

#include "awq_device.cuh"

namespace awq {

struct GroupParams {
  float step;  // fp32 step the codes are decided with
  float zero;  // zero point as a float (exact small integer)
};

__device__ __forceinline__ void load_scaled8(const __half* __restrict__ w_row8,
                                             const float* __restrict__ s8, bool valid,
                                             float (&wp)[8], float (&w)[8]) {
  if (!valid) {
#pragma unroll
    for (int i = 0; i < 8; ++i) { wp[i] = 0.f; w[i] = 0.f; }
    return;
  }
  const uint4 raw = *reinterpret_cast<const uint4*>(w_row8);
  const __half2* h2 = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __half22float2(h2[i]);
    w[2 * i] = f.x;
    w[2 * i + 1] = f.y;
  }
  if (s8 != nullptr) {
    const float4 sa = __ldg(reinterpret_cast<const float4*>(s8));
    const float4 sb = __ldg(reinterpret_cast<const float4*>(s8) + 1);
    const float sv[8] = {sa.x, sa.y, sa.z, sa.w, sb.x, sb.y, sb.z, sb.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) wp[i] = __fmul_rn(w[i], sv[i]);
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) wp[i] = w[i];
  }
}

// Group step and zero point; TEAM = G / 8 consecutive lanes hold one group.
template <int TEAM>
__device__ __forceinline__ GroupParams group_params(const float (&wp)[8], bool symmetric) {
  float lo = wp[0], hi = wp[0], amax = fabsf(wp[0]);
#pragma unroll
  for (int i = 1; i < 8; ++i) {
    lo = fminf(lo, wp[i]);
    hi = fmaxf(hi, wp[i]);
    amax = fmaxf(amax, fabsf(wp[i]));
  }
#pragma unroll
  for (int o = TEAM / 2; o >= 1; o >>= 1) {
    lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  }
  GroupParams g;
  if (symmetric) {
    float st = __fdiv_rn(amax, 8.0f);
    if (st == 0.0f) st = 1.0f;
    g.step = st;
    g.zero = 8.0f;
  } else {
    hi = fmaxf(hi, 0.0f);
    lo = fminf(lo, 0.0f);
    float st = __fdiv_rn(__fsub_rn(hi, lo), 15.0f);
    if (st == 0.0f) st = 1.0f;
    float z = rintf(__fdiv_rn(-lo, st));
    z = fminf(fmaxf(z, 0.0f), 15.0f);
    g.step = st;
    g.zero = z;
  }
  return g;
}

// Stored code (0..15) of one scaled weight.
__device__ __forceinline__ uint32_t code_of(float wp, const GroupParams& g, bool symmetric) {
  float r = rintf(__fdiv_rn(wp, g.step));
  if (symmetric) {
    r = fminf(fmaxf(r, -8.0f), 7.0f) + 8.0f;
  } else {
    r = fminf(fmaxf(__fadd_rn(r, g.zero), 0.0f), 15.0f);
  }
  return static_cast<uint32_t>(r);
}

// ------------------------------------------------------------------ quantize + pack kernel

struct QuantArgs {
  const __half* W;      // [N, K]
  const float* s;       // [K] or nullptr
  uint32_t* qweight;    // [N, K/8]
  __half* scales;       // [K/G, N]
  uint8_t* zeros;       // [K/G, N] or nullptr
  int N, K, symmetric;
};

template <int G>
__global__ void __launch_bounds__(256) quantize_pack_kernel(QuantArgs a) {
  constexpr int TEAM = G / 8;
  const int kw = a.K >> 3;                                   // words per row
  const long long total = static_cast<long long>(a.N) * kw;
  const long long word = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const bool valid = word < total;
  const int n = valid ? static_cast<int>(word / kw) : 0;
  const int w = valid ? static_cast<int>(word - static_cast<long long>(n) * kw) : 0;
  const int k0 = w * 8;
  float wp[8], wv[8];
  load_scaled8(a.W + static_cast<long long>(n) * a.K + k0, a.s ? a.s + k0 : nullptr, valid, wp,
               wv);
  const bool sym = a.symmetric != 0;
  const GroupParams g = group_params<TEAM>(wp, sym);
  if (!valid) return;
  uint32_t packed = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) packed |= code_of(wp[i], g, sym) << (4 * i);
  a.qweight[word] = packed;
  if ((threadIdx.x & (TEAM - 1)) == 0) {
    const long long gi = static_cast<long long>(k0 / G) * a.N + n;
    a.scales[gi] = __float2half_rn(g.step);
    if (!sym && a.zeros) a.zeros[gi] = static_cast<uint8_t>(g.zero);
  }
}

// ------------------------------------------------------------------ search-side kernels

// s[i, k] = fp32(max(m_k, 1e-6)^alpha_i) computed in fp64; inv_s = 1 / s (IEEE fp32).
struct GridArgs {
  const float* m;  // [K]
  float* s;        // [n_alpha, K]
  float* inv_s;    // [n_alpha, K]
  int K, n_alpha;
  float alphas[64];
};

__global__ void __launch_bounds__(256) scale_grid_kernel(GridArgs a) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= a.K * a.n_alpha) return;
  const int i = idx / a.K, k = idx - i * a.K;
  const double base = fmax(static_cast<double>(a.m[k]), 1e-6);
  const float s = static_cast<float>(pow(base, static_cast<double>(a.alphas[i])));
  a.s[idx] = s;
  a.inv_s[idx] = __fdiv_rn(1.0f, s);
}

// max |W| over the whole matrix, as the bit pattern of a non-negative float (atomicMax on
// unsigned int orders non-negative floats correctly; the result is order-independent).
__global__ void __launch_bounds__(256) absmax_kernel(const __half* __restrict__ W, long long n8,
                                                     unsigned int* out) {
  float m = 0.f;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const uint4 raw = __ldg(reinterpret_cast<const uint4*>(W) + i);
    const __half2* h2 = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = __half22float2(__habs2(h2[j]));
      m = fmaxf(m, fmaxf(f.x, f.y));
    }
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) atomicMax(out, __float_as_uint(m));
}

// Power-of-two factor 2^p applied to the residual before it is rounded to fp16: p puts
// max|W| (which bounds every |W - w_hat|, see the residual kernel) just below 2^14.
__device__ __forceinline__ int residual_exponent(unsigned int absmax_bits) {
  const float mx = __uint_as_float(absmax_bits);
  if (!(mx > 0.f)) return 0;
  int e;
  frexpf(mx, &e);  // mx = f * 2^e, f in [0.5, 1)  =>  mx < 2^e
  return 14 - e;
}

struct ResidualArgs {
  const __half* W;             // [N, K]
  const float* s;              // [K] scale of this alpha
  const float* inv_s;          // [K] 1 / s
  const unsigned int* absmax;  // max |W| bits
  __half* D;                   // [N, K] out: 2^p (W - Q(W diag(s)) diag(s)^-1)
  int N, K, symmetric;
};

// Residual of one alpha candidate: D = W - w_hat with w_hat = (q - z) * step16 / s, the
// dequantised weight the layer would run with. The codes are the ones quantize_pack_kernel
// writes for the same s (same code path). |W - w_hat| <= |W|: an unclamped code rounds w' to
// within step/2, and a weight whose |w'| is below step/2 rounds to the zero level (w_hat = 0),
// so either the error is at most step/(2 s) <= |w| or it equals |w|; a clamped code sits at
// least 7.5 steps out, where the one-step error is below |w'| too. Hence 2^p max|W| < 2^14
// keeps every residual inside the fp16 range.
template <int G>
__global__ void __launch_bounds__(256) residual_kernel(ResidualArgs a) {
  constexpr int TEAM = G / 8;
  const int kw = a.K >> 3;
  const long long total = static_cast<long long>(a.N) * kw;
  const long long word = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const bool valid = word < total;
  const int n = valid ? static_cast<int>(word / kw) : 0;
  const int w = valid ? static_cast<int>(word - static_cast<long long>(n) * kw) : 0;
  const int k0 = w * 8;
  float wp[8], wv[8];
  load_scaled8(a.W + static_cast<long long>(n) * a.K + k0, a.s + k0, valid, wp, wv);
  const bool sym = a.symmetric != 0;
  const GroupParams g = group_params<TEAM>(wp, sym);
  if (!valid) return;
  const float step16 = __half2float(__float2half_rn(g.step));
  const float p2 = ldexpf(1.0f, residual_exponent(*a.absmax));
  const float4 ia = __ldg(reinterpret_cast<const float4*>(a.inv_s + k0));
  const float4 ib = __ldg(reinterpret_cast<const float4*>(a.inv_s + k0) + 1);
  const float inv[8] = {ia.x, ia.y, ia.z, ia.w, ib.x, ib.y, ib.z, ib.w};
  __align__(16) __half out[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float qz = static_cast<float>(code_of(wp[i], g, sym)) - g.zero;  // exact
    const float w_hat = __fmul_rn(__fmul_rn(qz, step16), inv[i]);
    out[i] = __float2half_rn(__fmul_rn(__fsub_rn(wv[i], w_hat), p2));
  }
  *reinterpret_cast<uint4*>(a.D + static_cast<long long>(n) * a.K + k0) =
      *reinterpret_cast<const uint4*>(out);
}

}  // namespace awq
