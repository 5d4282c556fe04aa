// Group-wise N-bit quantiser of W diag(s) and the kernels built on it.
//
// "AWQ Math", "Weight-only quantization and where it breaks": Q(w) = step * round(w / step)
// with step = max|w| / 2^(N-1) for N-bit codes (the symmetric variant, codes clamped to
// [-2^(N-1), 2^(N-1) - 1] and stored as q + 8). "Shapes, granularity, and complexity" and
// "AWQ > Benefits and Practical Considerations": one step and one zero point per group of input
// channels (asymmetric variant: the group range widened to hold 0, step = (hi - lo) / (2^N - 1),
// z = rint(-lo / step)). N is 4 by default, 3 or 2 for the narrower variants; every width is
// stored in 4-bit nibbles.
//
// Every operation that decides a code is an IEEE fp32 operation written as an intrinsic
// (__fmul_rn, __fsub_rn, __fdiv_rn, rintf), so nothing is contracted into an FMA and the codes
// are reproducible bit for bit; the per-weight division is replaced by a multiplication with
// the correctly rounded reciprocal wherever that provably gives the same rounded quotient.
//
// Thread layout shared by the quantising kernels here: a lane owns one packed word (8
// consecutive input channels) of several rows; the G/8 lanes of a group are consecutive lanes
// of one warp and reduce the group's min/max with shuffles.
#pragma once

#include "awq_device.cuh"

namespace awq {

struct GroupParams {
  float step;  // fp32 step the codes are decided with
  float zero;  // zero point as a float (exact small integer)
  float rcp;   // 1 / step, correctly rounded
  float clo;   // smallest and largest stored code: 0 and 2^N - 1, or 8 -+ 2^(N-1) (symmetric)
  float chi;
};

__device__ __forceinline__ GroupParams group_params_of(float lo, float hi, bool symmetric,
                                                      int bits);

// Round to the nearest integer, ties to even, for |x| < 2^22: x + 1.5 * 2^23 lies in a binade
// whose unit in the last place is 1, so that IEEE addition rounds x itself (1.5 * 2^23 is even,
// so ties land on even integers) and the subtraction is exact. Two full-rate adds.
__device__ __forceinline__ float rint_small(float x) {
  return __fsub_rn(__fadd_rn(x, 0x1.8p23f), 0x1.8p23f);
}

// fl32(d / n) for d >= 0 and n = 2^bits - 1 (15, 7 or 3) without a division: q0 = fl32(d * r)
// with r = fl32(1/n), the remainder e = d - n q0 (exact in one FMA), and one correction
// q0 + e r rounded once (Markstein's correction step, "IA-64 and Elementary Functions", 2000).
// The result is the correctly rounded quotient for every d whose quotient is a normal float:
// the rounding pattern of d / n depends only on d's significand, and all 2^23 significands were
// checked against exact rational arithmetic for each n. Smaller d take the IEEE division.
__device__ __forceinline__ float div_levels(float d, int bits) {
  const float n = bits == 4 ? 15.0f : (bits == 3 ? 7.0f : 3.0f);
  const float r = bits == 4 ? 0x1.111112p-4f : (bits == 3 ? 0x1.24924ap-3f : 0x1.555556p-2f);
  if (d < 0x1p-100f) return __fdiv_rn(d, n);
  const float q0 = __fmul_rn(d, r);
  return __fmaf_rn(__fmaf_rn(-q0, n, d), r, q0);
}

// Step, zero point, reciprocal and code range of a group from the min and max of its w'.
__device__ __forceinline__ GroupParams group_params_of(float lo, float hi, bool symmetric,
                                                      int bits) {
  GroupParams g;
  if (symmetric) {
    const float half = bits == 4 ? 8.0f : (bits == 3 ? 4.0f : 2.0f);  // 2^(N-1)
    const float amax = fmaxf(hi, -lo);  // max |w'| of the group
    // fl32(amax / 2^(N-1)) as a multiplication by the exact power of two: the same value,
    // rounded once
    float st = __fmul_rn(amax, bits == 4 ? 0.125f : (bits == 3 ? 0.25f : 0.5f));
    if (st == 0.0f) st = 1.0f;
    g.step = st;
    g.zero = 8.0f;
    g.rcp = __frcp_rn(st);
    g.clo = 8.0f - half;
    g.chi = 7.0f + half;
  } else {
    const float qmax = bits == 4 ? 15.0f : (bits == 3 ? 7.0f : 3.0f);  // 2^N - 1
    hi = fmaxf(hi, 0.0f);
    lo = fminf(lo, 0.0f);
    float st = div_levels(__fsub_rn(hi, lo), bits);
    if (st == 0.0f) st = 1.0f;
    g.step = st;
    g.rcp = __frcp_rn(st);
    // rint(fl32(-lo / st)) as in rint_quotient: 0 <= -lo <= hi - lo, so the quotient is below 16
    const float t = __fmul_rn(-lo, g.rcp);
    float z = rint_small(t);
    if (fabsf(__fsub_rn(t, z)) >= 0.5f - 0x1p-17f) z = rintf(__fdiv_rn(-lo, st));
    g.zero = fminf(fmaxf(z, 0.0f), qmax);
    g.clo = 0.0f;
    g.chi = qmax;
  }
  return g;
}

// The rule every kernel here decides codes by, in its plainest form (the kernels apply it in
// the shifted domain below, with the same integers): rint(fl32(wp / step)) without a division
// in the common case. |wp / step| <= 15 for every
// weight of the group, so t = fl32(wp * fl32(1 / step)) is within 2^-19 of the exact quotient
// and fl32 of the quotient within 2^-20 of it: unless t lies within 2^-17 of a half-integer (a
// rounding boundary of rint), t and the IEEE quotient round to the same integer. With
// r = rint(t), t - r is exact and t is that close to a half-integer exactly when
// |t - r| >= 1/2 - 2^-17; there (about 1.5e-5 of all weights) the quotient is computed with
// IEEE division.
__device__ __forceinline__ float rint_quotient(float wp, const GroupParams& g) {
  const float t = __fmul_rn(wp, g.rcp);
  const float r = rint_small(t);
  if (fabsf(__fsub_rn(t, r)) >= 0.5f - 0x1p-17f) return rintf(__fdiv_rn(wp, g.step));
  return r;
}

struct QuantArgs {
  const __half* W;      // [N, K]
  const float* s;       // [K] or nullptr
  const float* clip;    // [K/G, N] clip ratios or nullptr (no clipping)
  uint32_t* qweight;    // [N, K/8]
  __half* scales;       // [K/G, N]
  uint8_t* zeros;       // [K/G, N] or nullptr
  int N, K, symmetric;
  int bits;             // code width: 4, 3 or 2
};

// Row-tiled launch shape of residual_kernel (and the residual warps of the search kernels): a
// block of 8 warps covers 32 packed words (256 channels) of 8 * QROWS rows (rows along grid x,
// 256-channel column chunks along grid y); lane l owns word 32 blockIdx.y + l of the QROWS rows
// of its warp. The per-channel scales are loaded once per lane and the QROWS 16-byte weight
// loads are issued together, so every thread keeps 64 bytes of HBM reads in flight. A group
// (G / 8 words) is G / 8 consecutive lanes of one row.
constexpr int QROWS = 4;

__device__ __forceinline__ void load8f(const float* p, bool ok, float fill, float (&v)[8]) {
  if (ok) {
    const float4 lo = __ldg(reinterpret_cast<const float4*>(p));
    const float4 hi = __ldg(reinterpret_cast<const float4*>(p) + 1);
    v[0] = lo.x; v[1] = lo.y; v[2] = lo.z; v[3] = lo.w;
    v[4] = hi.x; v[5] = hi.y; v[6] = hi.z; v[7] = hi.w;
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = fill;
  }
}

__device__ __forceinline__ void unpack8(const uint4& raw, float (&w)[8]) {
  const __half2* h2 = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __half22float2(h2[i]);
    w[2 * i] = f.x;
    w[2 * i + 1] = f.y;
  }
}

// ------------------------------------------------------------------ quantize + pack kernel

// Run-per-thread launch shape of quantize_pack_kernel and clip_search_kernel: a thread owns a
// run of RUN consecutive channels of one row (RUN <= G), so a group is G / RUN adjacent lanes
// (TEAM). The group's min and max then take log2(TEAM) shuffles and its step and zero point are
// computed once per thread, not once per 8 channels. A block of 256 threads covers 256 / TEAM
// consecutive rows of one group (rows along grid x, groups along grid y); its lanes read the
// same channels of different rows, so the per-channel loads (scales, energies) are warp-wide
// broadcasts, and the step and zero point stores are coalesced. Both run 32 channels per thread:
// the pack in 64 registers (four blocks per SM keep enough reads in flight), the clipping
// search, which holds its run's w' over all ratios, at three blocks per SM (measured against
// 64-channel runs at two).
template <int G, int MAXRUN>
struct RunShape {
  static constexpr int RUN = G < MAXRUN ? G : MAXRUN;   // channels per thread
  static constexpr int TEAM = G / RUN;                  // threads per group: 1, 2 or 4
  static constexpr int ROWS = 256 / TEAM;               // rows per block
  static_assert(G % RUN == 0 && TEAM <= 4, "group sizes 32, 64 and 128");
};
constexpr int PACK_RUN = 32;
constexpr int CLIP_RUN = 32;

// min and max over the TEAM lanes of a group (adjacent lanes; every lane takes the shuffles)
template <int TEAM>
__device__ __forceinline__ void team_range(float& lo, float& hi) {
#pragma unroll
  for (int o = TEAM / 2; o >= 1; o >>= 1) {
    lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
  }
}

// The thread's run: its RUN / 8 16-byte weight loads issued together, then w' = fl32(w s) as
// RUN / 2 pairs (w itself without a scale) and the run's smallest and largest w'. Rows past N
// load zeros (their results are never stored).
template <int RUN>
__device__ __forceinline__ void load_run(const __half* W, const float* s, long long off, int k0,
                                         bool ok, float2 (&v)[RUN / 2], float& lo, float& hi) {
  uint4 raw[RUN / 8];
#pragma unroll
  for (int i = 0; i < RUN / 8; ++i)
    raw[i] = ok ? __ldg(reinterpret_cast<const uint4*>(W + off) + i) : make_uint4(0, 0, 0, 0);
#pragma unroll
  for (int i = 0; i < RUN / 8; ++i) {
    const __half2* h2 = reinterpret_cast<const __half2*>(&raw[i]);
    float sv[8];
    load8f(s + k0 + 8 * i, s != nullptr, 1.0f, sv);
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const float2 w2 = __half22float2(h2[p]);
      v[4 * i + p] = s ? mul2_rn(w2, make_float2(sv[2 * p], sv[2 * p + 1])) : w2;
    }
  }
  lo = fminf(v[0].x, v[0].y);
  hi = fmaxf(v[0].x, v[0].y);
#pragma unroll
  for (int p = 1; p < RUN / 2; ++p) {
    lo = fminf(lo, fminf(v[p].x, v[p].y));
    hi = fmaxf(hi, fmaxf(v[p].x, v[p].y));
  }
}

// The codes in the shifted domain: with C = 1.5 * 2^23 + zero (an integer whose unit in the
// last place is 1), u = fl32(w' rcp + C) = C + rint(w' rcp) in one FMA, exactly the integer
// rint_quotient gives unless w' rcp - rint(w' rcp) lies within 2^-17 of +-1/2 (checked per
// 8 channels, IEEE division there). The clamped u holds the stored code in its low four bits.
// Element pairs go through the paired fp32 instructions (the same IEEE operations).
constexpr float kShift = 0x1.8p23f;
constexpr float kNearTie = 0.5f - 0x1p-17f;

template <int G>
__global__ void __launch_bounds__(256, 4) quantize_pack_kernel(QuantArgs a) {
  using S = RunShape<G, PACK_RUN>;
  constexpr int RUN = S::RUN;
  const int t = threadIdx.x % S::TEAM;                      // run within the group
  const int row = blockIdx.x * S::ROWS + threadIdx.x / S::TEAM;
  const int gi = blockIdx.y;                                // group index along K
  const int k0 = gi * G + t * RUN;
  const bool ok = row < a.N;
  const long long r64 = ok ? row : 0;
  float2 v[RUN / 2];
  float lo, hi;
  load_run<RUN>(a.W, a.s, r64 * a.K + k0, k0, ok, v, lo, hi);
  team_range<S::TEAM>(lo, hi);
  if (a.clip != nullptr) {
    // magnitudes bounded by b = fl32(c max|w'|): the range ends are cut to it
    const float cr = a.clip[static_cast<long long>(gi) * a.N + r64];
    const float b = __fmul_rn(fmaxf(hi, -lo), cr);
    hi = fminf(fmaxf(hi, 0.0f), b);
    lo = fmaxf(fminf(lo, 0.0f), -b);
  }
  const GroupParams g = group_params_of(lo, hi, a.symmetric != 0, a.bits);
  const float c = __fadd_rn(kShift, g.zero);
  const float2 c2 = make_float2(c, c), rcp2 = make_float2(g.rcp, g.rcp);
  const float2 m1 = make_float2(-1.0f, -1.0f);
  const float ulo = __fadd_rn(kShift, g.clo), uhi = __fadd_rn(kShift, g.chi);
  uint32_t words[RUN / 8];
#pragma unroll
  for (int i = 0; i < RUN / 8; ++i) {
    float2 u[4];
    float fm = 0.0f;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      u[p] = fma2_rn(v[4 * i + p], rcp2, c2);
      const float2 f = fma2_rn(v[4 * i + p], rcp2, fma2_rn(u[p], m1, c2));
      fm = fmaxf(fm, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
    if (fm >= kNearTie) {   // see rint_quotient
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        u[p].x = __fadd_rn(rintf(__fdiv_rn(v[4 * i + p].x, g.step)), c);
        u[p].y = __fadd_rn(rintf(__fdiv_rn(v[4 * i + p].y, g.step)), c);
      }
    }
    uint32_t packed = 0;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const uint32_t c0 = __float_as_uint(fminf(fmaxf(u[p].x, ulo), uhi)) & 0xFu;
      const uint32_t c1 = __float_as_uint(fminf(fmaxf(u[p].y, ulo), uhi)) & 0xFu;
      packed |= (c0 | (c1 << 4)) << (8 * p);
    }
    words[i] = packed;
  }
  if (ok) {
    uint4* dst = reinterpret_cast<uint4*>(a.qweight + r64 * (a.K >> 3) + (k0 >> 3));
#pragma unroll
    for (int i = 0; i < RUN / 32; ++i)
      dst[i] = make_uint4(words[4 * i], words[4 * i + 1], words[4 * i + 2], words[4 * i + 3]);
    static_assert(RUN % 32 == 0, "a run packs into whole 16-byte stores");
    if (t == 0) {
      const long long gidx = static_cast<long long>(gi) * a.N + row;
      a.scales[gidx] = __float2half_rn(g.step);
      if (a.symmetric == 0 && a.zeros) a.zeros[gidx] = static_cast<uint8_t>(g.zero);
    }
  }
}

// ------------------------------------------------------------------ clipping search

// Per-group clip ratio (a reading; the pages print no clipping step): for each ratio c of the
// grid, the group's magnitudes are bounded by b = fl32(c max|w'|) (asymmetric ends cut to
// min(hi, b) and max(lo, -b), symmetric max|w'| -> b), the group is quantised exactly as the
// pack kernel does with that bound, and its error e(c) = sum_k h_k (W - w_hat)^2 (h the channel
// energy sum_t x_tk^2, w_hat = (q - z) step16 / s) is accumulated in fp32 in the scaled domain:
// W - w_hat = (w' - (q - z) step16) / s, so each term is g_k r_k^2 with g_k = fl32(h_k / fl32(s_k^2))
// and r_k = fl32(w' - (q - z) step16) in one FMA ((q - z) step16 is exact: a small integer times
// an fp16 value). Against the exact terms, r_k / s_k is within 2^-23 (|W| + |w_hat|) of
// W - w_hat and g_k within 2^-23 relative of h_k / s_k^2; a thread adds its run in two fixed
// chains of pairs (pair index mod 2), the lanes of a group their sums in a butterfly. The first ratio with the smallest error wins; the
// group's first thread writes it to clip[g, n].
constexpr int MAX_CLIP_RATIOS = 32;

struct ClipArgs {
  const __half* W;       // [N, K]
  const float* s;        // [K] or nullptr
  const float* energy;   // [K] sum_t x^2
  float* clip;           // [K/G, N] out
  int N, K, symmetric, bits, n_ratio;
  float ratios[MAX_CLIP_RATIOS];
};

// 16-byte shared-memory load kept inside its loop (volatile): the channel weights are read
// again for every ratio instead of being held in 64 registers beside the run's w'.
__device__ __forceinline__ float4 lds_f4(const float* p) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))));
  return v;
}

// 16-byte read-only global loads the compiler may not merge with earlier loads of the same
// address (volatile): the near-tie path reloads its run instead of keeping the first loads live.
__device__ __forceinline__ uint4 ldg_u4_again(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(reinterpret_cast<uint64_t>(p)));
  return v;
}
__device__ __forceinline__ float4 ldg_f4_again(const float* p) {
  float4 v;
  asm volatile("ld.global.nc.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(reinterpret_cast<uint64_t>(p)));
  return v;
}

// One pair's term of the clipping criterion: g (w' - (code - zero) step16)^2 added to acc, with
// -(code - zero) = nq clamped to [nlo, nhi].
__device__ __forceinline__ void clip_term(float2 vp, float2 nq, float nlo, float nhi, float2 st2,
                                          float2 gp, float2& acc) {
  const float2 nc = make_float2(fminf(fmaxf(nq.x, nlo), nhi), fminf(fmaxf(nq.y, nlo), nhi));
  const float2 r = fma2_rn(nc, st2, vp);           // w' - (code - zero) step16
  acc = fma2_rn(mul2_rn(gp, r), r, acc);
}

// The quantiser of one clip ratio in the form the criterion uses: the IEEE step (for the
// near-tie division), its reciprocal, C = 1.5 * 2^23 + zero, the clamp range of -(code - zero)
// and the stored fp16 step.
struct RatioParams {
  float step, rcp, c, nlo, nhi, st16;
};

__device__ __forceinline__ RatioParams ratio_params(float lo, float hi, float amax, float ratio,
                                                    bool sym, int bits) {
  const float b = __fmul_rn(amax, ratio);
  const GroupParams g = group_params_of(fmaxf(fminf(lo, 0.0f), -b), fminf(fmaxf(hi, 0.0f), b),
                                        sym, bits);
  RatioParams r;
  r.step = g.step;
  r.rcp = g.rcp;
  r.c = __fadd_rn(kShift, g.zero);
  r.nlo = __fsub_rn(g.zero, g.chi);   // -(code - zero) lies in [zero - chi, zero - clo]
  r.nhi = __fsub_rn(g.zero, g.clo);
  r.st16 = __half2float(__float2half_rn(g.step));
  return r;
}

template <int G>
__global__ void __launch_bounds__(256, 3) clip_search_kernel(ClipArgs a) {
  using S = RunShape<G, CLIP_RUN>;
  constexpr int RUN = S::RUN;
  constexpr int GP = RUN + 4;   // run stride in shared memory: a group's runs start on other banks
  __shared__ __align__(16) float gsh[S::TEAM * GP];
  const int gi = blockIdx.y;
  for (int i = threadIdx.x; i < G; i += blockDim.x) {
    const int k = gi * G + i;
    float gk = a.energy[k];
    if (a.s) {
      const float sk = a.s[k];
      gk = __fdiv_rn(gk, __fmul_rn(sk, sk));
    }
    gsh[(i / RUN) * GP + i % RUN] = gk;
  }
  __syncthreads();
  const int t = threadIdx.x % S::TEAM;
  const int row = blockIdx.x * S::ROWS + threadIdx.x / S::TEAM;
  const int k0 = gi * G + t * RUN;
  const bool ok = row < a.N;
  const long long off = (ok ? row : 0) * static_cast<long long>(a.K) + k0;
  float2 v[RUN / 2];
  float lo, hi;
  load_run<RUN>(a.W, a.s, off, k0, ok, v, lo, hi);
  team_range<S::TEAM>(lo, hi);
  const float* gt = gsh + t * GP;
  const bool sym = a.symmetric != 0;
  const float amax = fmaxf(hi, -lo);
  const float2 m1 = make_float2(-1.0f, -1.0f);
  float best_e = 0.0f;
  int best_j = 0;
#pragma unroll 1
  for (int j = 0; j < a.n_ratio; ++j) {
    const RatioParams P = ratio_params(lo, hi, amax, a.ratios[j], sym, a.bits);
    const float2 c2 = make_float2(P.c, P.c), rcp2 = make_float2(P.rcp, P.rcp);
    const float2 st2 = make_float2(P.st16, P.st16);
    // two independent chains of pairs (pair index mod 2) for the sums and the near-tie test
    // (four chains cost spills at three blocks per SM and measured 2.6 % slower). The test
    // takes the remainder g = w' rcp + nc against the clamped code: the IEEE rounding can give
    // another clamped code only where the fast one lies within 2^-17 of a rounding boundary
    // (|f| >= 1/2 - 2^-17 for f = w' rcp + nq, see rint_quotient) and the other candidate
    // clamps differently, and then |g| is within 2^-17 of 1/2 (g = f inside the range, f -+ 1
    // where the fast code is one past an end). Clamped weights far outside the range, such as
    // a group's largest magnitude under ratio 0.6 (exactly 12.5 steps), do not trigger it.
    // |g^2 - 1/4| <= 2^-16 covers |g| - 1/2 within 2^-17.
    float2 e[2];
    float fm[2];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      e[c] = make_float2(0.0f, 0.0f);
      fm[c] = 1.0f;
    }
    const float2 mq2 = make_float2(-0.25f, -0.25f);
#pragma unroll
    for (int q = 0; q < RUN / 4; ++q) {
      const float4 gq = lds_f4(gt + 4 * q);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int c = h;
        const float2 vp = v[2 * q + h];
        const float2 u = fma2_rn(vp, rcp2, c2);          // C + rint(w' rcp)
        const float2 nq = fma2_rn(u, m1, c2);            // -rint(w' rcp), exact
        const float2 nc = make_float2(fminf(fmaxf(nq.x, P.nlo), P.nhi),
                                      fminf(fmaxf(nq.y, P.nlo), P.nhi));
        const float2 g = fma2_rn(vp, rcp2, nc);          // remainder against the clamped code
        const float2 tq = fma2_rn(g, g, mq2);            // g^2 - 1/4
        fm[c] = fminf(fm[c], fminf(fabsf(tq.x), fabsf(tq.y)));
        const float2 r = fma2_rn(nc, st2, vp);           // w' - (code - zero) step16
        const float2 gp = h ? make_float2(gq.z, gq.w) : make_float2(gq.x, gq.y);
        e[c] = fma2_rn(mul2_rn(gp, r), r, e[c]);
      }
    }
    if (fminf(fm[0], fm[1]) <= 0x1p-16f) {
      // a near-tie in the run (rare): the same sum with IEEE division at the near-ties, the
      // run's w' rebuilt from memory 8 channels at a time (the same products)
#pragma unroll
      for (int c = 0; c < 2; ++c) e[c] = make_float2(0.0f, 0.0f);
#pragma unroll 1
      for (int i = 0; i < RUN / 8; ++i) {
        const uint4 raw = ok ? ldg_u4_again(a.W + off + 8 * i) : make_uint4(0, 0, 0, 0);
        const __half2* h2 = reinterpret_cast<const __half2*>(&raw);
        float sv[8] = {1.0f, 1.0f, 1.0f, 1.0f, 1.0f, 1.0f, 1.0f, 1.0f};
        if (a.s) {
          const float4 s0 = ldg_f4_again(a.s + k0 + 8 * i), s1 = ldg_f4_again(a.s + k0 + 8 * i + 4);
          sv[0] = s0.x; sv[1] = s0.y; sv[2] = s0.z; sv[3] = s0.w;
          sv[4] = s1.x; sv[5] = s1.y; sv[6] = s1.z; sv[7] = s1.w;
        }
        const float4 ga = lds_f4(gt + 8 * i), gb = lds_f4(gt + 8 * i + 4);
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const float2 w2 = __half22float2(h2[p]);
          const float2 vp = a.s ? mul2_rn(w2, make_float2(sv[2 * p], sv[2 * p + 1])) : w2;
          float2 nq = fma2_rn(fma2_rn(vp, rcp2, c2), m1, c2);
          const float2 f = fma2_rn(vp, rcp2, nq);
          if (fabsf(f.x) >= kNearTie) nq.x = -rintf(__fdiv_rn(vp.x, P.step));
          if (fabsf(f.y) >= kNearTie) nq.y = -rintf(__fdiv_rn(vp.y, P.step));
          const float4 gg = p < 2 ? ga : gb;
          clip_term(vp, nq, P.nlo, P.nhi, st2,
                    (p & 1) ? make_float2(gg.z, gg.w) : make_float2(gg.x, gg.y), e[p & 1]);
        }
      }
    }
    float err = __fadd_rn(__fadd_rn(e[0].x, e[0].y), __fadd_rn(e[1].x, e[1].y));
    // the team's lanes add the same two values (in either order: the same sum in every lane)
#pragma unroll
    for (int o = S::TEAM / 2; o >= 1; o >>= 1)
      err = __fadd_rn(err, __shfl_xor_sync(0xffffffffu, err, o));
    if (j == 0 || err < best_e) {
      best_e = err;
      best_j = j;
    }
  }
  if (ok && t == 0) a.clip[static_cast<long long>(gi) * a.N + row] = a.ratios[best_j];
}

// ------------------------------------------------------------------ search-side kernels

// s[i, k] = max(m_k, 1e-6)^alpha_i in fp32, inv_s = 1 / s (IEEE fp32). The logarithm
// L = log2(base) is taken once per channel in fp64 and y = alpha_i L in fp64 (for base in
// [1e-6, 2^64], |L| <= 64, so y is within about 2^-46 of exact); y splits into an integer n =
// rint(y) and f = fl32(y - n) with |f| <= 1/2 (y - n is exact in fp64, its rounding to fp32 at
// most 2^-25), and s = 2^n exp2f(f), the scaling by 2^n exact. exp2f is within 2 ulp (CUDA's
// documented bound) and f's rounding moves the power by at most 2^-25 ln 2 relative, so s lies
// within 3 fp32 spacings of the exact power: below 4e-7 relative. Only the logarithm and one
// product per alpha run in fp64, whose rate on this part is a small fraction of fp32's.
struct GridArgs {
  const float* m;  // [K]
  float* s;        // [n_alpha, K]
  float* inv_s;    // [n_alpha, K]
  int K, n_alpha;
  float alphas[64];
};

constexpr int GRID_ALPHAS = 4;  // alphas per thread (blockIdx.y picks the chunk)

__global__ void __launch_bounds__(128) scale_grid_kernel(GridArgs a) {
  const int k = blockIdx.x * blockDim.x + threadIdx.x;
  if (k >= a.K) return;
  const double lb = log2(fmax(static_cast<double>(a.m[k]), 1e-6));
  const int i0 = blockIdx.y * GRID_ALPHAS;
#pragma unroll
  for (int j = 0; j < GRID_ALPHAS; ++j) {
    const int i = i0 + j;
    if (i < a.n_alpha) {
      const double y = lb * static_cast<double>(a.alphas[i]);
      const double n = rint(y);
      const float s = ldexpf(exp2f(static_cast<float>(y - n)), static_cast<int>(n));
      const long long idx = static_cast<long long>(i) * a.K + k;
      a.s[idx] = s;
      a.inv_s[idx] = __fdiv_rn(1.0f, s);
    }
  }
}

// max |W| over the whole matrix, as the bit pattern of a non-negative float (atomicMax on
// unsigned int orders non-negative floats correctly; the result is order-independent).
// Four 16-byte loads in flight per thread per step.
__global__ void __launch_bounds__(256) absmax_kernel(const __half* __restrict__ W, long long n8,
                                                     unsigned int* out) {
  float m = 0.f;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i0 = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i0 < n8;
       i0 += 4 * stride) {
    uint4 raw[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const long long i = i0 + u * stride;
      raw[u] = i < n8 ? __ldg(reinterpret_cast<const uint4*>(W) + i) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const __half2* h2 = reinterpret_cast<const __half2*>(&raw[u]);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = __half22float2(__habs2(h2[j]));
        m = fmaxf(m, fmaxf(f.x, f.y));
      }
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
  int bits;                    // code width: 4, 3 or 2
};

// Residual of one alpha candidate: D = W - w_hat with w_hat = (q - z) * step16 / s, the
// dequantised weight the layer would run with. The codes are the ones quantize_pack_kernel
// writes for the same s (same code path). |W - w_hat| <= |W|: an unclamped code rounds w' to
// within step/2, and a weight whose |w'| is below step/2 rounds to the zero level (w_hat = 0),
// so either the error is at most step/(2 s) <= |w| or it equals |w|; a clamped code sits at
// least 7.5 steps out, where the one-step error is below |w'| too. Hence 2^p max|W| < 2^14
// keeps every residual inside the fp16 range.
// One block of the residual, `warps` warps high (8 in residual_kernel): warp `warp` covers rows
// (rb * warps + warp) * QROWS .. + QROWS - 1, lane `lane` the packed word 32 chunk + lane of each. Split into the loads
// (residual_load: the lane's QROWS weight words, from HBM) and the rest (residual_store, which
// reads the lane's 8 channels of s and 1/s, shared by every row and so cached), so a caller
// can overlap the next block's weight loads with this block's work.
struct ResidualRegs {
  uint4 raw[QROWS];
  int rbase, k0;
  bool wok;
};

__device__ __forceinline__ void residual_load(const ResidualArgs& a, int rb, int chunk, int warp,
                                              int lane, ResidualRegs& r, int warps = 8) {
  const int w = chunk * 32 + lane;
  r.wok = w < (a.K >> 3);
  r.k0 = (r.wok ? w : 0) * 8;
  r.rbase = (rb * warps + warp) * QROWS;
#pragma unroll
  for (int q = 0; q < QROWS; ++q) {
    const int row = r.rbase + q;
    r.raw[q] = (r.wok && row < a.N)
                   ? __ldg(reinterpret_cast<const uint4*>(a.W + static_cast<long long>(row) * a.K + r.k0))
                   : make_uint4(0, 0, 0, 0);
  }
}

// The arithmetic runs in phases over RB rows at a time, so the rows' independent chains
// interleave: w' and the lane's min/max; the team shuffles; the group parameters; the rounded
// quotients, with one check per lane for a quotient near a rounding boundary (a single rare
// branch instead of one per weight, redone with IEEE division for the lane's RB rows, which
// gives the same integers everywhere else); then the codes, w_hat and the residual. RB is
// bounded by the registers the calling kernel can spare.
constexpr int RES_RB = 2;

template <int TEAM, int RB>
__device__ __forceinline__ void residual_rows(const ResidualArgs& a, const ResidualRegs& r, int q0,
                                              const float (&sv)[8], const float (&iv)[8],
                                              float p2) {
  const bool sym = a.symmetric != 0;
  // Element pairs (2 i, 2 i + 1) go through the paired fp32 instructions (fma2_rn, mul2_rn):
  // the same IEEE operations as one element at a time, half the instructions.
  float2 v[RB][4];  // w', then the shifted rounded quotients
  float lo[RB], hi[RB];
#pragma unroll
  for (int q = 0; q < RB; ++q) {
    float wv[8];
    unpack8(r.raw[q0 + q], wv);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      v[q][i] = mul2_rn(make_float2(wv[2 * i], wv[2 * i + 1]), make_float2(sv[2 * i], sv[2 * i + 1]));
    lo[q] = fminf(v[q][0].x, v[q][0].y);
    hi[q] = fmaxf(v[q][0].x, v[q][0].y);
#pragma unroll
    for (int i = 1; i < 4; ++i) {
      lo[q] = fminf(lo[q], fminf(v[q][i].x, v[q][i].y));
      hi[q] = fmaxf(hi[q], fmaxf(v[q][i].x, v[q][i].y));
    }
  }
#pragma unroll
  for (int o = TEAM / 2; o >= 1; o >>= 1) {
#pragma unroll
    for (int q = 0; q < RB; ++q) {
      lo[q] = fminf(lo[q], __shfl_xor_sync(0xffffffffu, lo[q], o));
      hi[q] = fmaxf(hi[q], __shfl_xor_sync(0xffffffffu, hi[q], o));
    }
  }
  GroupParams g[RB];
#pragma unroll
  for (int q = 0; q < RB; ++q) g[q] = group_params_of(lo[q], hi[q], sym, a.bits);
  // The integers are carried shifted by kM = 1.5 * 2^23, where the unit in the last place is 1:
  // u = fl32(w' rcp + kM) = kM + rint(w' rcp) in one FMA, and kM - u = -rint(w' rcp) exactly
  // (formed as fma(u, -1, kM), the same exact value), so fma(w', rcp, kM - u) is
  // w' rcp - rint(w' rcp) rounded once. Where that lies within 2^-17 of +-1/2 the exact product
  // w' rcp (within 2^-19 of the quotient, like t in rint_quotient) may round differently from
  // fl32(w' / step); elsewhere both give rint_quotient's integer.
  constexpr float kM = 0x1.8p23f;
  const float2 kM2 = make_float2(kM, kM), m1 = make_float2(-1.0f, -1.0f);
  float fmax_abs = 0.0f;
#pragma unroll
  for (int q = 0; q < RB; ++q) {
    const float2 rcp2 = make_float2(g[q].rcp, g[q].rcp);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 u = fma2_rn(v[q][i], rcp2, kM2);
      const float2 f = fma2_rn(v[q][i], rcp2, fma2_rn(u, m1, kM2));
      fmax_abs = fmaxf(fmax_abs, fmaxf(fabsf(f.x), fabsf(f.y)));
      v[q][i] = u;
    }
  }
  if (fmax_abs >= 0.5f - 0x1p-17f) {  // see rint_quotient
#pragma unroll
    for (int q = 0; q < RB; ++q) {
      float wv[8];
      unpack8(r.raw[q0 + q], wv);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        v[q][i].x = __fadd_rn(rintf(__fdiv_rn(__fmul_rn(wv[2 * i], sv[2 * i]), g[q].step)), kM);
        v[q][i].y = __fadd_rn(rintf(__fdiv_rn(__fmul_rn(wv[2 * i + 1], sv[2 * i + 1]), g[q].step)), kM);
      }
    }
  }
  const float2 p22 = make_float2(p2, p2);
#pragma unroll
  for (int q = 0; q < RB; ++q) {
    const int row = r.rbase + q0 + q;
    // kM + (code - zero), clamped as code_f clamps the code (exact small integers plus kM)
    const float ulo = __fadd_rn(kM, __fsub_rn(g[q].clo, g[q].zero));
    const float uhi = __fadd_rn(kM, __fsub_rn(g[q].chi, g[q].zero));
    // With sp = step16 p2 (p2 a power of two, so exact): fma(u, sp, -kM sp) = (code - zero) sp
    // exactly (an integer below 16 times an 11-bit significand), times -1/s rounded once is
    // -fl32((code - zero) step16 / s) p2 = -w_hat p2, and fma(w, p2, -w_hat p2) =
    // fl32(w - w_hat) p2: the same bits as scaling after each rounding.
    const float sp = __fmul_rn(__half2float(__float2half_rn(g[q].step)), p2);
    const float2 sp2 = make_float2(sp, sp);
    const float2 msp2 = make_float2(-__fmul_rn(kM, sp), -__fmul_rn(kM, sp));
    float wv[8];
    unpack8(r.raw[q0 + q], wv);
    uint32_t out[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 uc = make_float2(fminf(fmaxf(v[q][i].x, ulo), uhi), fminf(fmaxf(v[q][i].y, ulo), uhi));
      const float2 nwh = mul2_rn(fma2_rn(uc, sp2, msp2), make_float2(-iv[2 * i], -iv[2 * i + 1]));
      const float2 d = fma2_rn(make_float2(wv[2 * i], wv[2 * i + 1]), p22, nwh);
      const __half2 h = __floats2half2_rn(d.x, d.y);
      memcpy(&out[i], &h, sizeof(uint32_t));
    }
    if (r.wok && row < a.N)
      *reinterpret_cast<uint4*>(a.D + static_cast<long long>(row) * a.K + r.k0) =
          make_uint4(out[0], out[1], out[2], out[3]);
  }
}

// One block's residual given the lane's 8 channels of s and 1/s.
template <int G>
__device__ __forceinline__ void residual_compute(const ResidualArgs& a, const ResidualRegs& r,
                                                 const float (&sv)[8], const float (&iv)[8],
                                                 float p2) {
  static_assert(QROWS % RES_RB == 0, "row batches must tile the rows");
#pragma unroll
  for (int q0 = 0; q0 < QROWS; q0 += RES_RB) residual_rows<G / 8, RES_RB>(a, r, q0, sv, iv, p2);
}

template <int G>
__device__ __forceinline__ void residual_store(const ResidualArgs& a, const ResidualRegs& r,
                                               float p2) {
  float sv[8], iv[8];
  load8f(a.s + r.k0, r.wok, 1.0f, sv);
  load8f(a.inv_s + r.k0, r.wok, 1.0f, iv);
  residual_compute<G>(a, r, sv, iv, p2);
}

// Row blocks of 8 * QROWS rows on grid x, 256-channel column chunks on grid y.
template <int G>
__global__ void __launch_bounds__(256) residual_kernel(ResidualArgs a) {
  ResidualRegs r;
  residual_load(a, blockIdx.x, blockIdx.y, threadIdx.x >> 5, threadIdx.x & 31, r);
  residual_store<G>(a, r, ldexpf(1.0f, residual_exponent(*a.absmax)));
}

}  // namespace awq
