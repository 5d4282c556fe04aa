// W4A16 decode GEMV (M <= 4 tokens) on the CUDA cores.
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
// x~ = fp16(x * inv_s) (what the folded activation would be) once in shared memory as 16-bit
// block fixed point, x~ = x_int 2^(e - 15) with one exponent e per 32 channels (max|x~| < 2^e,
// so |x_int| < 2^15; exact for every x~ within 2^5 of the block's maximum, rounded to the
// nearest integer below that), split into a low byte plane (0..255) and a signed high byte
// plane (x_int = 256 hi + lo), and each lane copies its K slice into registers. Afterwards the
// only shared-memory traffic per code is the bulk copy's write and one 16-byte read per item.
// Per item and row:
//   * the 8 codes of a word become two words of 4 bytes (even and odd nibbles: one AND, one
//     shift-and-AND);
//   * four DP4A integer dot products (codes x low plane unsigned, codes x high plane signed)
//     accumulate sum q x_int exactly in 32-bit integers;
//   * the zero point comes off as z * sum x_int (staged per item), and the exact integer is
//     scaled by step * 2^(e - 15) into an fp32 row accumulator.
// So the only roundings are the fixed point of small activations and the fp32 accumulation
// over items. Row partials are reduced with shuffles and written to shared memory per (row,
// part); the parts are added in a fixed order at the end, so the result is deterministic.
//
// The group parameters of the CTA's rows (fp16 steps and uint8 zero points, [K/G, N] in global
// memory) arrive by two 2-D TMA box loads issued before the weight stream: a box of the CTA's
// rows (its start rounded down to 16 rows) by up to 256 groups, so they land in a microsecond
// or so instead of being gathered element by element. Shapes whose parameter arrays cannot be
// described by such boxes (N not a multiple of 16, more rows per CTA than a box holds) stage
// them with plain loads instead.
//
// Launched with programmatic dependent launch: the kernel lets the next W4A16 launch of the
// stream start right after its own set-up, and it streams its weights and loads its group
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
constexpr int MAX_M = 4;
constexpr int MAX_STAGES = 8;
constexpr int SMEM_BUDGET = 220 * 1024;

// Items per lane for M tokens: the registers holding x~ stay at 64 per thread or below.
__host__ __device__ constexpr int items_per_lane(int M) { return M == 1 ? 4 : (M == 2 ? 2 : 1); }

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
  int pbox_cols;          // TMA parameter boxes: rows per box (a multiple of 16), 0 = plain loads
  int pbox_groups;        // groups per box (<= 256); the boxes are stacked along the groups
  int x_direct;           // 1: each lane converts its own activations (no staged x planes)
  int* status;
  unsigned long long limit_ns;
};

// Shared-memory footprint for the given launch shape (the host sizes the launch with it).
__host__ __device__ inline int ysum_floats(const Args& a) {
  return (a.rows_max * a.parts * a.M + 3) & ~3;
}
// Boxes of group parameters: ceil((K / G) / pbox_groups), each pbox_groups x pbox_cols.
__host__ __device__ inline int pbox_count(const Args& a) {
  return (a.pstride - 1 + a.pbox_groups - 1) / a.pbox_groups;
}
// Shared-memory words of the group parameters: packed (step, zero) words per (row, group) for
// the plain staging, or the TMA boxes of fp16 steps (and, asymmetric, uint8 zero points) with
// 128-byte aligned bases.
__host__ __device__ inline int param_words(const Args& a) {
  if (a.pbox_cols == 0) return (a.rows_max * a.pstride + 3) & ~3;
  const int rows = pbox_count(a) * a.pbox_groups;
  const int sbytes = (rows * a.pbox_cols * 2 + 127) & ~127;
  const int zbytes = a.zeros ? ((rows * a.pbox_cols + 127) & ~127) : 0;
  return (sbytes + zbytes) / 4;
}
// x planes: 16 words per (token, 32-channel item), i.e. 2 bytes per activation (none when each
// lane converts its own)
__host__ __device__ inline size_t xs_bytes(const Args& a) {
  return a.x_direct ? 0 : static_cast<size_t>(a.M) * static_cast<size_t>(a.K) * 2;
}
// per (token, item): sum of x_int (int) and 2^(e - 15) (float)
__host__ __device__ inline size_t xitem_bytes(const Args& a) {
  return a.x_direct ? 0 : static_cast<size_t>(a.M) * static_cast<size_t>(a.K / ITEM_CH) * 8;
}
// [ring | x planes | x item sums and scales | (128-byte aligned) parameters | row sums |
//  barriers]; 128 bytes of slack for the alignment of the parameters
__host__ __device__ inline size_t smem_bytes(const Args& a) {
  return static_cast<size_t>(a.nstages) * a.stage_bytes + xs_bytes(a) + xitem_bytes(a) + 128 +
         static_cast<size_t>(param_words(a)) * 4 + static_cast<size_t>(ysum_floats(a)) * 4 +
         (2 * MAX_STAGES + 1) * 8 + 16;
}

__device__ __forceinline__ uint32_t dp4a_uu(uint32_t a, uint32_t b, uint32_t c) {
  return __dp4a(a, b, c);
}
__device__ __forceinline__ int dp4a_ss(uint32_t a, uint32_t b, int c) {
  return __dp4a(static_cast<int>(a), static_cast<int>(b), c);
}

// Group parameters of every row of the CTA, one word each: the fp16 step in the low half and
// the zero point in bits 16..23, row-major with a padded row stride (pstride = K / G + 1) so
// neither the staging writes nor the per-item reads conflict on banks.
template <int G>
__device__ __forceinline__ void stage_params(const Args& a, uint32_t* prm, int r0, int nrows) {
  const int ng = a.K / G;
  for (int idx = threadIdx.x; idx < ng * nrows; idx += CTHREADS) {
    const int g = idx / nrows, rl = idx - (idx / nrows) * nrows;
    const long long gi = static_cast<long long>(g) * a.N + r0 + rl;
    const __half st = a.scales[gi];
    const uint32_t z = a.zeros ? static_cast<uint32_t>(a.zeros[gi]) : 8u;
    prm[rl * a.pstride + g] = static_cast<uint32_t>(__half_as_ushort(st)) | (z << 16);
  }
}

// x~ of every token as 16-bit block fixed point, staged once per CTA. Slot s (token m, item
// it, word w: channels 32 it + 8 w .. + 7) goes to consumer thread s mod CTHREADS, so the four
// words of an item sit on four consecutive lanes; each thread issues the loads of up to four
// slots before converting any (the loads come from L2 or HBM, so batching them shortens the
// prologue). A lane rounds x * inv_s of its 8 channels to fp16; the four lanes take the item's
// max|x~| (a max over the float bits, which order like the values for |x~|) and e with
// max|x~| < 2^e; each lane forms x_int = rint(x~ 2^(15 - e)) and packs its word's four byte
// planes with byte permutes: the low bytes of channels 8w + 0, 2, 4, 6 (even nibbles), of
// 8w + 1, 3, 5, 7 (odd nibbles), then the signed high bytes in the same two orders
// (x_int = 256 hi + lo). The 16 bytes go to xs[(m * 4 + w) * items + it], so a warp that reads
// word w of 32 consecutive items reads 512 contiguous bytes (no bank conflict). The item's sum
// of x_int and 2^(e - 15) go to xsum / xsc.
template <int M>
__device__ __forceinline__ void stage_x(const Args& a, uint32_t* xs, int* xsum, float* xsc) {
  constexpr int U = 4;                      // slots per thread whose loads are in flight together
  const int wpt = a.K / 8;                  // words (slots) per token
  const int items = a.K / ITEM_CH;
  const int total = M * wpt;                // a multiple of 4: K is a multiple of 32
  const int lane = threadIdx.x & 31;
  for (int s0 = threadIdx.x - lane; s0 < total; s0 += U * CTHREADS) {   // warp-uniform bound
    uint4 raw[U];
    float4 ia[U], ib[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int s = s0 + u * CTHREADS + lane;
      const bool on = s < total;
      const int m = on ? s / wpt : 0, k = on ? (s - m * wpt) * 8 : 0;
      raw[u] = on ? __ldg(reinterpret_cast<const uint4*>(a.X + static_cast<long long>(m) * a.K + k))
                  : make_uint4(0, 0, 0, 0);
      if (a.inv_s && on) {
        ia[u] = __ldg(reinterpret_cast<const float4*>(a.inv_s + k));
        ib[u] = __ldg(reinterpret_cast<const float4*>(a.inv_s + k) + 1);
      } else {
        ia[u] = make_float4(1.f, 1.f, 1.f, 1.f);
        ib[u] = ia[u];
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (s0 + u * CTHREADS >= total) break;   // warp-uniform: the shuffles below need all lanes
      const int s = s0 + u * CTHREADS + lane;
      const bool on = s < total;
      const __half* xv = reinterpret_cast<const __half*>(&raw[u]);
      const float iv[8] = {ia[u].x, ia[u].y, ia[u].z, ia[u].w, ib[u].x, ib[u].y, ib[u].z, ib[u].w};
      float f[8];
      if (a.inv_s) {
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = __half2float(__float2half_rn(__half2float(xv[e]) * iv[e]));
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = __half2float(xv[e]);
      }
      float mx = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) mx = fmaxf(mx, fabsf(f[e]));
      unsigned mb = __float_as_uint(mx);
      mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
      mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
      int ex = 0;
      frexpf(__uint_as_float(mb), &ex);       // max|x~| < 2^ex (0 for an all-zero item)
      const float up = ldexpf(1.0f, 15 - ex);
      int xi[8];
      int sum = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        xi[e] = __float2int_rn(f[e] * up);    // the product is exact (a power-of-two scale)
        sum += xi[e];
      }
      sum += __shfl_xor_sync(0xffffffffu, sum, 1);
      sum += __shfl_xor_sync(0xffffffffu, sum, 2);
      if (on) {
        // byte 0 (low) or 1 (high) of channels (0, 2) and (4, 6), or (1, 3) and (5, 7)
        const uint32_t le = __byte_perm(__byte_perm(xi[0], xi[2], 0x0040), __byte_perm(xi[4], xi[6], 0x0040), 0x5410);
        const uint32_t lo = __byte_perm(__byte_perm(xi[1], xi[3], 0x0040), __byte_perm(xi[5], xi[7], 0x0040), 0x5410);
        const uint32_t he = __byte_perm(__byte_perm(xi[0], xi[2], 0x0051), __byte_perm(xi[4], xi[6], 0x0051), 0x5410);
        const uint32_t ho = __byte_perm(__byte_perm(xi[1], xi[3], 0x0051), __byte_perm(xi[5], xi[7], 0x0051), 0x5410);
        const int mi = s >> 2;                  // m * items + it
        const int m = mi / items, it = mi - m * items, w = s & 3;
        reinterpret_cast<uint4*>(xs)[(m * 4 + w) * items + it] = make_uint4(le, lo, he, ho);
        if (w == 0) {
          xsum[mi] = sum;
          xsc[mi] = ldexpf(1.0f, ex - 15);
        }
      }
    }
  }
}

// The same conversion done by one lane for one whole item it owns (long K: every lane's items
// are its own, so nothing is shared and nothing staged): the 32 activations from global memory,
// max|x~| and e within the lane, the four words' byte planes with byte permutes.
__device__ __forceinline__ void convert_item(const Args& a, int m, int it, uint32_t (&planes)[16],
                                             int& xsum_out, float& xsc_out) {
  const int k0 = it * ITEM_CH;
  __half2 h[16];
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    const uint4 raw = __ldg(reinterpret_cast<const uint4*>(a.X + static_cast<long long>(m) * a.K +
                                                           k0 + 8 * v));
    const __half* xv = reinterpret_cast<const __half*>(&raw);
    float f[8];
    if (a.inv_s) {
      const float4 ia = __ldg(reinterpret_cast<const float4*>(a.inv_s + k0 + 8 * v));
      const float4 ib = __ldg(reinterpret_cast<const float4*>(a.inv_s + k0 + 8 * v) + 1);
      const float iv[8] = {ia.x, ia.y, ia.z, ia.w, ib.x, ib.y, ib.z, ib.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) f[e] = __half2float(xv[e]) * iv[e];
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) f[e] = __half2float(xv[e]);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e)
      h[4 * v + e] = __halves2half2(__float2half_rn(f[2 * e]), __float2half_rn(f[2 * e + 1]));
  }
  float mx = 0.f;
#pragma unroll
  for (int c = 0; c < 16; ++c) {
    const float2 p = __half22float2(h[c]);
    mx = fmaxf(mx, fmaxf(fabsf(p.x), fabsf(p.y)));
  }
  int ex = 0;
  frexpf(mx, &ex);                          // max|x~| < 2^ex (0 for an all-zero item)
  const float up = ldexpf(1.0f, 15 - ex);
  int sum = 0;
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    int xi[8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 p = __half22float2(h[4 * w + e]);
      xi[2 * e] = __float2int_rn(p.x * up);      // the product is exact (a power-of-two scale)
      xi[2 * e + 1] = __float2int_rn(p.y * up);
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) sum += xi[e];
    planes[4 * w + 0] = __byte_perm(__byte_perm(xi[0], xi[2], 0x0040), __byte_perm(xi[4], xi[6], 0x0040), 0x5410);
    planes[4 * w + 1] = __byte_perm(__byte_perm(xi[1], xi[3], 0x0040), __byte_perm(xi[5], xi[7], 0x0040), 0x5410);
    planes[4 * w + 2] = __byte_perm(__byte_perm(xi[0], xi[2], 0x0051), __byte_perm(xi[4], xi[6], 0x0051), 0x5410);
    planes[4 * w + 3] = __byte_perm(__byte_perm(xi[1], xi[3], 0x0051), __byte_perm(xi[5], xi[7], 0x0051), 0x5410);
  }
  xsum_out = sum;
  xsc_out = ldexpf(1.0f, ex - 15);
}

// One pass of a consumer warp over NR rows of a stage (rows r, r + RG, ...): each lane's
// items of every row against its activation planes, the row sums reduced over the warp and
// written per (row, K part).
template <int M, int G, int IPL, int NR>
__device__ __forceinline__ void row_pass(const Args& a, const uint8_t* stage, uint32_t row_bytes,
                                         int row_lo, int r, int part, int lane, int items,
                                         const __half* sbox, const uint8_t* zbox, int poff,
                                         const uint32_t* prm, const uint32_t (&xr)[M][IPL][16],
                                         const int (&sx)[M][IPL], const float (&sc)[M][IPL],
                                         float* ysum) {
  int rl[NR];
  const uint8_t* codes[NR];
#pragma unroll
  for (int h = 0; h < NR; ++h) {
    rl[h] = row_lo + r + h * a.row_groups;
    codes[h] = stage + static_cast<size_t>(r + h * a.row_groups) * row_bytes;
  }
  float acc[NR][M];
#pragma unroll
  for (int h = 0; h < NR; ++h)
#pragma unroll
    for (int m = 0; m < M; ++m) acc[h][m] = 0.f;
#pragma unroll
  for (int u = 0; u < IPL; ++u) {
    const int it = part * IPL * 32 + lane + 32 * u;
    if (it < items) {
      const int g = (it * ITEM_CH) / G;
#pragma unroll
      for (int h = 0; h < NR; ++h) {
        const uint4 qv = *reinterpret_cast<const uint4*>(codes[h] + it * 16);
        float step;
        int z;
        if (a.pbox_cols) {
          const int gi = g * a.pbox_cols + rl[h] + poff;
          step = __half2float(sbox[gi]);
          z = a.zeros ? static_cast<int>(zbox[gi]) : 8;
        } else {
          const uint32_t pw = prm[rl[h] * a.pstride + g];
          step = __half2float(__ushort_as_half(static_cast<unsigned short>(pw & 0xFFFFu)));
          z = static_cast<int>((pw >> 16) & 0xFFu);
        }
        const uint32_t wq[4] = {qv.x, qv.y, qv.z, qv.w};
        uint32_t ev[4], od[4];
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          ev[v] = wq[v] & 0x0F0F0F0Fu;          // nibbles 0, 2, 4, 6 as bytes
          od[v] = (wq[v] >> 4) & 0x0F0F0F0Fu;   // nibbles 1, 3, 5, 7
        }
#pragma unroll
        for (int m = 0; m < M; ++m) {
          // four independent chains of four DP4A (even / odd nibbles, low / high planes), so
          // consecutive instructions do not wait on each other's results
          uint32_t lo0 = 0u, lo1 = 0u;
          int hi0 = 0, hi1 = 0;
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            lo0 = dp4a_uu(ev[v], xr[m][u][4 * v + 0], lo0);
            lo1 = dp4a_uu(od[v], xr[m][u][4 * v + 1], lo1);
            hi0 = dp4a_ss(ev[v], xr[m][u][4 * v + 2], hi0);
            hi1 = dp4a_ss(od[v], xr[m][u][4 * v + 3], hi1);
          }
          // sum (q - z) x_int, exact: |.| < 32 * 15 * 2^15 < 2^24, so the float is exact too
          const int t = (hi0 + hi1) * 256 + static_cast<int>(lo0 + lo1) - z * sx[m][u];
          acc[h][m] = fmaf(static_cast<float>(t), step * sc[m][u], acc[h][m]);
        }
      }
    }
  }
#pragma unroll
  for (int m = 0; m < M; ++m) {
    float v[NR];
#pragma unroll
    for (int h = 0; h < NR; ++h) v[h] = acc[h][m];
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1)
#pragma unroll
      for (int h = 0; h < NR; ++h) v[h] += __shfl_xor_sync(0xffffffffu, v[h], o);
    if (lane == 0)
#pragma unroll
      for (int h = 0; h < NR; ++h) ysum[(rl[h] * a.parts + part) * M + m] = v[h];
  }
}

template <int M, int G>
__global__ void __launch_bounds__(THREADS, 1)
    gemv_kernel(const __grid_constant__ CUtensorMap tmS, const __grid_constant__ CUtensorMap tmZ,
                Args a) {
  constexpr int IPL = items_per_lane(M);
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;
  uint32_t* xs = reinterpret_cast<uint32_t*>(smem + static_cast<size_t>(a.nstages) * a.stage_bytes);
  int* xsum = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(xs) + xs_bytes(a));
  float* xsc = reinterpret_cast<float*>(xsum + M * (a.K / ITEM_CH));
  uint32_t* prm = reinterpret_cast<uint32_t*>(
      (reinterpret_cast<uintptr_t>(xs) + xs_bytes(a) + xitem_bytes(a) + 127) & ~uintptr_t{127});
  float* ysum = reinterpret_cast<float*>(prm + param_words(a));
  uint64_t* full = reinterpret_cast<uint64_t*>(ysum + ysum_floats(a));
  uint64_t* empty = full + MAX_STAGES;
  uint64_t* pbar = empty + MAX_STAGES;          // the parameter boxes
  volatile int* abort_flag = reinterpret_cast<volatile int*>(pbar + 1);
  // TMA parameter boxes: fp16 steps [boxes * pbox_groups][pbox_cols], then (asymmetric) the
  // uint8 zero points in the same shape, 128-byte aligned; column c of a box is output row
  // x0 + c, x0 = r0 rounded down to 16
  const int prows = a.pbox_cols ? pbox_count(a) * a.pbox_groups : 0;
  const __half* sbox = reinterpret_cast<const __half*>(prm);
  const uint8_t* zbox = reinterpret_cast<const uint8_t*>(prm) + ((prows * a.pbox_cols * 2 + 127) & ~127);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = static_cast<int>(static_cast<long long>(a.N) * blockIdx.x / gridDim.x);
  const int r1 = static_cast<int>(static_cast<long long>(a.N) * (blockIdx.x + 1) / gridDim.x);
  const int nrows = r1 - r0;
  const int nstage_total = (nrows + a.rows_stage - 1) / a.rows_stage;
  const uint32_t row_bytes = static_cast<uint32_t>(a.K) / 2u;

  const int x0 = r0 & ~15;
  if (threadIdx.x == 0) {
    for (int s = 0; s < a.nstages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], CWARPS);
    }
    mbar_init(pbar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    if (a.pbox_cols) {
      prefetch_tensormap(&tmS);
      if (a.zeros) prefetch_tensormap(&tmZ);
    }
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
      if (a.pbox_cols) {   // the group parameters first: the consumers need them at once
        const int nb = pbox_count(a);
        const uint32_t box = static_cast<uint32_t>(a.pbox_groups * a.pbox_cols);
        mbar_arrive_expect_tx(pbar, static_cast<uint32_t>(nb) * box * (a.zeros ? 3u : 2u));
        for (int b = 0; b < nb; ++b) {
          tma_load_2d(const_cast<__half*>(sbox) + static_cast<size_t>(b) * box, &tmS, pbar, x0,
                      b * a.pbox_groups);
          if (a.zeros)
            tma_load_2d(const_cast<uint8_t*>(zbox) + static_cast<size_t>(b) * box, &tmZ, pbar, x0,
                        b * a.pbox_groups);
        }
      }
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
        if (a.pbox_cols) wait_drain(pbar, 0, a.limit_ns);
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const bool active = warp < a.parts * a.row_groups;
  const int part = warp % a.parts, rg = warp / a.parts;
  const int items = a.K / ITEM_CH;
  if (!a.pbox_cols) stage_params<G>(a, prm, r0, nrows);
  // Activations (and the output) may belong to the previous kernel of the stream: everything
  // below waits for it. The weight stream and the group parameters above do not.
  pdl_wait();
  if (!a.x_direct) stage_x<M>(a, xs, xsum, xsc);
  named_bar_sync(1, CTHREADS);
  bool ok = true;
  if (a.pbox_cols) ok = wait_bounded(pbar, 0, wc);
  // each lane's x planes (16 words per item: four 16-byte loads), the item's sum of x_int and
  // its 2^(e - 15), kept in registers for the whole kernel
  uint32_t xr[M][IPL][16];
  int sx[M][IPL];
  float sc[M][IPL];
  if (active) {
#pragma unroll
    for (int u = 0; u < IPL; ++u) {
      const int it = part * IPL * 32 + lane + 32 * u;
#pragma unroll
      for (int m = 0; m < M; ++m) {
        const bool ok_it = it < items;
        if (a.x_direct) {
          if (ok_it) {
            convert_item(a, m, it, xr[m][u], sx[m][u], sc[m][u]);
          } else {
#pragma unroll
            for (int v = 0; v < 16; ++v) xr[m][u][v] = 0u;
            sx[m][u] = 0;
            sc[m][u] = 0.0f;
          }
          continue;
        }
        const int xi = m * items + (ok_it ? it : 0);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const uint4 q = ok_it ? reinterpret_cast<const uint4*>(xs)[(m * 4 + v) * items + it]
                                : make_uint4(0, 0, 0, 0);
          xr[m][u][4 * v + 0] = q.x;
          xr[m][u][4 * v + 1] = q.y;
          xr[m][u][4 * v + 2] = q.z;
          xr[m][u][4 * v + 3] = q.w;
        }
        sx[m][u] = ok_it ? xsum[xi] : 0;
        sc[m][u] = ok_it ? xsc[xi] : 0.0f;
      }
    }
  }

  const int poff = r0 - x0;   // column of the CTA's first row in the parameter boxes
  for (int j = 0; j < nstage_total; ++j) {
    const int s = j % a.nstages;
    const uint32_t ph = (j / a.nstages) & 1u;
    if (ok) ok = wait_bounded(&full[s], ph, wc);
    ok = __all_sync(0xffffffffu, ok);
    const int row_lo = j * a.rows_stage;               // CTA-local
    const int nr = min(a.rows_stage, nrows - row_lo);
    if (ok && active) {
      const uint8_t* stage = ring + static_cast<size_t>(s) * a.stage_bytes;
      // two rows per pass where the stage has them (r and r + RG): twice the independent work
      // between the shuffle reductions, whose latency the second row's arithmetic hides
      int r = rg;
      for (; r + a.row_groups < nr; r += 2 * a.row_groups)
        row_pass<M, G, IPL, 2>(a, stage, row_bytes, row_lo, r, part, lane, items, sbox, zbox, poff,
                               prm, xr, sx, sc, ysum);
      if (r < nr)
        row_pass<M, G, IPL, 1>(a, stage, row_bytes, row_lo, r, part, lane, items, sbox, zbox, poff,
                               prm, xr, sx, sc, ysum);
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
