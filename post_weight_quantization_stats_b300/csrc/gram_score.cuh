// Output-error scoring through the Gram matrix of the calibration activations.
//
// "AWQ Math", "Searching the scale": the error of one alpha candidate is
//     E = 1/(T N) * sum_{t,n} ( sum_k X[t,k] D[n,k] )^2,   D = W - w_hat.
// For each output n, sum_t (X d_n)_t^2 = d_n^T H d_n with H = X^T X (K x K, symmetric), so
// E = 1/(T N) * sum_n d_n^T H d_n as well (the same number in exact arithmetic). H is formed
// once per layer (a K x K x T contraction); each candidate then costs a product over K x K
// instead of T x K. With H' = the lower triangle of H with its diagonal halved,
// d^T H d = 2 d^T H' d, so only the column blocks j <= k of H' are multiplied: about N K^2
// multiply-adds per candidate against T N K for the direct form.
//
// One persistent tcgen05 kernel (one CTA per SM; warp 0 TMA producer, warp 1 TMEM owner and
// MMA issuer, warps 2-5 epilogue; 128 x 256 fp32 tiles double-buffered in 512 TMEM columns; a
// 4-stage ring of 128 x 64 and 256 x 64 fp16 tiles with 128-byte swizzle), two modes:
//   GRAM   tile (kt, jt) of Xt Xt^T, Xt = X^T zero-padded to Tp tokens, for jt <= kt / 2 (the
//          lower triangle plus the diagonal band the scoring reads). The epilogue writes
//          B[k][j] = fp16(2^-h H[k][j]) for j < k, fp16(2^-h H[k][k] / 2) for j = k and 0 for
//          j > k, with 2^-h a power of two that keeps every entry below 2^14.
//   SCORE  tile (nt, ct) of D B^T over the column blocks j < (ct + 1) 256 (B is zero above
//          its diagonal). The epilogue reads the tile's own D[n][k] and adds
//          sum_k D[n][k] (D B^T)[n][k] into the CTA's fp64 partial.
// SCORE tiles differ in length (the triangle), so tiles are listed longest first and dealt to
// the CTAs in a fixed serpentine order (CTA c takes list positions c, 2P-1-c, 2P+c, ...); each
// CTA's partial sums its tiles in that order, so the result does not depend on timing.
//
// Warps 6-15 build the residual of the NEXT candidate meanwhile (the GRAM launch builds
// candidate 0's, the SCORE launch of candidate i builds candidate i + 1's) into the other of two
// residual buffers: 10-warp residual blocks (quant.cuh) dealt round-robin over the CTAs. The kernel
// boundary orders that residual before its own scoring launch, so no launch waits on another.
#pragma once

#include "awq_device.cuh"
#include "quant.cuh"

namespace awq {
namespace gram {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int RES_WARPS = 10;               // residual warps: one block is RES_WARPS * QROWS rows
constexpr int THREADS = 192 + 32 * RES_WARPS;
constexpr uint32_t TMEM_COLS = 512;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;
constexpr int TOK_BLOCK = 64;  // tokens per transpose block (Tp is a multiple of it)
static_assert(TOK_BLOCK == BK, "one GRAM k-block per token block");

enum Mode { GRAM = 0, SCORE = 1 };

struct Params {
  int num_tiles;
  int row_tiles;              // SCORE: ceil(N / BM)
  int col_tiles;              // SCORE: ceil(K / BN)
  int num_kb;                 // GRAM: Tp / BK
  int K, N;
  const __half* D;            // SCORE: [N, K] scaled residual, read again by the epilogue
  __half* B;                  // GRAM: [K, K] output
  const unsigned int* hmax;   // GRAM: bit pattern of max_k sum_t x_tk^2 (fp32, >= 0)
  double* partial;            // SCORE: [gridDim.x]
  ResidualArgs res;           // the next candidate's residual (when res_on)
  int res_on;
  int* status;
  unsigned long long limit_ns;
};

// Exponent h of the power-of-two scale of H: max_k H[k][k] 2^-h < 2^14, so every entry
// |H[j][k]| <= sqrt(H[j][j] H[k][k]) fits fp16 with room to spare. Bounded below so that 2^-h
// stays a normal fp32 number.
__host__ __device__ inline int gram_exponent(unsigned int hmax_bits) {
  const int biased = static_cast<int>((hmax_bits >> 23) & 0xffu);
  if ((hmax_bits & 0x7fffffffu) == 0u) return 0;
  // hmax = 1.f * 2^(biased - 127) < 2^(biased - 126) for a normal number; a subnormal one is
  // below 2^-126
  const int e = biased == 0 ? -126 : biased - 126;
  const int h = e - 14;
  return h < -100 ? -100 : h;
}

// Tile u of the mode's list: A operand rows [ra * BM, +BM), B operand rows [rb * BN, +BN),
// k-blocks [0, nkb).
struct Tile {
  int ra, rb, nkb;
};

__device__ __forceinline__ Tile decode(const Params& p, int u, int mode) {
  if (mode == SCORE) {
    const int q = u / p.row_tiles;
    const int ct = p.col_tiles - 1 - q;  // longest tiles first
    const int jend = min((ct + 1) * BN, p.K);
    return {u - q * p.row_tiles, ct, (jend + BK - 1) / BK};
  }
  // GRAM: the row tiles 2i and 2i + 1 both take jt = 0..i, and the pairs before i hold
  // i (i + 1) tiles
  int i = static_cast<int>((sqrtf(4.f * static_cast<float>(u) + 1.f) - 1.f) * 0.5f);
  while (i > 0 && i * (i + 1) > u) --i;
  while ((i + 1) * (i + 2) <= u) ++i;
  const int r = u - i * (i + 1);
  return {2 * i + r / (i + 1), r % (i + 1), p.num_kb};
}

// List position of CTA c's r-th tile (serpentine deal over P CTAs).
__device__ __forceinline__ int snake(int r, int c, int P) {
  return r * P + ((r & 1) ? P - 1 - c : c);
}

__device__ __forceinline__ float2 h2f2(uint32_t w) {
  __half2 h;
  memcpy(&h, &w, sizeof(h));
  return __half22float2(h);
}

template <int MODE, int G>
__global__ void __launch_bounds__(THREADS, 1)
    tri_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
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
  const int P = static_cast<int>(gridDim.x), cta = static_cast<int>(blockIdx.x);

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
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
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
      for (int r = 0; ok; ++r) {
        const int u = snake(r, cta, P);
        if (u >= p.num_tiles) break;
        const Tile t = decode(p, u, MODE);
        for (int kb = 0; kb < t.nkb; ++kb, ++it) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
          if (!wait_bounded(&empty[s], ph ^ 1u, wc)) { ok = false; break; }
          mbar_arrive_expect_tx(&full[s], STAGE_BYTES);
          tma_load_2d(sA + s * A_BYTES, &tmA, &full[s], kb * BK, t.ra * BM);
          tma_load_2d(sB + s * B_BYTES, &tmB, &full[s], kb * BK, t.rb * BN);
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
      for (int r = 0; ok; ++r, ++local) {
        const int u = snake(r, cta, P);
        if (u >= p.num_tiles) break;
        const Tile t = decode(p, u, MODE);
        const uint32_t acc = local & 1u, use = local >> 1;
        if (!wait_bounded(&tempty[acc], (use & 1u) ^ 1u, wc)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < t.nkb; ++kb, ++it) {
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
  } else if (warp >= 6) {
    if (p.res_on) {
      // the residual warps take blocks cta, cta + P, ...; the next block's loads are issued
      // before this block's arithmetic
      const int rw = warp - 6;
      const int chunks = (p.res.K / 8 + 31) / 32;
      const int items = (p.res.N + RES_WARPS * QROWS - 1) / (RES_WARPS * QROWS) * chunks;
      const int stride = P;
      const float p2 = ldexpf(1.0f, residual_exponent(*p.res.absmax));
      int item = cta;
      ResidualRegs cur, nxt;
      if (item < items) residual_load(p.res, item / chunks, item % chunks, rw, lane, cur, RES_WARPS);
      for (; item < items; item += stride) {
        const int next = item + stride;
        if (next < items)
          residual_load(p.res, next / chunks, next % chunks, rw, lane, nxt, RES_WARPS);
        residual_store<G>(p.res, cur, p2);
        if (next < items) cur = nxt;
      }
    }
  } else {
    const uint32_t q = static_cast<uint32_t>(warp & 3);  // TMEM lane quarter of this warp
    const uint32_t lane_base = tmem_base + ((q * 32u) << 16);
    double total = 0.0;
    float scale = 1.f;
    if (MODE == GRAM) scale = ldexpf(1.f, -gram_exponent(*p.hmax));
    uint32_t local = 0;
    for (int r = 0;; ++r, ++local) {
      const int u = snake(r, cta, P);
      if (u >= p.num_tiles) break;
      const Tile t = decode(p, u, MODE);
      const int row = t.ra * BM + static_cast<int>(q) * 32 + lane;  // SCORE: n, GRAM: k
      const int col0 = t.rb * BN;
      const uint32_t acc = local & 1u, use = local >> 1;
      if (MODE == SCORE) {
        // this row's D[n][col0 .. col0 + 255] in 32-column chunks; chunks c and c + 4 share a
        // slot, so the first 128 columns are fetched while the tile's MMAs run and chunk c + 4
        // as soon as chunk c is used
        const bool rok = row < p.N;
        const __half* drow = p.D + static_cast<long long>(rok ? row : 0) * p.K + col0;
        auto ld = [&](int v) -> uint4 {
          return (rok && col0 + v * 8 < p.K) ? __ldg(reinterpret_cast<const uint4*>(drow + v * 8))
                                             : make_uint4(0u, 0u, 0u, 0u);
        };
        uint4 dv[16];
#pragma unroll
        for (int v = 0; v < 16; ++v) dv[v] = ld(v);
        const bool got = wait_bounded(&tfull[acc], use & 1u, wc);
        if (!__all_sync(0xffffffffu, got)) break;  // warp-uniform: tcgen05.ld is .sync.aligned
        tc_fence_after();
        float sum = 0.f;
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t e[32];
          tmem_ld_x32(lane_base + acc * BN + c * 32, e);
          tmem_ld_wait();
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const uint4 w = dv[(c & 3) * 4 + v];
            if (c < 4) dv[(c & 3) * 4 + v] = ld((c + 4) * 4 + v);
            const uint32_t wd[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              const float2 f = h2f2(wd[h]);
              sum = fmaf(__uint_as_float(e[v * 8 + 2 * h]), f.x, sum);
              sum = fmaf(__uint_as_float(e[v * 8 + 2 * h + 1]), f.y, sum);
            }
          }
        }
        total += static_cast<double>(sum);
      } else {
        const bool got = wait_bounded(&tfull[acc], use & 1u, wc);
        if (!__all_sync(0xffffffffu, got)) break;
        tc_fence_after();
        const bool rok = row < p.K;
        __half* brow = p.B + static_cast<long long>(rok ? row : 0) * p.K;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t e[32];
          tmem_ld_x32(lane_base + acc * BN + c * 32, e);
          tmem_ld_wait();
          const int j0 = col0 + c * 32;
          if (rok && j0 < p.K) {  // K is a multiple of 64: the 32 columns are all in range
            uint32_t o[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int j = j0 + 2 * i;
              float v0 = __uint_as_float(e[2 * i]) * scale;
              float v1 = __uint_as_float(e[2 * i + 1]) * scale;
              v0 = j < row ? v0 : (j == row ? v0 * 0.5f : 0.f);
              v1 = j + 1 < row ? v1 : (j + 1 == row ? v1 * 0.5f : 0.f);
              const __half2 hv = __floats2half2_rn(v0, v1);
              memcpy(&o[i], &hv, sizeof(uint32_t));
            }
            uint4* dst = reinterpret_cast<uint4*>(brow + j0);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
    }
    if (MODE == SCORE) {
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) total += __shfl_xor_sync(0xffffffffu, total, o);
      if (lane == 0) red[warp - 2] = total;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (MODE == SCORE && threadIdx.x == 0)
    p.partial[blockIdx.x] = ((red[0] + red[1]) + red[2]) + red[3];
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// X [T, K] fp16 (row stride K) -> Xt [K, Tp] fp16 with zero columns t >= T, and
// colsq[tb][k] = sum of x_tk^2 over the 64 tokens of block tb (fp32, fixed order).
// Grid (K / 64, Tp / 64), 256 threads. Thread i reads channels 8 (i % 8) .. + 7 of tokens
// 2 (i / 8) and 2 (i / 8) + 1 (a warp reads eight whole 128-byte row pieces) and keeps them in
// shared memory as token pairs: tw[k][p] holds (x[2p][k], x[2p+1][k]), rows of 33 words, so the
// pair stores conflict at most two-way and the row reads below not at all. Thread i then
// writes tokens 16 (i % 4) .. + 15 of channel i / 4 (a warp writes eight 128-byte row pieces).
__global__ void __launch_bounds__(256) transpose_kernel(const __half* __restrict__ X, int T, int K,
                                                        int Tp, __half* __restrict__ Xt,
                                                        float* __restrict__ colsq) {
  __shared__ uint32_t tw[64][33];
  __shared__ float part[8][64];
  const int k0 = blockIdx.x * 64, t0 = blockIdx.y * TOK_BLOCK;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  {
    const int c8 = tid & 7, q = tid >> 3;
    const int ta = t0 + 2 * q, tb = ta + 1;
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    const uint4 ra = ta < T ? __ldg(reinterpret_cast<const uint4*>(X + static_cast<long long>(ta) * K + k0 + c8 * 8)) : zero;
    const uint4 rb = tb < T ? __ldg(reinterpret_cast<const uint4*>(X + static_cast<long long>(tb) * K + k0 + c8 * 8)) : zero;
    const uint32_t wa[4] = {ra.x, ra.y, ra.z, ra.w}, wb[4] = {rb.x, rb.y, rb.z, rb.w};
    float sq[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      __half2 ha, hb;
      memcpy(&ha, &wa[j], 4);
      memcpy(&hb, &wb[j], 4);
      const __half2 lo = __lows2half2(ha, hb), hi = __highs2half2(ha, hb);  // (a_k, b_k)
      uint32_t ulo, uhi;
      memcpy(&ulo, &lo, 4);
      memcpy(&uhi, &hi, 4);
      tw[c8 * 8 + 2 * j][q] = ulo;
      tw[c8 * 8 + 2 * j + 1][q] = uhi;
      const float2 fa = __half22float2(ha), fb = __half22float2(hb);
      sq[2 * j] = fmaf(fb.x, fb.x, fa.x * fa.x);
      sq[2 * j + 1] = fmaf(fb.y, fb.y, fa.y * fa.y);
    }
    // lanes with the same c8 (xor 8, 16) hold the warp's 8 tokens of these channels
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      sq[j] += __shfl_xor_sync(0xffffffffu, sq[j], 8);
      sq[j] += __shfl_xor_sync(0xffffffffu, sq[j], 16);
    }
    if (lane < 8) {
#pragma unroll
      for (int j = 0; j < 8; ++j) part[warp][c8 * 8 + j] = sq[j];
    }
  }
  __syncthreads();
  {
    const int k = tid >> 2, w4 = tid & 3;
    uint32_t v[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) v[c] = tw[k][w4 * 8 + c];
    uint4* dst = reinterpret_cast<uint4*>(Xt + static_cast<long long>(k0 + k) * Tp + t0 + w4 * 16);
    dst[0] = make_uint4(v[0], v[1], v[2], v[3]);
    dst[1] = make_uint4(v[4], v[5], v[6], v[7]);
  }
  if (tid < 64) {
    float s2 = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) s2 += part[w][tid];
    colsq[static_cast<long long>(blockIdx.y) * K + k0 + tid] = s2;
  }
}

// hmax = max_k sum_tb colsq[tb][k] as fp32 bits (each channel's sum in fixed order; the max of
// non-negative floats is order-free, so atomicMax on the bits is deterministic). hmax must be
// zero on entry. Grid ceil(K / 32), 256 threads: 32 channels x 8 slices of the token blocks.
__global__ void __launch_bounds__(256) colsq_max_kernel(const float* __restrict__ colsq, int nblk,
                                                        int K, unsigned int* hmax) {
  __shared__ float part[8][32];
  const int kl = threadIdx.x & 31, sl = threadIdx.x >> 5;
  const int k = blockIdx.x * 32 + kl;
  float s = 0.f;
  if (k < K) {
#pragma unroll 4
    for (int b = sl; b < nblk; b += 8) s += colsq[static_cast<long long>(b) * K + k];
  }
  part[sl][kl] = s;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) v += part[i][kl];
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (threadIdx.x == 0) atomicMax(hmax, __float_as_uint(v));
  }
}

}  // namespace gram
}  // namespace awq
