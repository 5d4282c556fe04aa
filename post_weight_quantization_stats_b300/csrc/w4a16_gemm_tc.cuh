// W4A16 matmul on the tcgen05 tensor cores: Y [M, N] = X [M, K] (dequant(Q) diag(inv_s))^T.
//
// "AWQ > Benefits and Practical Considerations": unpack the 4-bit integers, apply the group
// scale and zero point and optionally the inverse scale, fused with the matmul so the fp16
// weight matrix is never materialised in HBM. Operand roles are swapped so that 128 weight rows
// fill the MMA M dimension and the (possibly small) token count is the MMA N dimension:
// D[n, t] = sum_k A[n, k] B[t, k].
//
// Two kernels share the pipeline skeleton (TMA producer warp, one MMA-issuing thread, four
// epilogue warps that own the 128 TMEM lanes, eight expander warps that build the A operand).
// The A operand lives in tensor memory: the expanders write it with tcgen05.st (each warp into
// the 32-lane quarter it may access) and tcgen05.mma reads it from there, so shared memory
// carries only the TMA traffic (codes, activations, inv_s) and the small B tile.
//
// grouped_kernel (M <= 16 tokens: decode and small batches; HBM-bound)
//   Moves the group scaling out of the per-weight work. A is the raw nibble expansion: a code q
//   becomes the exact half 1024 + q (low nibbles) or 1024 + 16 q (high nibbles) by one LOP3 per
//   two codes, in the pair order (q0,q4), (q1,q5), (q2,q6), (q3,q7) of each packed word. B
//   holds the activations x~ = fp16(x * inv_s) in the same order, the high-nibble positions
//   divided by 16 (exact unless subnormal), so for one group g, with fp32 accumulation,
//       D_g[n, t] = sum_{k in g} A B = sum_{k in g} q x~ + C[g, t],  C = 1024 sum_k B.
//   Two A rows of every 32-lane TMEM quarter are constants instead of weights: lane 30 is all
//   1024 (its D is C) and lane 31 is (1, 1, 16, 16, ...) in the pair order (its D is
//   S = sum_{k in g} x~), so each epilogue warp reads C and S from its own accumulator lanes by
//   warp shuffle. A tile therefore carries 120 weight rows. Each group accumulates into its own
//   TMEM slot and the epilogue adds
//       y[t, n] += step[n, g] * (D_g[n, t] - C[g, t] - z[n, g] S[g, t]),
//   so the expanders spend no FMA-pipe instruction per weight. TMA brings 256 channels of codes
//   per stage (128 bytes per row, the width at which the box stream reaches HBM speed), the MMA
//   consumes them in 64-channel steps, two CTAs share an SM, and K is split across a cluster of
//   CTAs whose partial sums are added in rank order through distributed shared memory
//   (deterministic, no global scratch).
//
// dequant_kernel (M > 16: prefill batches; tensor-bound)
//   A is the fp16 weight (q - z) * step (* inv_s) in natural channel order; X arrives by TMA in
//   the 128B-swizzled K-major layout. One 128 x BN accumulator per CTA; K split across a
//   cluster as above when the tiles alone do not fill the GPU.
//
// The codes of every stage arrive by TMA (a [N, K/8] uint32 tensor map), so the ring keeps
// several stages of weight reads in flight. Every wait is bounded.
#pragma once

#include <cooperative_groups.h>

#include "awq_device.cuh"

namespace awq {
namespace w4tc {

constexpr int BM = 128;
constexpr int THREADS = 448;   // 14 warps
constexpr int W_PRODUCER = 0, W_MMA = 1, W_EPI0 = 2, W_EXP0 = 6;
constexpr int EXP_THREADS = 256;
constexpr int EXP_WARPS = 8;   // expander barriers count one arrival per warp

struct Args {
  const uint32_t* Q;      // [N, K/8]
  const __half* scales;   // [K/G, N]
  const uint8_t* zeros;   // [K/G, N] (asymmetric only)
  const float* inv_s;     // [K] or nullptr
  __half* Y;              // [M, N]
  int M, N, K;
  int splits;             // CTAs per cluster along K (grid z)
  int* status;
  unsigned long long limit_ns;
};

// ============================================================================ grouped kernel
namespace grouped {

constexpr int BK = 64;                       // channels per MMA stage
constexpr int RK = 256;                      // channels per raw stage (TMA): 128 B of codes per row
constexpr int SUBS = RK / BK;                // MMA stages per raw stage
constexpr int BN = 16;                       // MMA N (tokens, padded)
constexpr int ROWS_Q = 30;                   // weight rows per 32-lane TMEM quarter
constexpr int ROWS = 4 * ROWS_Q;             // weight rows per tile (120)
constexpr int AB_STAGES = 3;                 // A (TMEM) / B (shared memory) stages
constexpr int NACC = 8;                      // TMEM accumulator slots (groups in flight)
constexpr int A_COLS = BK / 2;               // TMEM columns of one A stage (2 fp16 per column)
constexpr int A_COL0 = NACC * BN;            // first TMEM column of the A stages
constexpr uint32_t TMEM_COLS = 256;          // 8 x 16 accumulators + 3 x 32 A columns; 2 CTAs/SM
constexpr int RAW_STAGES = 4;
constexpr int CODES_BYTES = ROWS * RK / 2;   // 15360
constexpr int INV_BYTES = RK * 4;            // 1024
constexpr int B_BYTES = BN * BK * 2;         // 2048: 128B-swizzled K-major B tile

// Raw stage of MT token rows: [codes 120 x 128 B, 128-byte swizzle | x MT x 512 B | inv_s 1 KB],
// 1024-byte units.
__host__ __device__ constexpr int xraw_bytes(int mt) { return mt * RK * 2; }
__host__ __device__ constexpr int raw_bytes(int mt) {
  return (CODES_BYTES + xraw_bytes(mt) + INV_BYTES + 1023) / 1024 * 1024;
}
// Shared memory: [B ring | raw ring | barriers]
__host__ __device__ constexpr int smem_bytes(int mt) {
  return 1024 + AB_STAGES * B_BYTES + RAW_STAGES * raw_bytes(mt) + 512;
}

// x~ for 8 channels (one packed word) of one token in the A pair order, the high-nibble
// positions divided by 16.
__device__ __forceinline__ uint4 permute_x8(const __half* xv, const float* iv, bool has_inv) {
  __half h[8];
#pragma unroll
  for (int e = 0; e < 8; ++e)
    h[e] = has_inv ? __float2half_rn(__fmul_rn(__half2float(xv[e]), iv[e])) : xv[e];
  const __half sixteenth = __float2half_rn(0.0625f);
  __align__(16) __half b[8];
  b[0] = h[0];
  b[1] = h[4];
  b[2] = __hmul(h[1], sixteenth);
  b[3] = __hmul(h[5], sixteenth);
  b[4] = h[2];
  b[5] = h[6];
  b[6] = __hmul(h[3], sixteenth);
  b[7] = __hmul(h[7], sixteenth);
  return *reinterpret_cast<const uint4*>(b);
}

template <int G, int MT>
__global__ void __launch_bounds__(THREADS, 2)
    grouped_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmX,
                   Args a) {
  namespace cg = cooperative_groups;
  constexpr int SPG = G / BK;           // MMA stages per group
  constexpr int PD = MT >= 16 ? 4 : 8;  // epilogue prefetch distance (groups)
  constexpr int RAW_BYTES = raw_bytes(MT);
  constexpr int XRAW_OFF = CODES_BYTES, INV_OFF = CODES_BYTES + xraw_bytes(MT);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* bring = smem;                             // B tiles
  uint8_t* raw = bring + AB_STAGES * B_BYTES;
  uint64_t* full_raw = reinterpret_cast<uint64_t*>(raw + RAW_STAGES * RAW_BYTES);
  uint64_t* empty_raw = full_raw + RAW_STAGES;
  uint64_t* full_ab = empty_raw + RAW_STAGES;
  uint64_t* empty_ab = full_ab + AB_STAGES;
  uint64_t* tfull = empty_ab + AB_STAGES;
  uint64_t* tempty = tfull + NACC;
  uint64_t* drain = tempty + NACC;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  cg::cluster_group cluster = cg::this_cluster();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * ROWS;
  const int rank = static_cast<int>(cluster.block_rank());
  // K is split in whole raw stages (256 channels, a whole number of groups)
  const int nraw_all = (a.K + RK - 1) / RK;
  const int r_lo = static_cast<int>(static_cast<long long>(nraw_all) * rank / a.splits);
  const int r_hi = static_cast<int>(static_cast<long long>(nraw_all) * (rank + 1) / a.splits);
  const int k_lo = r_lo * RK, k_hi = min(a.K, r_hi * RK);
  const int g_lo = k_lo / G;
  const int ngr = (k_hi - k_lo) / G;     // groups of this CTA
  const int nst = (k_hi - k_lo) / BK;    // MMA stages of this CTA
  const int nraw = r_hi - r_lo;          // raw stages of this CTA
  const int Mt = a.M;                    // tokens (<= MT <= BN)

  if (threadIdx.x == 0) {
    for (int s = 0; s < RAW_STAGES; ++s) {
      mbar_init(&full_raw[s], 1);
      mbar_init(&empty_raw[s], EXP_WARPS);
    }
    for (int s = 0; s < AB_STAGES; ++s) {
      mbar_init(&full_ab[s], EXP_WARPS);
      mbar_init(&empty_ab[s], 1);
    }
    for (int s = 0; s < NACC; ++s) {
      mbar_init(&tfull[s], 1);
      mbar_init(&tempty[s], 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tensormap(&tmQ);
    prefetch_tensormap(&tmX);
  }
  if (warp == W_MMA) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  if (warp >= W_EXP0) {
    // the padded token rows of every B tile stay zero for the whole kernel
    const int et = threadIdx.x - W_EXP0 * 32;
    for (int i = et; i < AB_STAGES * BN * 8; i += EXP_THREADS) {
      const int s = i / (BN * 8), t = (i / 8) % BN, c = i % 8;
      if (t >= Mt)
        *reinterpret_cast<uint4*>(bring + s * B_BYTES + sw128_offset(t, c)) = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const WaitCtx wc{a.limit_ns, abort_flag, a.status};
  float y[MT];   // epilogue: partial outputs of this thread's row (MT >= M tokens)

  if (warp == W_PRODUCER) {
    // ---------------------------------------------------------------- TMA: codes, X, inv_s
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      int j = 0;
      bool ok = true;
      for (; j < nraw; ++j) {
        const int s = j % RAW_STAGES;
        if (!wait_bounded(&empty_raw[s], ((j / RAW_STAGES) & 1u) ^ 1u, wc)) { ok = false; break; }
        const int k0 = k_lo + j * RK;
        const uint32_t inv_bytes = static_cast<uint32_t>(min(RK, k_hi - k0)) * 4u;
        uint8_t* st = raw + s * RAW_BYTES;
        mbar_arrive_expect_tx(&full_raw[s], CODES_BYTES + xraw_bytes(MT) + (a.inv_s ? inv_bytes : 0u));
        tma_load_2d_hint(st, &tmQ, &full_raw[s], k0 / 8, n0, pol);
        tma_load_2d(st + XRAW_OFF, &tmX, &full_raw[s], k0, 0);
        if (a.inv_s) bulk_load_plain(st + INV_OFF, a.inv_s + k0, inv_bytes, &full_raw[s]);
      }
      {  // let the copies issued last land before the CTA exits (at once unless it gave up)
        for (int jj = (j > RAW_STAGES ? j - RAW_STAGES : 0); jj < j; ++jj)
          wait_drain(&full_raw[jj % RAW_STAGES], (jj / RAW_STAGES) & 1u, a.limit_ns);
      }
    }
  } else if (warp == W_MMA) {
    // ---------------------------------------------------------------- MMA issue
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16_f32(BM, BN);
      bool ok = true;
      for (int j = 0; ok && j < nst; ++j) {
        const int sab = j % AB_STAGES;
        const int gl = j / SPG, slot = gl % NACC;
        const bool first = (j % SPG) == 0, last = (j % SPG) == SPG - 1;
        if (first && !wait_bounded(&tempty[slot], ((gl / NACC) & 1u) ^ 1u, wc)) { ok = false; break; }
        if (!wait_bounded(&full_ab[sab], (j / AB_STAGES) & 1u, wc)) { ok = false; break; }
        tc_fence_after();
        const uint32_t a0 = tmem_base + static_cast<uint32_t>(A_COL0 + sab * A_COLS);
        const uint32_t b0 = smem_u32(bring + sab * B_BYTES);
        const uint32_t d = tmem_base + static_cast<uint32_t>(slot * BN);
#pragma unroll
        for (int k = 0; k < BK / 16; ++k)
          mma_f16_ts(d, a0 + k * 8, sw128_kmajor_desc(b0 + k * 32), idesc,
                     (first && k == 0) ? 0u : 1u);
        mma_commit(&empty_ab[sab]);
        if (last) mma_commit(&tfull[slot]);
      }
      mma_commit(drain);
      wait_drain(drain, 0, a.limit_ns);
    }
  } else if (warp >= W_EXP0) {
    // ---------------------------------------------------------------- expanders
    // Warp w writes TMEM lanes 32 (w % 4) .. + 31 (the lane quarter it may access): A row
    // r = 32 (w % 4) + lane, channels 32 h .. 32 h + 31 of each 64-channel stage.
    const int et = threadIdx.x - W_EXP0 * 32;
    const int quarter = warp & 3, h = (warp - W_EXP0) >> 2;
    const bool weight_row = lane < ROWS_Q;
    const int crow = quarter * ROWS_Q + lane;       // row of the codes box (128 B per row)
    const uint32_t a_lane = static_cast<uint32_t>(quarter * 32) << 16;
    const int bt = et >> 3, bw = et & 7;            // B item: token, word (first 128 threads)
    bool ok = true;
    for (int i = 0; i < nraw; ++i) {
      const int s = i % RAW_STAGES;
      if (ok) ok = wait_bounded(&full_raw[s], (i / RAW_STAGES) & 1u, wc);
      ok = __all_sync(0xffffffffu, ok);   // warp-uniform: one lane arrives for the warp
      const uint8_t* st = raw + s * RAW_BYTES;
      const int nsub = min(SUBS, nst - i * SUBS);
      for (int sub = 0; sub < nsub; ++sub) {
        const int j = i * SUBS + sub, sab = j % AB_STAGES;
        if (ok) ok = wait_bounded(&empty_ab[sab], ((j / AB_STAGES) & 1u) ^ 1u, wc);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        uint32_t av[16];
        if (weight_row) {
          // 16-byte chunk c of a 128-byte code row sits at chunk c ^ (row & 7) (TMA 128B swizzle)
          const uint4 qv = *reinterpret_cast<const uint4*>(
              st + crow * (RK / 2) + (((sub * 2 + h) ^ (crow & 7)) << 4));
          const uint32_t wq[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint32_t w = wq[e], w8 = wq[e] >> 8;
            av[4 * e + 0] = lop3_and_or(w, 0x000F000Fu, 0x64006400u);    // 1024 + q0 | 1024 + q4
            av[4 * e + 1] = lop3_and_or(w, 0x00F000F0u, 0x64006400u);    // 1024 + 16 q1 | 1024 + 16 q5
            av[4 * e + 2] = lop3_and_or(w8, 0x000F000Fu, 0x64006400u);   // 1024 + q2 | 1024 + q6
            av[4 * e + 3] = lop3_and_or(w8, 0x00F000F0u, 0x64006400u);   // 1024 + 16 q3 | 1024 + 16 q7
          }
        } else {
          // lane 30: all 1024 (its accumulator is C); lane 31: (1, 1, 16, 16) (its accumulator is S)
#pragma unroll
          for (int e = 0; e < 16; ++e)
            av[e] = lane == 30 ? 0x64006400u : ((e & 1) ? 0x4C004C00u : 0x3C003C00u);
        }
        tmem_st_x16(tmem_base + a_lane + static_cast<uint32_t>(A_COL0 + sab * A_COLS + h * 16), av);
        if (et < 8 * MT && bt < Mt) {   // B item: token bt, word bw of this 64-channel stage
          const __half* xv = reinterpret_cast<const __half*>(st + XRAW_OFF + bt * (RK * 2) + sub * (BK * 2) + bw * 16);
          const float* iv = reinterpret_cast<const float*>(st + INV_OFF + sub * (BK * 4) + bw * 32);
          *reinterpret_cast<uint4*>(bring + sab * B_BYTES + sw128_offset(bt, bw)) =
              permute_x8(xv, iv, a.inv_s != nullptr);
        }
        tmem_st_wait();
        fence_proxy_async_smem();   // B tile writes -> visible to the tensor core
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&full_ab[sab]);
      }
      __syncwarp();
      if (ok && lane == 0) mbar_arrive(&empty_raw[s]);
    }
  } else {
    // ---------------------------------------------------------------- epilogue (warps 2-5)
    const uint32_t q = static_cast<uint32_t>(warp & 3);        // TMEM lane quarter
    const int n = n0 + static_cast<int>(q) * ROWS_Q + lane;
    const bool row_ok = lane < ROWS_Q && n < a.N;
#pragma unroll
    for (int t = 0; t < MT; ++t) y[t] = 0.f;
    // group parameters PD groups ahead, kept as loaded (fp16 step, uint8 zero point) so the
    // loads stay in flight until the group is reached
    __half pst[PD];
    uint8_t pz[PD];
#pragma unroll
    for (int u = 0; u < PD; ++u) {
      pst[u] = __float2half_rn(0.f);
      pz[u] = 8;
      if (row_ok && u < ngr) {
        const long long gi = static_cast<long long>(g_lo + u) * a.N + n;
        pst[u] = a.scales[gi];
        if (a.zeros) pz[u] = a.zeros[gi];
      }
    }
    bool ok = true;
    for (int gl0 = 0; gl0 < ngr; gl0 += PD) {
#pragma unroll
      for (int u = 0; u < PD; ++u) {
        const int gl = gl0 + u;
        if (gl < ngr) {
          const int slot = gl % NACC;
          if (ok) ok = wait_bounded(&tfull[slot], (gl / NACC) & 1u, wc);
          ok = __all_sync(0xffffffffu, ok);
          if (ok) {
            tc_fence_after();
            const uint32_t taddr = tmem_base + ((q * 32u) << 16) + static_cast<uint32_t>(slot * BN);
            float d[MT];
            if constexpr (MT == 1) {
              d[0] = __uint_as_float(tmem_ld_x1(taddr));
              tmem_ld_wait();
            } else {
              uint32_t v[MT];
              tmem_ld_n(taddr, v);
              tmem_ld_wait();
#pragma unroll
              for (int t = 0; t < MT; ++t) d[t] = __uint_as_float(v[t]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[slot]);
            const float step = __half2float(pst[u]), z = static_cast<float>(pz[u]);
#pragma unroll
            for (int t = 0; t < MT; ++t) {
              const float C = __shfl_sync(0xffffffffu, d[t], 30);
              const float S = __shfl_sync(0xffffffffu, d[t], 31);
              y[t] = fmaf(step, fmaf(-z, S, d[t] - C), y[t]);
            }
          }
          // prefetch the parameters of group gl + PD into this register slot
          if (row_ok && gl + PD < ngr) {
            const long long gi = static_cast<long long>(g_lo + gl + PD) * a.N + n;
            pst[u] = a.scales[gi];
            if (a.zeros) pz[u] = a.zeros[gi];
          }
        }
      }
    }
  }

  // ------------------------------------------------------------------ split-K reduction, Y
  tc_fence_before();
  __syncthreads();
  const bool epi = warp >= W_EPI0 && warp < W_EPI0 + 4;
  const int q = warp & 3;
  const int n = n0 + q * ROWS_Q + lane;
  const bool out_row = epi && lane < ROWS_Q && n < a.N && !*abort_flag;
  float* red = reinterpret_cast<float*>(raw);   // [t][128 A rows]; every ring is idle now
  if (a.splits > 1) {
    if (epi) {
#pragma unroll
      for (int t = 0; t < MT; ++t) red[t * BM + q * 32 + lane] = y[t];
    }
    cluster.sync();
    // rank p adds up tokens p, p + splits, ... of every row, reading all ranks in rank order
    if (out_row) {
      for (int t = rank; t < Mt; t += a.splits) {
        float v[8];
#pragma unroll
        for (int p = 0; p < 8; ++p)
          v[p] = p < a.splits ? cluster.map_shared_rank(red, p)[t * BM + q * 32 + lane] : 0.f;
        float sum = 0.f;
#pragma unroll
        for (int p = 0; p < 8; ++p) sum += v[p];
        a.Y[static_cast<long long>(t) * a.N + n] = __float2half_rn(sum);
      }
    }
    cluster.sync();
  } else if (out_row) {
#pragma unroll
    for (int t = 0; t < MT; ++t)
      if (t < Mt) a.Y[static_cast<long long>(t) * a.N + n] = __float2half_rn(y[t]);
  }
  if (warp == W_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

}  // namespace grouped

// ============================================================================ dequant kernel
namespace dequant {

constexpr int BK = 128;
constexpr int CODES_BYTES = BM * BK / 2;   // 8192
constexpr int INV_BYTES = BK * 4;          // 512
constexpr int AB_STAGES = 4;               // A stages in TMEM
constexpr int A_COLS = BK / 2;             // TMEM columns of one A stage (2 fp16 per column)

template <int BN>
struct Cfg {
  static constexpr int B_SUB = BN * 128;
  static constexpr int B_BYTES = 2 * B_SUB;
  static constexpr int RAW_BYTES = (B_BYTES + CODES_BYTES + INV_BYTES + 1023) / 1024 * 1024;
  static constexpr int RAW_STAGES = (220 * 1024 / RAW_BYTES) > 8 ? 8 : (220 * 1024 / RAW_BYTES);
  static constexpr int SMEM = 1024 + RAW_STAGES * RAW_BYTES + 512;
  static constexpr int A_COL0 = BN;        // A stages follow the accumulator
  static constexpr uint32_t TMEM_COLS = (BN + AB_STAGES * A_COLS) <= 256 ? 256u : 512u;
  static constexpr int RED_LD = BN + 4;    // floats per row of the split-K exchange buffer
};

// 8 codes (channels 8w..8w+7 in natural order) -> 8 fp16 (q - z) * step in natural order.
__device__ __forceinline__ uint4 dequant8_f16(uint32_t w, __half2 zlo, __half2 zhi, __half2 st2) {
  const uint32_t t0 = lop3_and_or(w, 0x000F000Fu, 0x64006400u);   // q0 | q4
  const uint32_t t1 = lop3_and_or(w, 0x00F000F0u, 0x64006400u);   // 16 q1 | 16 q5
  const uint32_t w8 = w >> 8;
  const uint32_t t2 = lop3_and_or(w8, 0x000F000Fu, 0x64006400u);  // q2 | q6
  const uint32_t t3 = lop3_and_or(w8, 0x00F000F0u, 0x64006400u);  // 16 q3 | 16 q7
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

// Same times the per-channel inverse scale, in half precision: the fp16 weight (q - z) * step
// times fp16(inv_s_k) (two roundings of 2^-11 relative each).
__device__ __forceinline__ uint4 dequant8_inv(uint32_t w, __half2 zlo, __half2 zhi, __half2 st2,
                                             const float* inv) {
  uint4 out = dequant8_f16(w, zlo, zhi, st2);
  const float4 ia = *reinterpret_cast<const float4*>(inv);
  const float4 ib = *reinterpret_cast<const float4*>(inv + 4);
  __half2* o = reinterpret_cast<__half2*>(&out);
  o[0] = __hmul2(o[0], __floats2half2_rn(ia.x, ia.y));
  o[1] = __hmul2(o[1], __floats2half2_rn(ia.z, ia.w));
  o[2] = __hmul2(o[2], __floats2half2_rn(ib.x, ib.y));
  o[3] = __hmul2(o[3], __floats2half2_rn(ib.z, ib.w));
  return out;
}

template <int BN, int G>
__global__ void __launch_bounds__(THREADS, 1)
    dequant_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmX,
                   Args a) {
  namespace cg = cooperative_groups;
  using C = Cfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* raw = smem;                                  // [B tile | codes | inv_s] per stage
  uint64_t* full_raw = reinterpret_cast<uint64_t*>(raw + C::RAW_STAGES * C::RAW_BYTES);
  uint64_t* empty_raw = full_raw + C::RAW_STAGES;
  uint64_t* full_ab = empty_raw + C::RAW_STAGES;
  uint64_t* empty_ab = full_ab + AB_STAGES;
  uint64_t* tfull = empty_ab + AB_STAGES;
  uint64_t* drain = tfull + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  cg::cluster_group cluster = cg::this_cluster();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * BM, m0 = blockIdx.y * BN;
  const int rank = static_cast<int>(cluster.block_rank());
  const int nkb = (a.K + BK - 1) / BK;
  const int kb_lo = static_cast<int>(static_cast<long long>(nkb) * rank / a.splits);
  const int kb_hi = static_cast<int>(static_cast<long long>(nkb) * (rank + 1) / a.splits);
  const int nst = kb_hi - kb_lo;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::RAW_STAGES; ++s) {
      mbar_init(&full_raw[s], 1);
      mbar_init(&empty_raw[s], 1);
    }
    for (int s = 0; s < AB_STAGES; ++s) {
      mbar_init(&full_ab[s], EXP_WARPS);
      mbar_init(&empty_ab[s], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tensormap(&tmQ);
    prefetch_tensormap(&tmX);
  }
  if (warp == W_MMA) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const WaitCtx wc{a.limit_ns, abort_flag, a.status};
  bool epi_ok = true;

  if (warp == W_PRODUCER) {
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      int j = 0;
      bool ok = true;
      for (; j < nst; ++j) {
        const int s = j % C::RAW_STAGES;
        if (!wait_bounded(&empty_raw[s], ((j / C::RAW_STAGES) & 1u) ^ 1u, wc)) { ok = false; break; }
        const int k0 = (kb_lo + j) * BK;
        const int klen = min(BK, a.K - k0);
        uint8_t* st = raw + s * C::RAW_BYTES;
        mbar_arrive_expect_tx(&full_raw[s], C::B_BYTES + CODES_BYTES +
                                                (a.inv_s ? static_cast<uint32_t>(klen) * 4u : 0u));
        tma_load_2d(st, &tmX, &full_raw[s], k0, m0);
        tma_load_2d(st + C::B_SUB, &tmX, &full_raw[s], k0 + 64, m0);
        tma_load_2d_hint(st + C::B_BYTES, &tmQ, &full_raw[s], k0 / 8, n0, pol);
        if (a.inv_s)
          bulk_load_plain(st + C::B_BYTES + CODES_BYTES, a.inv_s + k0,
                          static_cast<uint32_t>(klen) * 4u, &full_raw[s]);
      }
      {  // let the copies issued last land before the CTA exits (at once unless it gave up)
        for (int jj = (j > C::RAW_STAGES ? j - C::RAW_STAGES : 0); jj < j; ++jj)
          wait_drain(&full_raw[jj % C::RAW_STAGES], (jj / C::RAW_STAGES) & 1u, a.limit_ns);
      }
    }
  } else if (warp == W_MMA) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16_f32(BM, BN);
      bool ok = true;
      for (int j = 0; ok && j < nst; ++j) {
        const int s = j % C::RAW_STAGES, sab = j % AB_STAGES;
        if (!wait_bounded(&full_raw[s], (j / C::RAW_STAGES) & 1u, wc) ||
            !wait_bounded(&full_ab[sab], (j / AB_STAGES) & 1u, wc)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = tmem_base + static_cast<uint32_t>(C::A_COL0 + sab * A_COLS);
        const uint32_t b0 = smem_u32(raw + s * C::RAW_BYTES);
#pragma unroll
        for (int sub = 0; sub < 2; ++sub)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_f16_ts(tmem_base, a0 + sub * 32 + k * 8,
                       sw128_kmajor_desc(b0 + sub * C::B_SUB + k * 32), idesc,
                       (j | sub | k) != 0 ? 1u : 0u);
        mma_commit(&empty_ab[sab]);
        mma_commit(&empty_raw[s]);
      }
      if (ok) mma_commit(tfull);
      mma_commit(drain);
      wait_drain(drain, 0, a.limit_ns);
    }
  } else if (warp >= W_EXP0) {
    // expander thread: A row r = 32 (w % 4) + lane (the TMEM lane quarter warp w may access),
    // channels 64 h .. 64 h + 63 of each stage
    const int quarter = warp & 3, h = (warp - W_EXP0) >> 2;
    const int r = quarter * 32 + lane;
    const uint32_t a_lane = static_cast<uint32_t>(quarter * 32) << 16;
    const int row = n0 + r;
    const bool row_ok = row < a.N;
    bool ok = true;
    // group parameters of stage j, loaded PD stages ahead and kept as loaded (fp16, uint8)
    // until used, so the loads stay in flight; a 64-channel half holds one group, or two when
    // G = 32 (NG sets per stage)
    constexpr int PD = 4;
    constexpr int NG = G >= 64 ? 1 : 64 / G;
    auto load_params = [&](int j, __half (&st)[NG], uint8_t (&z)[NG]) {
      const int k = (kb_lo + j) * BK + h * 64;
#pragma unroll
      for (int g = 0; g < NG; ++g) {
        if (row_ok && j < nst && k + g * G < a.K) {
          const long long gi = static_cast<long long>((k + g * G) / G) * a.N + row;
          st[g] = a.scales[gi];
          if (a.zeros) z[g] = a.zeros[gi];
        }
      }
    };
    __half pst[PD][NG];
    uint8_t pz[PD][NG];
#pragma unroll
    for (int u = 0; u < PD; ++u) {
#pragma unroll
      for (int g = 0; g < NG; ++g) {
        pst[u][g] = __float2half_rn(0.f);
        pz[u][g] = 8;
      }
      load_params(u, pst[u], pz[u]);
    }
    for (int j0 = 0; j0 < nst; j0 += PD) {
#pragma unroll
    for (int u = 0; u < PD; ++u) {
      const int j = j0 + u;
      if (j >= nst) break;
      float st_cur[NG], z_cur[NG];
#pragma unroll
      for (int g = 0; g < NG; ++g) {
        st_cur[g] = __half2float(pst[u][g]);
        z_cur[g] = static_cast<float>(pz[u][g]);
      }
      load_params(j + PD, pst[u], pz[u]);
      const int s = j % C::RAW_STAGES, sab = j % AB_STAGES;
      if (ok) ok = wait_bounded(&full_raw[s], (j / C::RAW_STAGES) & 1u, wc);
      if (ok) ok = wait_bounded(&empty_ab[sab], ((j / AB_STAGES) & 1u) ^ 1u, wc);
      ok = __all_sync(0xffffffffu, ok);   // warp-uniform: one lane arrives for the warp
      if (ok) {
        tc_fence_after();
        const int kbase = (kb_lo + j) * BK + h * 64;
        const uint8_t* st = raw + s * C::RAW_BYTES;
        const bool live = row_ok && kbase < a.K;
        uint32_t av[32];
        if (!live) {
#pragma unroll
          for (int c = 0; c < 32; ++c) av[c] = 0u;
        } else {
          const uint4 q0 = *reinterpret_cast<const uint4*>(st + C::B_BYTES + r * 64 + h * 32);
          const uint4 q1 = *reinterpret_cast<const uint4*>(st + C::B_BYTES + r * 64 + h * 32 + 16);
          const uint32_t wq[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
          const float* inv = reinterpret_cast<const float*>(st + C::B_BYTES + CODES_BYTES) + h * 64;
          auto expand = [&](int c) -> uint4 {
            const int g = (c * 8) / (64 / NG);   // the group of word c (8 channels)
            const __half2 zlo = __float2half2_rn(-(1024.f + z_cur[g]));
            const __half2 zhi = __float2half2_rn(-(64.f + z_cur[g]));
            const __half2 st2 = __float2half2_rn(st_cur[g]);
            return a.inv_s ? dequant8_inv(wq[c], zlo, zhi, st2, inv + 8 * c)
                           : dequant8_f16(wq[c], zlo, zhi, st2);
          };
          if (kbase + 64 <= a.K) {
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const uint4 v = expand(c);
              av[4 * c + 0] = v.x;
              av[4 * c + 1] = v.y;
              av[4 * c + 2] = v.z;
              av[4 * c + 3] = v.w;
            }
          } else {
            // the half reaches past K (K % 128 == 32 or 96, G = 32): the codes and inv_s slots
            // of channels past K hold fill or stale data, so their weights are zeroed
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const uint4 v = kbase + 8 * c < a.K ? expand(c) : make_uint4(0u, 0u, 0u, 0u);
              av[4 * c + 0] = v.x;
              av[4 * c + 1] = v.y;
              av[4 * c + 2] = v.z;
              av[4 * c + 3] = v.w;
            }
          }
        }
        tmem_st_x32(tmem_base + a_lane + static_cast<uint32_t>(C::A_COL0 + sab * A_COLS + h * 32), av);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&full_ab[sab]);
      }
    }
    }
  } else {
    // epilogue warps 2-5 wait for the accumulator
    if (epi_ok) epi_ok = wait_bounded(tfull, 0, wc);
    epi_ok = __all_sync(0xffffffffu, epi_ok);
  }

  // ------------------------------------------------------------------ epilogue, split-K, Y
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const bool epi = warp >= W_EPI0 && warp < W_EPI0 + 4;
  const uint32_t q = static_cast<uint32_t>(warp & 3);
  const int r = static_cast<int>(q) * 32 + lane;
  const int n = n0 + r;
  float* red = reinterpret_cast<float*>(smem);   // [128 rows][RED_LD]; every ring is idle now
  const bool good = epi && epi_ok && !*abort_flag;
  if (a.splits > 1) {
    if (good) {
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t v[32];
        tmem_ld_x32(tmem_base + ((q * 32u) << 16) + c * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; j += 4)
          *reinterpret_cast<float4*>(red + r * C::RED_LD + c * 32 + j) =
              make_float4(__uint_as_float(v[j]), __uint_as_float(v[j + 1]),
                          __uint_as_float(v[j + 2]), __uint_as_float(v[j + 3]));
      }
    }
    cluster.sync();
    // rank p adds up its slice of the tile's tokens (a multiple of 4 wide), reading every rank
    // in rank order
    const int per = ((BN + a.splits - 1) / a.splits + 3) / 4 * 4;
    const int t_lo = min(BN, rank * per);
    const int t_hi = min(min(BN, t_lo + per), ((a.M - m0) + 3) / 4 * 4);
    if (good && n < a.N) {
      for (int t = t_lo; t < t_hi; t += 4) {
        float4 v[8];
#pragma unroll
        for (int p = 0; p < 8; ++p)
          if (p < a.splits)
            v[p] = *reinterpret_cast<const float4*>(cluster.map_shared_rank(red, p) + r * C::RED_LD + t);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int p = 0; p < 8; ++p)
          if (p < a.splits) {
            acc.x += v[p].x;
            acc.y += v[p].y;
            acc.z += v[p].z;
            acc.w += v[p].w;
          }
        const float o4[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (m0 + t + e < a.M) a.Y[static_cast<long long>(m0 + t + e) * a.N + n] = __float2half_rn(o4[e]);
      }
    }
    cluster.sync();
  } else if (good) {
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      uint32_t v[32];
      tmem_ld_x32(tmem_base + ((q * 32u) << 16) + c * 32, v);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int t = m0 + c * 32 + j;
        if (t < a.M && n < a.N) a.Y[static_cast<long long>(t) * a.N + n] = __float2half_rn(__uint_as_float(v[j]));
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == W_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

}  // namespace dequant
}  // namespace w4tc
}  // namespace awq
