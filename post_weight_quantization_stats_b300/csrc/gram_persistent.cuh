// The whole Gram-schedule search in one persistent, cooperatively launched kernel.
//
// Same arithmetic as tri_kernel (gram_score.cuh), phase by phase: phase 0 forms the scaled
// triangle B of H = X^T X, phase 1 + a scores candidate a through it ("AWQ Math", "Searching the
// scale"). Every CTA walks the same phase sequence with the same roles (warp 0 TMA producer,
// warp 1 MMA issuer, warps 2-5 epilogue, warps 6-15 residual builders) and the same serpentine
// tile deal, so each CTA's fp64 partials are summed in a fixed order, as with one launch per
// phase (a phase's tiles go to its first min(tiles, CTAs) CTAs, the grid of the launch that
// phase would get, so both schedules give the same bits). What one launch per phase got from
// kernel boundaries is done here with counters in
// global memory (zeroed before the launch), each a count of CTAs:
//   res_done[a]    CTAs whose residual warps have written their share of candidate a's
//                  residual (buffer a % 2); the producer waits for all of them before loading
//                  candidate a's tiles.
//   gram_done      CTAs whose epilogue has written its tiles of B; the producer waits for all
//                  before candidate 0's tiles.
//   reads_done[a]  CTAs whose epilogue has finished candidate a (so its MMAs, and the TMA loads
//                  behind them, are done with buffer a % 2); the residual warps wait for all
//                  before writing candidate a + 2's residual into that buffer.
// The producer's tiles of the next phase therefore follow the current phase's without draining
// the pipeline or the TMEM accumulators, and a CTA that finishes its share of one candidate
// early starts on the next. The kernel is launched cooperatively (all CTAs resident), and every
// wait on a counter is bounded like the mbarrier waits: a CTA that gives up raises the device
// status, stops signalling, and the others give up after the same limit.
//
// Memory ordering: writers fence (fence.proxy.async for the TMA readers of B and of the
// residuals, then a gpu-scope fence) before a single thread bumps the counter after a named
// barrier; readers poll with ld.acquire.gpu and the producer fences the async proxy before its
// TMA loads. The epilogue reads the residual with L1-bypassing loads, since a buffer is written
// again while the kernel runs.
#pragma once

#include "gram_score.cuh"

namespace awq {
namespace gram {

struct SearchParams {
  int K, N, n_alpha;
  int gram_tiles, gram_kb;    // phase 0: tiles and k-blocks (Tp / BK)
  int row_tiles, col_tiles;   // scoring phases
  __half* B;                  // [K, K] scaled triangle of H
  const unsigned int* hmax;
  __half* D[2];               // residual buffers
  ResidualArgs res;           // W, absmax, N, K, symmetric (s, inv_s, D set per candidate)
  const float* s_grid;        // [n_alpha, K]
  const float* inv_grid;      // [n_alpha, K]
  double* partial;            // [n_alpha, pstride]
  int pstride;
  unsigned int* sync;         // res_done[n_alpha], reads_done[n_alpha], gram_done
  int* status;
  unsigned long long limit_ns;
};

__device__ __forceinline__ unsigned int ld_acquire_gpu(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Waits until *c >= target; gives up like wait_bounded (abort flag, or limit_ns and then the
// timeout status).
__device__ __forceinline__ bool wait_count(const unsigned int* c, unsigned int target,
                                           const WaitCtx& w) {
  if (ld_acquire_gpu(c) >= target) return true;
  if (w.limit_ns == 0) {  // never waits (see wait_bounded)
    *w.abort_flag = 1;
    atomicCAS(w.status, 0, kStatusTimeout);
    return false;
  }
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    __nanosleep(100);
    if (ld_acquire_gpu(c) >= target) return true;
    if ((it & 7u) == 0u) {
      if (*w.abort_flag) return false;
      if (globaltimer_ns() - t0 > w.limit_ns) {
        *w.abort_flag = 1;
        atomicCAS(w.status, 0, kStatusTimeout);
        return false;
      }
    }
  }
}

template <int G>
__global__ void __launch_bounds__(THREADS, 1)
    search_kernel(const __grid_constant__ CUtensorMap tmXa, const __grid_constant__ CUtensorMap tmXb,
                  const __grid_constant__ CUtensorMap tmD0, const __grid_constant__ CUtensorMap tmD1,
                  const __grid_constant__ CUtensorMap tmB, SearchParams p) {
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
  volatile int* res_ok = abort_flag + 1;
  double* red = reinterpret_cast<double*>(tmem_slot + 4);  // [4]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int P = static_cast<int>(gridDim.x), cta = static_cast<int>(blockIdx.x);
  const unsigned int nP = static_cast<unsigned int>(P);
  const int nph = p.n_alpha + 1;
  unsigned int* res_done = p.sync;
  unsigned int* reads_done = p.sync + p.n_alpha;
  unsigned int* gram_done = p.sync + 2 * p.n_alpha;

  // tile decoding parameters (decode() reads row_tiles, col_tiles, K and num_kb)
  Params dp{};
  dp.row_tiles = p.row_tiles;
  dp.col_tiles = p.col_tiles;
  dp.K = p.K;
  dp.N = p.N;
  dp.num_kb = p.gram_kb;
  const int score_tiles = p.row_tiles * p.col_tiles;

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
    prefetch_tensormap(&tmXa);
    prefetch_tensormap(&tmXb);
    prefetch_tensormap(&tmD0);
    prefetch_tensormap(&tmD1);
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
      for (int ph = 0; ok && ph < nph; ++ph) {
        const int mode = ph == 0 ? GRAM : SCORE;
        const int ntiles = ph == 0 ? p.gram_tiles : score_tiles;
        const int Pd = min(ntiles, P);  // the tiles of a phase are dealt over its first Pd CTAs
        const CUtensorMap* mA = ph == 0 ? &tmXa : (((ph - 1) & 1) ? &tmD1 : &tmD0);
        const CUtensorMap* mB = ph == 0 ? &tmXb : &tmB;
        if (ph >= 1) {
          ok = wait_count(&res_done[ph - 1], nP, wc) && (ph > 1 || wait_count(gram_done, nP, wc));
          if (!ok) break;
          fence_proxy_async_global();
        }
        for (int r = 0; ok; ++r) {
          const int u = snake(r, cta, Pd);
          if (cta >= Pd || u >= ntiles) break;
          const Tile t = decode(dp, u, mode);
          for (int kb = 0; kb < t.nkb; ++kb, ++it) {
            const uint32_t s = it % STAGES, ph2 = (it / STAGES) & 1u;
            if (!wait_bounded(&empty[s], ph2 ^ 1u, wc)) { ok = false; break; }
            mbar_arrive_expect_tx(&full[s], STAGE_BYTES);
            tma_load_2d(sA + s * A_BYTES, mA, &full[s], kb * BK, t.ra * BM);
            tma_load_2d(sB + s * B_BYTES, mB, &full[s], kb * BK, t.rb * BN);
          }
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
      for (int ph = 0; ok && ph < nph; ++ph) {
        const int mode = ph == 0 ? GRAM : SCORE;
        const int ntiles = ph == 0 ? p.gram_tiles : score_tiles;
        const int Pd = min(ntiles, P);  // the tiles of a phase are dealt over its first Pd CTAs
        for (int r = 0; ok; ++r, ++local) {
          const int u = snake(r, cta, Pd);
          if (cta >= Pd || u >= ntiles) break;
          const Tile t = decode(dp, u, mode);
          const uint32_t acc = local & 1u, use = local >> 1;
          if (!wait_bounded(&tempty[acc], (use & 1u) ^ 1u, wc)) { ok = false; break; }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + acc * BN;
          for (int kb = 0; kb < t.nkb; ++kb, ++it) {
            const uint32_t s = it % STAGES, ph2 = (it / STAGES) & 1u;
            if (!wait_bounded(&full[s], ph2, wc)) { ok = false; break; }
            tc_fence_after();
            const uint32_t a0 = smem_u32(sA + s * A_BYTES), b0 = smem_u32(sB + s * B_BYTES);
#pragma unroll
            for (int k = 0; k < BK / 16; ++k)
              mma_f16(d_tmem, sw128_kmajor_desc(a0 + k * 32), sw128_kmajor_desc(b0 + k * 32),
                      idesc, (kb | k) != 0);
            mma_commit(&empty[s]);
          }
          if (!ok) break;
          mma_commit(&tfull[acc]);
        }
      }
      mma_commit(drain);  // every MMA issued above has finished once this arrives
      wait_drain(drain, 0, p.limit_ns);
    }
  } else if (warp >= 6) {
    // residual a is built during phase a (the triangle's phase for a = 0), into buffer a % 2,
    // once every CTA is done reading that buffer for candidate a - 2
    constexpr int TW = RES_WARPS;  // warps per residual block
    const int rw = warp - 6;
    const int chunks = (p.K / 8 + 31) / 32;
    const int items = (p.N + TW * QROWS - 1) / (TW * QROWS) * chunks;
    const float p2 = ldexpf(1.0f, residual_exponent(*p.res.absmax));
    for (int a = 0; a < p.n_alpha; ++a) {
      if (rw == 0 && lane == 0) {
        bool ok = !*abort_flag;
        if (ok && a >= 2) ok = wait_count(&reads_done[a - 2], nP, wc);
        *res_ok = ok ? 1 : 0;
      }
      named_bar_sync(2, 32 * RES_WARPS);
      const bool ok = *res_ok != 0;
      if (ok) {
        ResidualArgs ra = p.res;
        ra.s = p.s_grid + static_cast<size_t>(a) * p.K;
        ra.inv_s = p.inv_grid + static_cast<size_t>(a) * p.K;
        ra.D = p.D[a & 1];
        int item = cta;
        ResidualRegs cur, nxt;
        if (item < items) residual_load(ra, item / chunks, item % chunks, rw, lane, cur, TW);
        for (; item < items; item += P) {
          const int next = item + P;
          if (next < items) residual_load(ra, next / chunks, next % chunks, rw, lane, nxt, TW);
          residual_store<G>(ra, cur, p2);
          if (next < items) cur = nxt;
        }
        fence_proxy_async_global();
        __threadfence();
      }
      named_bar_sync(2, 32 * RES_WARPS);
      if (ok && rw == 0 && lane == 0) {
        __threadfence();
        atomicAdd(&res_done[a], 1u);
      }
    }
  } else {
    const uint32_t q = static_cast<uint32_t>(warp & 3);  // TMEM lane quarter of this warp
    const uint32_t lane_base = tmem_base + ((q * 32u) << 16);
    const float scale = ldexpf(1.f, -gram_exponent(*p.hmax));
    uint32_t local = 0;
    bool ok = true;
    for (int ph = 0; ph < nph; ++ph) {
      const int mode = ph == 0 ? GRAM : SCORE;
      const int ntiles = ph == 0 ? p.gram_tiles : score_tiles;
      const int Pd = min(ntiles, P);
      const __half* Dph = ph == 0 ? nullptr : p.D[(ph - 1) & 1];
      // the residual this phase reads was written by other CTAs: acquire its counter
      if (ok && ph >= 1) ok = wait_count(&res_done[ph - 1], nP, wc);
      double total = 0.0;
      for (int r = 0; ok; ++r, ++local) {
        const int u = snake(r, cta, Pd);
        if (cta >= Pd || u >= ntiles) break;
        const Tile t = decode(dp, u, mode);
        const int row = t.ra * BM + static_cast<int>(q) * 32 + lane;  // SCORE: n, GRAM: k
        const int col0 = t.rb * BN;
        const uint32_t acc = local & 1u, use = local >> 1;
        if (mode == SCORE) {
          const bool rok = row < p.N;
          const __half* drow = Dph + static_cast<long long>(rok ? row : 0) * p.K + col0;
          auto ld = [&](int v) -> uint4 {
            return (rok && col0 + v * 8 < p.K) ? __ldcg(reinterpret_cast<const uint4*>(drow + v * 8))
                                               : make_uint4(0u, 0u, 0u, 0u);
          };
          uint4 dv[8];  // chunks c and c + 2 share a slot: 64 columns in flight
#pragma unroll
          for (int v = 0; v < 8; ++v) dv[v] = ld(v);
          const bool got = wait_bounded(&tfull[acc], use & 1u, wc);
          if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
          tc_fence_after();
          float sum = 0.f;
#pragma unroll
          for (int c = 0; c < BN / 32; ++c) {
            uint32_t e[32];
            tmem_ld_x32(lane_base + acc * BN + c * 32, e);
            tmem_ld_wait();
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const uint4 w = dv[(c & 1) * 4 + v];
              if (c < 6) dv[(c & 1) * 4 + v] = ld((c + 2) * 4 + v);
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
          if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
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
              for (int i = 0; i < 4; ++i)
                dst[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[acc]);
      }
      // end of the phase: publish B (phase 0) or this candidate's partial, then count the CTA
      if (mode == GRAM) fence_proxy_async_global();
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) total += __shfl_xor_sync(0xffffffffu, total, o);
      if (lane == 0) red[warp - 2] = total;
      __threadfence();
      named_bar_sync(1, 128);
      if (warp == 2 && lane == 0) {
        if (ph >= 1) p.partial[static_cast<size_t>(ph - 1) * p.pstride + cta] =
            ((red[0] + red[1]) + red[2]) + red[3];
        if (ok && !*abort_flag) {
          __threadfence();
          atomicAdd(ph == 0 ? gram_done : &reads_done[ph - 1], 1u);
        }
      }
      named_bar_sync(1, 128);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

}  // namespace gram
}  // namespace awq
