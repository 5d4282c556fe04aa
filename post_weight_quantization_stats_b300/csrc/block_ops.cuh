// Folding the inverse scale into the previous operation, and the two elementwise operations a
// synthetic MLP block needs around its linears.
//
// "AWQ Math", "The equivalent transform": with W' = W diag(s) the layer computes the same
// output from x' = diag(s)^-1 x, so 1/s can be folded into whatever produces x (a norm's weight
// or the previous linear's output rows) and the quantised layer runs with inv_s = NULL.
// "AWQ > Benefits and Practical Considerations": the scale folds into the previous layer.
//
// scale_rows_kernel   A[r][c] = fp16(fl32(A[r][c] * row_scale[r])) in place.
// rmsnorm_kernel      Y[t][j] = fp16(X[t][j] * r_t * gamma[j]), r_t = 1 / sqrt(mean_j X[t][j]^2 +
//                     eps), fp32 arithmetic, the sum of squares in a fixed order.
// silu_mul_kernel     H = fp16(silu(G) * U) with silu(g) = g / (1 + e^-g), fp32 arithmetic.
#pragma once

#include "awq_device.cuh"

namespace awq {
namespace block {

// Grid-stride over rows x cols; 8 columns per thread when every row starts 16-byte aligned.
__global__ void __launch_bounds__(256) scale_rows_kernel(__half* __restrict__ A, long long rows,
                                                         long long cols, long long lda,
                                                         const float* __restrict__ row_scale,
                                                         int vec8) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  const long long start = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (vec8) {
    const long long cw = cols / 8;
    for (long long i = start; i < rows * cw; i += stride) {
      const long long r = i / cw, c = (i - r * cw) * 8;
      uint4* p = reinterpret_cast<uint4*>(A + r * lda + c);
      const float sc = row_scale[r];
      uint4 v = *p;
      uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        __half2 h;
        memcpy(&h, &w[j], 4);
        const float2 f = __half22float2(h);
        h = __floats2half2_rn(__fmul_rn(f.x, sc), __fmul_rn(f.y, sc));
        memcpy(&w[j], &h, 4);
      }
      *p = make_uint4(w[0], w[1], w[2], w[3]);
    }
  } else {
    for (long long i = start; i < rows * cols; i += stride) {
      const long long r = i / cols, c = i - r * cols;
      __half* p = A + r * lda + c;
      *p = __float2half_rn(__fmul_rn(__half2float(*p), row_scale[r]));
    }
  }
}

// One CTA of 256 threads per token; D % 8 == 0. Thread i sums squares of the 8-channel words
// i, i + 256, ... in order; the 256 sums are combined by a fixed tree.
__global__ void __launch_bounds__(256) rmsnorm_kernel(const __half* __restrict__ X, int D,
                                                      const __half* __restrict__ gamma,
                                                      float eps, __half* __restrict__ Y) {
  __shared__ float part[256];
  const long long t = blockIdx.x;
  const __half* x = X + t * D;
  __half* y = Y + t * D;
  const int words = D / 8;
  float ss = 0.f;
  for (int w = threadIdx.x; w < words; w += 256) {
    const uint4 v = *reinterpret_cast<const uint4*>(x + w * 8);
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      __half2 h;
      memcpy(&h, &u[j], 4);
      const float2 f = __half22float2(h);
      ss = fmaf(f.x, f.x, ss);
      ss = fmaf(f.y, f.y, ss);
    }
  }
  part[threadIdx.x] = ss;
  __syncthreads();
  for (int o = 128; o >= 1; o >>= 1) {
    if (threadIdx.x < o) part[threadIdx.x] += part[threadIdx.x + o];
    __syncthreads();
  }
  const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(part[0], static_cast<float>(D)), eps)));
  for (int w = threadIdx.x; w < words; w += 256) {
    const uint4 v = *reinterpret_cast<const uint4*>(x + w * 8);
    const uint4 g = *reinterpret_cast<const uint4*>(gamma + w * 8);
    const uint32_t u[4] = {v.x, v.y, v.z, v.w}, gu[4] = {g.x, g.y, g.z, g.w};
    uint32_t o4[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      __half2 h, hg;
      memcpy(&h, &u[j], 4);
      memcpy(&hg, &gu[j], 4);
      const float2 f = __half22float2(h), fg = __half22float2(hg);
      const __half2 out = __floats2half2_rn(__fmul_rn(__fmul_rn(f.x, r), fg.x),
                                            __fmul_rn(__fmul_rn(f.y, r), fg.y));
      memcpy(&o4[j], &out, 4);
    }
    *reinterpret_cast<uint4*>(y + w * 8) = make_uint4(o4[0], o4[1], o4[2], o4[3]);
  }
}

// n % 8 == 0; grid-stride over 8-element words.
__global__ void __launch_bounds__(256) silu_mul_kernel(const __half* __restrict__ G,
                                                       const __half* __restrict__ U,
                                                       long long n, __half* __restrict__ H) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n / 8;
       i += stride) {
    const uint4 gv = reinterpret_cast<const uint4*>(G)[i];
    const uint4 uv = reinterpret_cast<const uint4*>(U)[i];
    const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w}, uw[4] = {uv.x, uv.y, uv.z, uv.w};
    uint32_t o4[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      __half2 hg, hu;
      memcpy(&hg, &gw[j], 4);
      memcpy(&hu, &uw[j], 4);
      const float2 g = __half22float2(hg), u = __half22float2(hu);
      const float s0 = __fdiv_rn(g.x, __fadd_rn(1.0f, expf(-g.x)));
      const float s1 = __fdiv_rn(g.y, __fadd_rn(1.0f, expf(-g.y)));
      const __half2 out = __floats2half2_rn(__fmul_rn(s0, u.x), __fmul_rn(s1, u.y));
      memcpy(&o4[j], &out, 4);
    }
    reinterpret_cast<uint4*>(H)[i] = make_uint4(o4[0], o4[1], o4[2], o4[3]);
  }
}

}  // namespace block
}  // namespace awq
