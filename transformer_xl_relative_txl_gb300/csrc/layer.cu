// The layer around the attention: the residual + normalisation kernel (the
// projections and the feed-forward are gemm_tc.cu's tensor-core GEMMs).
//
// "Implementing Transformer-XL", recurrent-memory chapter (forward,
// layer_norm, feed_forward): x = LN1(h + attention(h, memory) W_o),
// out = LN2(x + ReLU(x W1 + b1) W2 + b2), LN(z) = gamma (z - mean) /
// (population std + 1e-6) + beta over the model width.
#include <cuda_bf16.h>

#include <cstdint>
#include <map>
#include <mutex>
#include <tuple>

#include "pdl.cuh"
#include "txl_internal.h"

namespace txl {
namespace {

constexpr float kLnEps = 1e-6f;

__device__ __forceinline__ float half_sum(float x) {  // over the 16 lanes of a half-warp
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

constexpr int kLnMaxD = 1024;

// Shared-memory layout of a per-column vector for add_ln_kernel: column
// 8 ch + e sits at half (e / 4), word 4 ch + e % 4, so the float4 reads of
// the 16 lanes of a half-warp (chunks ch, ch + 1, ...) are consecutive
// 16-byte words: no bank conflicts.
__device__ __forceinline__ int ln_slot(int col) { return (col & 4) * (kLnMaxD / 8) + (col >> 3) * 4 + (col & 3); }

__device__ __forceinline__ void lds_chunk(const float* s, int ch, float (&v)[8]) {
  const float4 x = *reinterpret_cast<const float4*>(s + ch * 4);
  const float4 y = *reinterpret_cast<const float4*>(s + kLnMaxD / 2 + ch * 4);
  v[0] = x.x, v[1] = x.y, v[2] = x.z, v[3] = x.w, v[4] = y.x, v[5] = y.y, v[6] = y.z, v[7] = y.w;
}

// out[row] = LN(a[row] + b[row] (+ bias)), one half-warp per row of d
// columns (d a multiple of 8, at most 16 * 8 * kC): lane l holds chunks
// l, l + 16, ... of 8 columns.  All of the row's loads are issued first;
// the block then stages gamma, beta (and the bias) in shared memory while
// they are in flight.  x = a + b (+ bias) is formed once, in fp32, and kept
// for the two reductions (mean, then the squared deviations) and the
// output: with kC fixed at compile time that takes no more registers than
// the loaded vectors, and without a bias five 256-thread blocks an SM fit
// (80 rows in flight per SM, so 11264 rows, 22 x 512, take one wave); with
// one, four.
template <int kC, bool kBias>
__global__ void __launch_bounds__(256, kC > 4 ? 2 : kBias ? 4 : 5) add_ln_kernel(const __nv_bfloat16* __restrict__ a,
                                                                     const __nv_bfloat16* __restrict__ b,
                                                                     const float* __restrict__ bias,
                                                                     const float* __restrict__ gamma,
                                                                     const float* __restrict__ beta,
                                                                     __nv_bfloat16* __restrict__ out,
                                                                     long long rows, int d) {
  grid_dep_wait();  // launched behind the previous kernel on the stream: it has completed from here on
  grid_dep_launch_dependents();
  __shared__ __align__(16) float s_gamma[kLnMaxD], s_beta[kLnMaxD], s_bias[kBias ? kLnMaxD : 4];
  const long long row = static_cast<long long>(blockIdx.x) * 16 + (threadIdx.x >> 4);
  const int hl = threadIdx.x & 15;
  const bool live = row < rows;  // both halves of a warp take part in the shuffles
  const int nchunk = d / 8;
  uint4 va[kC], vb[kC];
#pragma unroll
  for (int c = 0; c < kC; ++c) {
    const int ch = hl + 16 * c;
    if (live && ch < nchunk) {
      va[c] = __ldg(reinterpret_cast<const uint4*>(a + row * d) + ch);
      vb[c] = __ldg(reinterpret_cast<const uint4*>(b + row * d) + ch);
    }
  }
  for (int i = threadIdx.x; i < d; i += blockDim.x) {
    s_gamma[ln_slot(i)] = __ldg(gamma + i);
    s_beta[ln_slot(i)] = __ldg(beta + i);
    if constexpr (kBias) s_bias[ln_slot(i)] = __ldg(bias + i);
  }
  __syncthreads();
  float x[kC][8];
  float s = 0.f;
#pragma unroll
  for (int c = 0; c < kC; ++c) {
    const int ch = hl + 16 * c;
    if (live && ch < nchunk) {
      float bb[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if constexpr (kBias) lds_chunk(s_bias, ch, bb);
      const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&va[c]);
      const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&vb[c]);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 fa = __bfloat1622float2(pa[e]), fb = __bfloat1622float2(pb[e]);
        x[c][2 * e] = fa.x + fb.x + bb[2 * e];
        x[c][2 * e + 1] = fa.y + fb.y + bb[2 * e + 1];
        s += x[c][2 * e] + x[c][2 * e + 1];
      }
    }
  }
  const float mean = half_sum(s) / d;
  float v = 0.f;
#pragma unroll
  for (int c = 0; c < kC; ++c)
    if (live && hl + 16 * c < nchunk)
#pragma unroll
      for (int e = 0; e < 8; ++e) v += (x[c][e] - mean) * (x[c][e] - mean);
  const float inv = 1.f / (sqrtf(half_sum(v) / d) + kLnEps);
  if (!live) return;
#pragma unroll
  for (int c = 0; c < kC; ++c) {
    const int ch = hl + 16 * c;
    if (ch < nchunk) {
      float g[8], bt[8];
      lds_chunk(s_gamma, ch, g);
      lds_chunk(s_beta, ch, bt);
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const __nv_bfloat162 p2 = __floats2bfloat162_rn(g[2 * e] * (x[c][2 * e] - mean) * inv + bt[2 * e],
                                                        g[2 * e + 1] * (x[c][2 * e + 1] - mean) * inv + bt[2 * e + 1]);
        w[e] = *reinterpret_cast<const uint32_t*>(&p2);
      }
      *reinterpret_cast<uint4*>(out + row * d + 8 * ch) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

}  // namespace

namespace {
template <int kC>
cudaError_t add_ln_dispatch(unsigned blocks, const __nv_bfloat16* a, const __nv_bfloat16* b, const float* bias,
                            const float* gamma, const float* beta, __nv_bfloat16* out, long long rows, int d,
                            cudaStream_t stream) {
  if (bias != nullptr)
    return launch_dependent(add_ln_kernel<kC, true>, dim3(blocks), dim3(256), 0, stream, a, b, bias, gamma, beta, out,
                            rows, d);
  return launch_dependent(add_ln_kernel<kC, false>, dim3(blocks), dim3(256), 0, stream, a, b, bias, gamma, beta, out,
                          rows, d);
}
}  // namespace

cudaError_t launch_add_ln(const void* a, const void* b, const float* bias, const float* gamma, const float* beta,
                          void* out, long long rows, int d, cudaStream_t stream) {
  if (d % 8 != 0 || d > kLnMaxD) return cudaErrorInvalidValue;
  if (rows <= 0) return cudaSuccess;
  const unsigned blocks = static_cast<unsigned>((rows + 15) / 16);
  const auto* pa = static_cast<const __nv_bfloat16*>(a);
  const auto* pb = static_cast<const __nv_bfloat16*>(b);
  auto* po = static_cast<__nv_bfloat16*>(out);
  const int per_lane = (d / 8 + 15) / 16;  // chunks of 8 columns a lane holds
  if (per_lane <= 1) return add_ln_dispatch<1>(blocks, pa, pb, bias, gamma, beta, po, rows, d, stream);
  if (per_lane <= 2) return add_ln_dispatch<2>(blocks, pa, pb, bias, gamma, beta, po, rows, d, stream);
  if (per_lane <= 4) return add_ln_dispatch<4>(blocks, pa, pb, bias, gamma, beta, po, rows, d, stream);
  return add_ln_dispatch<8>(blocks, pa, pb, bias, gamma, beta, po, rows, d, stream);
}

}  // namespace txl
