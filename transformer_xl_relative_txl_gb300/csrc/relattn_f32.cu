// Exact fp32 relative attention on CUDA cores.
//
//   s[i,j] = scale * ((q_i + u) . k_j + (q_i + v) . r_{M+i-j}),   j <= M+i
//   o_i = softmax(s[i,.]) V,   lse_i = log sum_j exp(s[i,j])
//
// ("Transformer-XL, explained", method steps 3-5; the mask and the
// 1/sqrt(d_head) scale of "Implementing Transformer-XL", relative_attention.)
// The distance term is indexed per (i, j) pair at row M+i-j of r, the same
// in-kernel distance index the tensor-core path uses.
//
// One CTA per (query i, head h, batch b), 128 threads.  Pass 1: each thread
// scores keys j = tid, tid+128, ... into shared memory and the block reduces
// the max; pass 2 exponentiates and reduces the sum; pass 3 forms o with
// threads over the head dimension (coalesced reads of the value rows).
// Accurate to ~1e-6 against the float64 definition; used for fp32 callers
// and small workloads, not for throughput.
#include <cfloat>

#include "txl_internal.h"

namespace txl {
namespace {

constexpr int kThreads = 128;

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

template <bool IS_MAX>
__device__ float block_reduce(float x, float* scratch) {
  x = IS_MAX ? warp_max(x) : warp_sum(x);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) scratch[warp] = x;
  __syncthreads();
  float y = scratch[0];
#pragma unroll
  for (int w = 1; w < kThreads / 32; ++w) y = IS_MAX ? fmaxf(y, scratch[w]) : y + scratch[w];
  return y;
}

__global__ void __launch_bounds__(kThreads) relattn_f32_kernel(
    const float* __restrict__ q, const float* __restrict__ k, const float* __restrict__ v,
    const float* __restrict__ r, const float* __restrict__ bias_u, const float* __restrict__ bias_v,
    float* __restrict__ o, float* __restrict__ lse, int W, int M, int H, int D, float scale) {
  extern __shared__ float smem[];
  float* qu = smem;             // [D]  q_i + u
  float* qv = smem + D;         // [D]  q_i + v
  float* sc = smem + 2 * D;     // [M + i + 1] scores, then probabilities
  __shared__ float red[kThreads / 32];

  const int i = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int L = M + W;
  const size_t qrow = ((static_cast<size_t>(b) * W + i) * H + h) * D;
  for (int d = threadIdx.x; d < D; d += kThreads) {
    const float x = q[qrow + d];
    qu[d] = x + bias_u[h * D + d];
    qv[d] = x + bias_v[h * D + d];
  }
  __syncthreads();

  const int nvis = M + i + 1;  // keys j = 0 .. M+i are visible
  float mx = -FLT_MAX;
  for (int j = threadIdx.x; j < nvis; j += kThreads) {
    const float* kr = k + ((static_cast<size_t>(b) * L + j) * H + h) * D;
    const float* rr = r + (static_cast<size_t>(M + i - j) * H + h) * D;  // distance M+i-j
    float ac = 0.f, bd = 0.f;
    for (int d = 0; d < D; ++d) {
      ac = fmaf(qu[d], kr[d], ac);
      bd = fmaf(qv[d], rr[d], bd);
    }
    const float s = scale * (ac + bd);
    sc[j] = s;
    mx = fmaxf(mx, s);
  }
  mx = block_reduce<true>(mx, red);

  float sum = 0.f;
  for (int j = threadIdx.x; j < nvis; j += kThreads) {
    const float p = expf(sc[j] - mx);
    sc[j] = p;
    sum += p;
  }
  sum = block_reduce<false>(sum, red);  // also orders the sc[] writes before pass 3
  const float inv = 1.f / sum;

  for (int d = threadIdx.x; d < D; d += kThreads) {
    float acc = 0.f;
    const float* vc = v + (static_cast<size_t>(b) * L * H + h) * D + d;
    const size_t vstride = static_cast<size_t>(H) * D;
    for (int j = 0; j < nvis; ++j) acc = fmaf(sc[j], vc[j * vstride], acc);
    o[qrow + d] = acc * inv;
  }
  if (lse != nullptr && threadIdx.x == 0) lse[(static_cast<size_t>(b) * H + h) * W + i] = mx + logf(sum);
}

}  // namespace

cudaError_t launch_relattn_f32(const float* q, const float* k, const float* v, const float* r,
                               const float* bias_u, const float* bias_v, float* o, float* lse, int B,
                               int W, int M, int H, int D, float scale, cudaStream_t stream) {
  const size_t smem = sizeof(float) * (2 * static_cast<size_t>(D) + M + W);
  cudaError_t e = cudaFuncSetAttribute(relattn_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid(W, H, B);
  relattn_f32_kernel<<<grid, kThreads, smem, stream>>>(q, k, v, r, bias_u, bias_v, o, lse, W, M, H, D, scale);
  return cudaGetLastError();
}

}  // namespace txl
