// Sinusoidal distance table R[n_dist, dim]:
//   R[d, 2k] = sin(d * w_k),  R[d, 2k+1] = cos(d * w_k),  w_k = 10000^(-2k/dim)
// ("Transformer-XL, explained", symbol legend: R_{i-j} is a parameter-free
// sinusoid of the distance; no clipping, so every distance has an encoding).
//
// Precision: the product d * w_k is carried as an unevaluated sum of floats
// (w_k split into hi + lo parts; the rounding error of d * w_hi recovered
// exactly with an FMA), and reduced modulo 2*pi with a three-constant
// Cody-Waite split before the fp32 sine / cosine.  The result stays within a
// few 1e-7 of the exact table for every distance this library meets, where a
// plain fp32 angle would lose ~1e-4 rad at d ~ 3000.
//
// Launch: block (64, 4) covers 64 frequencies x 64 distances; grid
// (ceil(dim/2 / 64), ceil(n_dist / 64)).  HBM-write bound, tiny.
#include <cuda_bf16.h>

#include "txl_internal.h"

namespace txl {
namespace {

constexpr int kPairsPerBlock = 64;
constexpr int kRowsPerBlock = 64;

template <bool BF16>
__global__ void __launch_bounds__(256) sinusoid_kernel(void* __restrict__ R, int n_dist, int dim, float c1,
                                                       float c2, float c3) {
  __shared__ float s_whi[kPairsPerBlock];
  __shared__ float s_wlo[kPairsPerBlock];
  const int npairs = dim / 2;
  const int k = blockIdx.x * kPairsPerBlock + threadIdx.x;
  if (threadIdx.y == 0) {
    float hi = 0.f, lo = 0.f;
    if (k < npairs) {
      const double w = pow(10000.0, -2.0 * static_cast<double>(k) / static_cast<double>(dim));
      hi = static_cast<float>(w);
      lo = static_cast<float>(w - static_cast<double>(hi));
    }
    s_whi[threadIdx.x] = hi;
    s_wlo[threadIdx.x] = lo;
  }
  __syncthreads();
  if (k >= npairs) return;
  const float whi = s_whi[threadIdx.x];
  const float wlo = s_wlo[threadIdx.x];
  const float inv_two_pi = 0.15915494309189535f;
  const int d0 = blockIdx.y * kRowsPerBlock;
  for (int dd = threadIdx.y; dd < kRowsPerBlock; dd += blockDim.y) {
    const int d = d0 + dd;
    if (d >= n_dist) break;
    const float df = static_cast<float>(d);
    const float p = df * whi;
    const float e = fmaf(df, whi, -p);   // p + e == d * whi exactly
    const float t = fmaf(df, wlo, e);    // small remainder of the angle
    const float n = rintf(p * inv_two_pi);
    float x = fmaf(-n, c1, p);           // exact: n*c1 exact and close to p
    x = fmaf(-n, c2, x);
    x = fmaf(-n, c3, x);
    x += t;
    float s, c;
    sincosf(x, &s, &c);
    const size_t off = static_cast<size_t>(d) * dim + 2 * static_cast<size_t>(k);
    if (BF16) {
      __nv_bfloat162 v;
      v.x = __float2bfloat16_rn(s);
      v.y = __float2bfloat16_rn(c);
      *reinterpret_cast<__nv_bfloat162*>(static_cast<__nv_bfloat16*>(R) + off) = v;
    } else {
      *reinterpret_cast<float2*>(static_cast<float*>(R) + off) = make_float2(s, c);
    }
  }
}

}  // namespace

cudaError_t launch_sinusoid(void* R, int n_dist, int dim, bool bf16, float c1, float c2, float c3,
                            cudaStream_t stream) {
  const int npairs = dim / 2;
  dim3 block(kPairsPerBlock, 4);
  dim3 grid((npairs + kPairsPerBlock - 1) / kPairsPerBlock, (n_dist + kRowsPerBlock - 1) / kRowsPerBlock);
  if (bf16)
    sinusoid_kernel<true><<<grid, block, 0, stream>>>(R, n_dist, dim, c1, c2, c3);
  else
    sinusoid_kernel<false><<<grid, block, 0, stream>>>(R, n_dist, dim, c1, c2, c3);
  return cudaGetLastError();
}

}  // namespace txl
