// The layer around the attention: the projections and the feed-forward as
// plain bf16 GEMMs (cuBLASLt, fp32 accumulation), and this file's kernels for
// the rest -- residual + normalisation, and bias + ReLU.
//
// "Implementing Transformer-XL", recurrent-memory chapter (forward,
// layer_norm, feed_forward): x = LN1(h + attention(h, memory) W_o),
// out = LN2(x + ReLU(x W1 + b1) W2 + b2), LN(z) = gamma (z - mean) /
// (population std + 1e-6) + beta over the model width.
#include <cublasLt.h>
#include <cuda_bf16.h>

#include <cstdint>
#include <map>
#include <mutex>
#include <tuple>

#include "txl_internal.h"

namespace txl {
namespace {

constexpr float kLnEps = 1e-6f;

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Eight fp32 values at p (32-byte aligned) as two vector loads.
__device__ __forceinline__ void load8(const float* __restrict__ p, float (&v)[8]) {
  const float4 x = __ldg(reinterpret_cast<const float4*>(p));
  const float4 y = __ldg(reinterpret_cast<const float4*>(p) + 1);
  v[0] = x.x, v[1] = x.y, v[2] = x.z, v[3] = x.w, v[4] = y.x, v[5] = y.y, v[6] = y.z, v[7] = y.w;
}

// out[row] = LN(a[row] + b[row] (+ bias)), one warp per row of d columns
// (d a multiple of 8, at most 1024): each lane holds up to 4 chunks of 8.
// All of a row's loads are issued before any arithmetic, and the per-column
// vectors are read as float4.
__global__ void __launch_bounds__(256) add_ln_kernel(const __nv_bfloat16* __restrict__ a,
                                                     const __nv_bfloat16* __restrict__ b,
                                                     const float* __restrict__ bias,
                                                     const float* __restrict__ gamma,
                                                     const float* __restrict__ beta, __nv_bfloat16* __restrict__ out,
                                                     long long rows, int d) {
  const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const int nchunk = d / 8;
  uint4 va[4], vb[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int ch = lane + 32 * c;
    if (ch < nchunk) {
      va[c] = __ldg(reinterpret_cast<const uint4*>(a + row * d) + ch);
      vb[c] = __ldg(reinterpret_cast<const uint4*>(b + row * d) + ch);
    }
  }
  float x[4][8];
  float s = 0.f;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int ch = lane + 32 * c;
    if (ch < nchunk) {
      float bb[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (bias != nullptr) load8(bias + 8 * ch, bb);
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
  const float mean = warp_sum(s) / d;
  float v = 0.f;
#pragma unroll
  for (int c = 0; c < 4; ++c)
    if (lane + 32 * c < nchunk)
#pragma unroll
      for (int e = 0; e < 8; ++e) v += (x[c][e] - mean) * (x[c][e] - mean);
  const float inv = 1.f / (sqrtf(warp_sum(v) / d) + kLnEps);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int ch = lane + 32 * c;
    if (ch < nchunk) {
      float g[8], bt[8];
      load8(gamma + 8 * ch, g);
      load8(beta + 8 * ch, bt);
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

// f = ReLU(f + bias) in place over [rows, n] (n a multiple of 8): four
// independent 16-byte vectors a thread per round, all loaded first.
__global__ void __launch_bounds__(256) bias_relu_kernel(__nv_bfloat16* __restrict__ f,
                                                        const float* __restrict__ bias, long long n_vec, int n) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long base = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; base < n_vec;
       base += 4 * stride) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (base + u * stride < n_vec) v[u] = reinterpret_cast<const uint4*>(f)[base + u * stride];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const long long i = base + u * stride;
      if (i < n_vec) {
        float bb[8];
        load8(bias + (i * 8) % n, bb);
        __nv_bfloat162* p = reinterpret_cast<__nv_bfloat162*>(&v[u]);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 x = __bfloat1622float2(p[e]);
          p[e] = __floats2bfloat162_rn(fmaxf(x.x + bb[2 * e], 0.f), fmaxf(x.y + bb[2 * e + 1], 0.f));
        }
        reinterpret_cast<uint4*>(f)[i] = v[u];
      }
    }
  }
}

// cuBLASLt: one handle per device; per (device, m, n, k) the layouts and the
// heuristic's algorithm.
struct GemmPlan {
  cublasLtMatmulDesc_t op = nullptr;
  cublasLtMatrixLayout_t la = nullptr, lb = nullptr, lc = nullptr;
  cublasLtMatmulAlgo_t algo;
  bool ok = false;
};
std::mutex g_gemm_mutex;
std::map<int, cublasLtHandle_t> g_lt;
std::map<std::tuple<int, int, int, int>, GemmPlan> g_plans;

}  // namespace

cudaError_t launch_add_ln(const void* a, const void* b, const float* bias, const float* gamma, const float* beta,
                          void* out, long long rows, int d, cudaStream_t stream) {
  if (d % 8 != 0 || d > 1024) return cudaErrorInvalidValue;
  const long long blocks = (rows + 7) / 8;
  add_ln_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(a), static_cast<const __nv_bfloat16*>(b), bias, gamma, beta,
      static_cast<__nv_bfloat16*>(out), rows, d);
  return cudaGetLastError();
}

cudaError_t launch_bias_relu(void* f, const float* bias, long long rows, int n, cudaStream_t stream) {
  if (n % 8 != 0) return cudaErrorInvalidValue;
  const long long n_vec = rows * n / 8;
  long long blocks = (n_vec + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  bias_relu_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(static_cast<__nv_bfloat16*>(f), bias, n_vec,
                                                                       n);
  return cudaGetLastError();
}

// Row-major C [m, n] = A [m, k] B [k, n], bf16, fp32 accumulation.  In
// cuBLASLt's column-major terms: C^T (n x m) = B^T (n x k) A^T (k x m), with
// every matrix taken as stored.
int gemm_bf16(const void* A, const void* B, void* C, int m, int n, int k, void* ws, size_t ws_bytes,
              cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  GemmPlan* plan = nullptr;
  cublasLtHandle_t lt = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_gemm_mutex);
    auto h = g_lt.find(dev);
    if (h == g_lt.end()) {
      if (cublasLtCreate(&lt) != CUBLAS_STATUS_SUCCESS) return 1;
      g_lt[dev] = lt;
    } else {
      lt = h->second;
    }
    GemmPlan& p = g_plans[std::make_tuple(dev, m, n, k)];
    if (!p.ok) {
      if (cublasLtMatmulDescCreate(&p.op, CUBLAS_COMPUTE_32F, CUDA_R_32F) != CUBLAS_STATUS_SUCCESS) return 1;
      if (cublasLtMatrixLayoutCreate(&p.la, CUDA_R_16BF, n, k, n) != CUBLAS_STATUS_SUCCESS ||
          cublasLtMatrixLayoutCreate(&p.lb, CUDA_R_16BF, k, m, k) != CUBLAS_STATUS_SUCCESS ||
          cublasLtMatrixLayoutCreate(&p.lc, CUDA_R_16BF, n, m, n) != CUBLAS_STATUS_SUCCESS)
        return 1;
      cublasLtMatmulPreference_t pref;
      if (cublasLtMatmulPreferenceCreate(&pref) != CUBLAS_STATUS_SUCCESS) return 1;
      cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES, &ws_bytes,
                                           sizeof(ws_bytes));
      cublasLtMatmulHeuristicResult_t res;
      int n_res = 0;
      const cublasStatus_t st =
          cublasLtMatmulAlgoGetHeuristic(lt, p.op, p.la, p.lb, p.lc, p.lc, pref, 1, &res, &n_res);
      cublasLtMatmulPreferenceDestroy(pref);
      if (st != CUBLAS_STATUS_SUCCESS || n_res < 1) return 1;
      p.algo = res.algo;
      p.ok = true;
    }
    plan = &p;
  }
  const float alpha = 1.f, beta = 0.f;
  return cublasLtMatmul(lt, plan->op, &alpha, B, plan->la, A, plan->lb, &beta, C, plan->lc, C, plan->lc,
                        &plan->algo, ws, ws_bytes, stream) == CUBLAS_STATUS_SUCCESS
             ? 0
             : 1;
}

}  // namespace txl
