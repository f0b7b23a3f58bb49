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

// Eight fp32 values at p (32-byte aligned) as two vector loads.
__device__ __forceinline__ void load8(const float* __restrict__ p, float (&v)[8]) {
  const float4 x = __ldg(reinterpret_cast<const float4*>(p));
  const float4 y = __ldg(reinterpret_cast<const float4*>(p) + 1);
  v[0] = x.x, v[1] = x.y, v[2] = x.z, v[3] = x.w, v[4] = y.x, v[5] = y.y, v[6] = y.z, v[7] = y.w;
}

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
// one, four.  The grid also runs the side jobs in cvt, an element a
// thread: dst[j][i] = bf16(src[j][i]) for i < n[j], vectors later kernels
// want in bf16, rounded without a launch of their own.
template <int kC, bool kBias>
__global__ void __launch_bounds__(256, kC > 4 ? 2 : kBias ? 4 : 5) add_ln_kernel(const __nv_bfloat16* __restrict__ a,
                                                                     const __nv_bfloat16* __restrict__ b,
                                                                     const float* __restrict__ bias,
                                                                     const float* __restrict__ gamma,
                                                                     const float* __restrict__ beta,
                                                                     __nv_bfloat16* __restrict__ out,
                                                                     long long rows, int d, CvtJobs cvt) {
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
#pragma unroll
  for (int j = 0; j < 2; ++j)  // the side jobs: dst = bf16(src), spread over the grid
    if (cvt.dst[j] != nullptr)
      for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < cvt.n[j];
           i += static_cast<long long>(gridDim.x) * blockDim.x)
        cvt.dst[j][i] = __float2bfloat16_rn(__ldg(cvt.src[j] + i));
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

// cuBLASLt: one handle per device; per (device, m, n, k, epilogue) the
// layouts and the heuristic's algorithm.  A plan whose heuristic found
// nothing is kept as unsupported so the search is not repeated.
struct GemmPlan {
  cublasLtMatmulDesc_t op = nullptr;
  cublasLtMatrixLayout_t la = nullptr, lb = nullptr, lc = nullptr;
  cublasLtMatmulAlgo_t algo;
  bool ok = false, unsupported = false;
};
std::mutex g_gemm_mutex;
std::map<int, cublasLtHandle_t> g_lt;
// key: device, m, n, k, epilogue (0 none, 1 bias, 2 ReLU + bias), batch, C's batch stride
std::map<std::tuple<int, int, int, int, int, int, long long>, GemmPlan> g_plans;

}  // namespace

namespace {
template <int kC>
void add_ln_dispatch(unsigned blocks, const __nv_bfloat16* a, const __nv_bfloat16* b, const float* bias,
                     const float* gamma, const float* beta, __nv_bfloat16* out, long long rows, int d,
                     const CvtJobs& cvt, cudaStream_t stream) {
  if (bias != nullptr)
    add_ln_kernel<kC, true><<<blocks, 256, 0, stream>>>(a, b, bias, gamma, beta, out, rows, d, cvt);
  else
    add_ln_kernel<kC, false><<<blocks, 256, 0, stream>>>(a, b, bias, gamma, beta, out, rows, d, cvt);
}
}  // namespace

cudaError_t launch_add_ln(const void* a, const void* b, const float* bias, const float* gamma, const float* beta,
                          void* out, long long rows, int d, cudaStream_t stream, const CvtJobs& cvt) {
  if (d % 8 != 0 || d > kLnMaxD || cvt.n[0] < 0 || cvt.n[1] < 0) return cudaErrorInvalidValue;
  if (rows <= 0) return cudaSuccess;
  const unsigned blocks = static_cast<unsigned>((rows + 15) / 16);
  const auto* pa = static_cast<const __nv_bfloat16*>(a);
  const auto* pb = static_cast<const __nv_bfloat16*>(b);
  auto* po = static_cast<__nv_bfloat16*>(out);
  const int per_lane = (d / 8 + 15) / 16;  // chunks of 8 columns a lane holds
  if (per_lane <= 1)
    add_ln_dispatch<1>(blocks, pa, pb, bias, gamma, beta, po, rows, d, cvt, stream);
  else if (per_lane <= 2)
    add_ln_dispatch<2>(blocks, pa, pb, bias, gamma, beta, po, rows, d, cvt, stream);
  else if (per_lane <= 4)
    add_ln_dispatch<4>(blocks, pa, pb, bias, gamma, beta, po, rows, d, cvt, stream);
  else
    add_ln_dispatch<8>(blocks, pa, pb, bias, gamma, beta, po, rows, d, cvt, stream);
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

// Row-major C [m, n] = A [m, k] B [k, n], bf16, fp32 accumulation; with
// bias (bf16, n values: cuBLASLt's bias epilogues take the bias in the
// output's type) C = A B + bias, or ReLU(A B + bias) with relu, the bias
// added to the fp32 accumulator before the one rounding.  In
// cuBLASLt's column-major terms: C^T (n x m) = B^T (n x k) A^T (k x m), with
// every matrix taken as stored; the bias runs along C^T's rows.  Returns 0,
// 1 on a cuBLASLt error, 2 when no algorithm takes the epilogue (the caller
// then applies it itself).  The plan cache and the per-call bias pointer are
// guarded by one lock held until the matmul is enqueued.
int gemm_bf16(const void* A, const void* B, void* C, int m, int n, int k, void* ws, size_t ws_bytes,
              cudaStream_t stream, const void* bias, bool relu) {
  return gemm_bf16_batched(A, B, C, m, n, k, 1, 0, ws, ws_bytes, stream, bias, relu);
}

// batch > 1: C_i = A B_i for i < batch, B_i = B + i k n elements (the
// matrices packed back to back), C_i = C + i c_stride elements; A is shared
// (batch stride 0).
int gemm_bf16_batched(const void* A, const void* B, void* C, int m, int n, int k, int batch, long long c_stride,
                      void* ws, size_t ws_bytes, cudaStream_t stream, const void* bias, bool relu) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (batch < 1 || (batch > 1 && c_stride < static_cast<long long>(m) * n)) return 1;
  const int epi = bias == nullptr ? 0 : relu ? 2 : 1;
  std::lock_guard<std::mutex> lk(g_gemm_mutex);
  cublasLtHandle_t lt = nullptr;
  auto h = g_lt.find(dev);
  if (h == g_lt.end()) {
    if (cublasLtCreate(&lt) != CUBLAS_STATUS_SUCCESS) return 1;
    g_lt[dev] = lt;
  } else {
    lt = h->second;
  }
  GemmPlan& p = g_plans[std::make_tuple(dev, m, n, k, epi, batch, batch > 1 ? c_stride : 0LL)];
  if (p.unsupported) return 2;
  if (!p.ok) {
    if (cublasLtMatmulDescCreate(&p.op, CUBLAS_COMPUTE_32F, CUDA_R_32F) != CUBLAS_STATUS_SUCCESS) return 1;
    if (epi) {
      const cublasLtEpilogue_t e = epi == 2 ? CUBLASLT_EPILOGUE_RELU_BIAS : CUBLASLT_EPILOGUE_BIAS;
      const cudaDataType_t bt = CUDA_R_16BF;
      if (cublasLtMatmulDescSetAttribute(p.op, CUBLASLT_MATMUL_DESC_EPILOGUE, &e, sizeof(e)) !=
              CUBLAS_STATUS_SUCCESS ||
          cublasLtMatmulDescSetAttribute(p.op, CUBLASLT_MATMUL_DESC_BIAS_DATA_TYPE, &bt, sizeof(bt)) !=
              CUBLAS_STATUS_SUCCESS) {
        p.unsupported = true;
        return 2;
      }
    }
    if (cublasLtMatrixLayoutCreate(&p.la, CUDA_R_16BF, n, k, n) != CUBLAS_STATUS_SUCCESS ||
        cublasLtMatrixLayoutCreate(&p.lb, CUDA_R_16BF, k, m, k) != CUBLAS_STATUS_SUCCESS ||
        cublasLtMatrixLayoutCreate(&p.lc, CUDA_R_16BF, n, m, n) != CUBLAS_STATUS_SUCCESS)
      return 1;
    if (batch > 1) {
      const long long sa = static_cast<long long>(k) * n, sb = 0;  // B^T packed; A^T shared
      const cublasLtMatrixLayoutAttribute_t cnt = CUBLASLT_MATRIX_LAYOUT_BATCH_COUNT,
                                            off = CUBLASLT_MATRIX_LAYOUT_STRIDED_BATCH_OFFSET;
      if (cublasLtMatrixLayoutSetAttribute(p.la, cnt, &batch, sizeof(batch)) != CUBLAS_STATUS_SUCCESS ||
          cublasLtMatrixLayoutSetAttribute(p.la, off, &sa, sizeof(sa)) != CUBLAS_STATUS_SUCCESS ||
          cublasLtMatrixLayoutSetAttribute(p.lb, cnt, &batch, sizeof(batch)) != CUBLAS_STATUS_SUCCESS ||
          cublasLtMatrixLayoutSetAttribute(p.lb, off, &sb, sizeof(sb)) != CUBLAS_STATUS_SUCCESS ||
          cublasLtMatrixLayoutSetAttribute(p.lc, cnt, &batch, sizeof(batch)) != CUBLAS_STATUS_SUCCESS ||
          cublasLtMatrixLayoutSetAttribute(p.lc, off, &c_stride, sizeof(c_stride)) != CUBLAS_STATUS_SUCCESS)
        return 1;
    }
    cublasLtMatmulPreference_t pref;
    if (cublasLtMatmulPreferenceCreate(&pref) != CUBLAS_STATUS_SUCCESS) return 1;
    cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES, &ws_bytes,
                                         sizeof(ws_bytes));
    cublasLtMatmulHeuristicResult_t res;
    int n_res = 0;
    const cublasStatus_t st = cublasLtMatmulAlgoGetHeuristic(lt, p.op, p.la, p.lb, p.lc, p.lc, pref, 1, &res, &n_res);
    cublasLtMatmulPreferenceDestroy(pref);
    if (st != CUBLAS_STATUS_SUCCESS || n_res < 1) {
      if (!epi) return 1;
      p.unsupported = true;
      return 2;
    }
    p.algo = res.algo;
    p.ok = true;
  }
  if (epi && cublasLtMatmulDescSetAttribute(p.op, CUBLASLT_MATMUL_DESC_BIAS_POINTER, &bias, sizeof(bias)) !=
                 CUBLAS_STATUS_SUCCESS)
    return 1;
  const float alpha = 1.f, beta = 0.f;
  return cublasLtMatmul(lt, p.op, &alpha, B, p.la, A, p.lb, &beta, C, p.lc, C, p.lc, &p.algo, ws, ws_bytes,
                        stream) == CUBLAS_STATUS_SUCCESS
             ? 0
             : 1;
}

}  // namespace txl
