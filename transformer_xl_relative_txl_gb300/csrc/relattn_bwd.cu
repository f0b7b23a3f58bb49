// Backward of the relative attention on CUDA cores, fp32 arithmetic, any
// input dtype (fp32 or bf16) and head dim D <= 256.
//
// With o = softmax(s) V, s[i,j] = scale ((q_i+u).k_j + (q_i+v).r_{M+i-j})
// for j <= M+i, and dO the gradient of the output:
//
//   p_ij  = exp(s_ij - lse_i)                  (the forward's lse)
//   Delta_i = dO_i . o_i                       (= sum_j p_ij dO_i.v_j)
//   g_ij  = scale p_ij (dO_i.v_j - Delta_i)    (gradient of the unscaled terms)
//   dq_i  = sum_j g_ij k_j  +  sum_j g_ij r_{M+i-j}
//   dk_j  = sum_i g_ij (q_i+u),   dv_j = sum_i p_ij dO_i   (segment rows j >= M)
//   dr_d  = sum over pairs with M+i-j = d of g_ij (q_i+v)
//   du    = sum_{b,i} sum_j g_ij k_j,   dv_bias = sum_{b,i} sum_j g_ij r_{M+i-j}
//
// "Transformer-XL, explained", method step 2 and the symbol SG(.): the memory
// is a fixed input and backpropagation stays inside the segment, so memory
// rows get no dk / dv.  r, u and v are shared by every pair.
//
// Four kernels, each recomputing p and g for the pairs it needs, so no
// gradient is accumulated with atomics and every result is deterministic:
//   delta   one warp per query row: Delta_i;
//   dq      one warp per query row, lanes over keys for the scores, then over
//           the head dimension for the sums (coalesced row reads); also the
//           per-CTA partial sums of the two halves of dq for du / dv_bias;
//   dkdv    one warp per segment key, lanes over queries;
//   dr      one warp per distance d, lanes over the queries of each batch;
//   bias    one CTA per head: sums the partials in a fixed order.
// Meant for fp32 callers and shapes the tensor-core path does not take.
#include <cuda_bf16.h>

#include <cstdint>

#include "pdl.cuh"
#include "txl_internal.h"

namespace txl {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kMaxDPerLane = 8;  // D <= 256

__device__ __forceinline__ float ldf(const float* p) { return __ldg(p); }
__device__ __forceinline__ float ldf(const __nv_bfloat16* p) { return __bfloat162float(*p); }

// row . vec over D, row in global memory (type T), vec in shared memory.
template <typename T>
__device__ __forceinline__ float dot_row(const T* __restrict__ row, const float* vec, int D, bool vec16) {
  float a0 = 0.f, a1 = 0.f;
  if constexpr (sizeof(T) == 2) {
    if (vec16) {
      for (int d = 0; d < D; d += 8) {
        const uint4 w = __ldg(reinterpret_cast<const uint4*>(row + d));
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ws[e]));
          a0 = fmaf(f.x, vec[d + 2 * e], a0);
          a1 = fmaf(f.y, vec[d + 2 * e + 1], a1);
        }
      }
      return a0 + a1;
    }
  } else {
    if (vec16) {
      for (int d = 0; d < D; d += 4) {
        const float4 f = __ldg(reinterpret_cast<const float4*>(row + d));
        a0 = fmaf(f.x, vec[d], a0);
        a1 = fmaf(f.y, vec[d + 1], a1);
        a0 = fmaf(f.z, vec[d + 2], a0);
        a1 = fmaf(f.w, vec[d + 3], a1);
      }
      return a0 + a1;
    }
  }
  for (int d = 0; d < D; ++d) a0 = fmaf(ldf(row + d), vec[d], a0);
  return a0;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

struct BwdArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* r;
  const float* bias_u;
  const float* bias_v;
  const void* o;
  const float* lse;
  const void* dout;
  float* dq;
  float* dk;
  float* dv;
  float* dr;
  float* delta;     // [B, H, W] scratch
  float* part;      // [B * gridDim.x of dq][H][2][D] scratch
  int B, W, M, H, D, n_r;
  float scale;
  bool vec16;       // every row of q, k, v, r starts on a 16-byte boundary and D fits the vector width
};

// Row pointers ([B, rows, H, D] layouts).
template <typename T>
__device__ __forceinline__ const T* row_of(const void* base, int b, int rows, int t, int h, int H, int D) {
  return static_cast<const T*>(base) + ((static_cast<long long>(b) * rows + t) * H + h) * D;
}

// Delta_i = dO_i . o_i, one warp per row (TG: dtype of o and dO).
template <typename TG>
__global__ void __launch_bounds__(kThreads) bwd_delta_kernel(BwdArgs a) {
  const int lane = threadIdx.x & 31;
  const int i = blockIdx.x * kWarps + (threadIdx.x >> 5), h = blockIdx.y, b = blockIdx.z;
  if (i >= a.W) return;
  const TG* o = row_of<TG>(a.o, b, a.W, i, h, a.H, a.D);
  const TG* g = row_of<TG>(a.dout, b, a.W, i, h, a.H, a.D);
  float s = 0.f;
  for (int d = lane; d < a.D; d += 32) s = fmaf(ldf(o + d), ldf(g + d), s);
  s = warp_sum(s);
  if (lane == 0) a.delta[(static_cast<long long>(b) * a.H + h) * a.W + i] = s;
}

// dq, one warp per query row; per-CTA partial sums of d(q+u) and d(q+v).
template <typename T, typename TG>
__global__ void __launch_bounds__(kThreads) bwd_dq_kernel(BwdArgs a) {
  extern __shared__ float sm[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int h = blockIdx.y, b = blockIdx.z, D = a.D, L = a.M + a.W;
  float* qu = sm + warp * 3 * D;  // q_i + u
  float* qv = qu + D;             // q_i + v
  float* go = qv + D;             // dO_i
  float* red = sm + kWarps * 3 * D;  // [kWarps][2][D]
  float su[kMaxDPerLane], sv[kMaxDPerLane];  // this warp's sums over its rows
#pragma unroll
  for (int c = 0; c < kMaxDPerLane; ++c) su[c] = sv[c] = 0.f;

  const int i = blockIdx.x * kWarps + warp;
  if (i < a.W) {
    const T* qrow = row_of<T>(a.q, b, a.W, i, h, a.H, D);
    const TG* grow = row_of<TG>(a.dout, b, a.W, i, h, a.H, D);
    for (int d = lane; d < D; d += 32) {
      const float x = ldf(qrow + d);
      qu[d] = x + a.bias_u[h * D + d];
      qv[d] = x + a.bias_v[h * D + d];
      go[d] = ldf(grow + d);
    }
    __syncwarp();
    const long long row = (static_cast<long long>(b) * a.H + h) * a.W + i;
    const float lse = a.lse[row], delta = a.delta[row];
    float au[kMaxDPerLane], av[kMaxDPerLane];
#pragma unroll
    for (int c = 0; c < kMaxDPerLane; ++c) au[c] = av[c] = 0.f;
    const int jmax = a.M + i;  // last visible key
    for (int j0 = 0; j0 <= jmax; j0 += 32) {
      const int j = j0 + lane;
      float g = 0.f;
      if (j <= jmax) {
        const T* krow = row_of<T>(a.k, b, L, j, h, a.H, D);
        const T* vrow = row_of<T>(a.v, b, L, j, h, a.H, D);
        const T* rrow = static_cast<const T*>(a.r) + (static_cast<long long>(jmax - j) * a.H + h) * D;
        const float s = a.scale * (dot_row(krow, qu, D, a.vec16) + dot_row(rrow, qv, D, a.vec16));
        const float p = expf(s - lse);
        g = a.scale * p * (dot_row(vrow, go, D, a.vec16) - delta);
      }
      const int nj = min(32, jmax - j0 + 1);
      for (int t = 0; t < nj; ++t) {
        const float gt = __shfl_sync(0xffffffffu, g, t);
        const int jt = j0 + t;
        const T* krow = row_of<T>(a.k, b, L, jt, h, a.H, D);
        const T* rrow = static_cast<const T*>(a.r) + (static_cast<long long>(jmax - jt) * a.H + h) * D;
#pragma unroll
        for (int c = 0; c < kMaxDPerLane; ++c) {
          const int d = lane + 32 * c;
          if (d < D) {
            au[c] = fmaf(gt, ldf(krow + d), au[c]);
            av[c] = fmaf(gt, ldf(rrow + d), av[c]);
          }
        }
      }
    }
    float* dqrow = a.dq + ((static_cast<long long>(b) * a.W + i) * a.H + h) * D;
#pragma unroll
    for (int c = 0; c < kMaxDPerLane; ++c) {
      const int d = lane + 32 * c;
      if (d < D) dqrow[d] = au[c] + av[c];
      su[c] += au[c];
      sv[c] += av[c];
    }
  }
  // Partial sums of this CTA's rows, warps added in a fixed order.
#pragma unroll
  for (int c = 0; c < kMaxDPerLane; ++c) {
    const int d = lane + 32 * c;
    if (d < D) {
      red[(warp * 2) * D + d] = su[c];
      red[(warp * 2 + 1) * D + d] = sv[c];
    }
  }
  __syncthreads();
  float* part = a.part + ((static_cast<long long>(b) * gridDim.x + blockIdx.x) * a.H + h) * 2 * D;
  for (int x = threadIdx.x; x < 2 * D; x += kThreads) {
    float s = 0.f;
    for (int w = 0; w < kWarps; ++w) s += red[w * 2 * D + x];
    part[x] = s;
  }
}

// dk, dv of segment key jj (row M + jj of k and v), one warp per key.
template <typename T, typename TG>
__global__ void __launch_bounds__(kThreads) bwd_dkdv_kernel(BwdArgs a) {
  extern __shared__ float sm[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int h = blockIdx.y, b = blockIdx.z, D = a.D, L = a.M + a.W;
  float* kj = sm + warp * 2 * D;
  float* vj = kj + D;
  float* bu = sm + kWarps * 2 * D;  // u, then v of head h
  float* bv = bu + D;
  for (int d = threadIdx.x; d < D; d += kThreads) {
    bu[d] = a.bias_u[h * D + d];
    bv[d] = a.bias_v[h * D + d];
  }
  __syncthreads();
  const int jj = blockIdx.x * kWarps + warp;
  if (jj >= a.W) return;
  const int j = a.M + jj;
  const T* krow = row_of<T>(a.k, b, L, j, h, a.H, D);
  const T* vrow = row_of<T>(a.v, b, L, j, h, a.H, D);
  for (int d = lane; d < D; d += 32) {
    kj[d] = ldf(krow + d);
    vj[d] = ldf(vrow + d);
  }
  __syncwarp();
  float ak[kMaxDPerLane], av[kMaxDPerLane];
#pragma unroll
  for (int c = 0; c < kMaxDPerLane; ++c) ak[c] = av[c] = 0.f;
  // Key j is visible to queries i >= jj; its distance there is i - jj.
  for (int i0 = jj; i0 < a.W; i0 += 32) {
    const int i = i0 + lane;
    float p = 0.f, g = 0.f;
    if (i < a.W) {
      const T* qrow = row_of<T>(a.q, b, a.W, i, h, a.H, D);
      const TG* grow = row_of<TG>(a.dout, b, a.W, i, h, a.H, D);
      const T* rrow = static_cast<const T*>(a.r) + (static_cast<long long>(i - jj) * a.H + h) * D;
      // (q_i + u).k_j and (q_i + v).r_d with the biases' parts added once
      float qk = 0.f, qr = 0.f, dp = 0.f, uk = 0.f, vr = 0.f;
      for (int d = 0; d < D; ++d) {
        const float x = ldf(qrow + d), rd = ldf(rrow + d);
        qk = fmaf(x, kj[d], qk);
        uk = fmaf(bu[d], kj[d], uk);
        qr = fmaf(x, rd, qr);
        vr = fmaf(bv[d], rd, vr);
        dp = fmaf(ldf(grow + d), vj[d], dp);
      }
      const long long row = (static_cast<long long>(b) * a.H + h) * a.W + i;
      p = expf(a.scale * ((qk + uk) + (qr + vr)) - a.lse[row]);
      g = a.scale * p * (dp - a.delta[row]);
    }
    const int ni = min(32, a.W - i0);
    for (int t = 0; t < ni; ++t) {
      const float pt = __shfl_sync(0xffffffffu, p, t);
      const float gt = __shfl_sync(0xffffffffu, g, t);
      const T* qrow = row_of<T>(a.q, b, a.W, i0 + t, h, a.H, D);
      const TG* grow = row_of<TG>(a.dout, b, a.W, i0 + t, h, a.H, D);
#pragma unroll
      for (int c = 0; c < kMaxDPerLane; ++c) {
        const int d = lane + 32 * c;
        if (d < D) {
          ak[c] = fmaf(gt, ldf(qrow + d) + bu[d], ak[c]);
          av[c] = fmaf(pt, ldf(grow + d), av[c]);
        }
      }
    }
  }
  const long long o = ((static_cast<long long>(b) * a.W + jj) * a.H + h) * D;
#pragma unroll
  for (int c = 0; c < kMaxDPerLane; ++c) {
    const int d = lane + 32 * c;
    if (d < D) {
      a.dk[o + d] = ak[c];
      a.dv[o + d] = av[c];
    }
  }
}

// dr of distance d (row d of r), one warp per distance; rows no pair uses
// (d >= M + W) are zero.
template <typename T, typename TG>
__global__ void __launch_bounds__(kThreads) bwd_dr_kernel(BwdArgs a) {
  extern __shared__ float sm[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int h = blockIdx.y, D = a.D, L = a.M + a.W;
  float* rd = sm + warp * D;
  float* bu = sm + kWarps * D;
  float* bv = bu + D;
  for (int x = threadIdx.x; x < D; x += kThreads) {
    bu[x] = a.bias_u[h * D + x];
    bv[x] = a.bias_v[h * D + x];
  }
  __syncthreads();
  const int dist = blockIdx.x * kWarps + warp;
  if (dist >= a.n_r) return;
  float* out = a.dr + (static_cast<long long>(dist) * a.H + h) * D;
  float ar[kMaxDPerLane];
#pragma unroll
  for (int c = 0; c < kMaxDPerLane; ++c) ar[c] = 0.f;
  if (dist < L) {
    const T* rrow = static_cast<const T*>(a.r) + (static_cast<long long>(dist) * a.H + h) * D;
    for (int x = lane; x < D; x += 32) rd[x] = ldf(rrow + x);
    __syncwarp();
    const float vr = [&] {
      float s = 0.f;
      for (int x = lane; x < D; x += 32) s = fmaf(bv[x], rd[x], s);
      return warp_sum(s);
    }();
    // Pairs at this distance: query i >= dist - M, key j = M + i - dist.
    const int ilo = max(0, dist - a.M);
    for (int b = 0; b < a.B; ++b) {
      for (int i0 = ilo; i0 < a.W; i0 += 32) {
        const int i = i0 + lane;
        float g = 0.f;
        if (i < a.W) {
          const int j = a.M + i - dist;
          const T* qrow = row_of<T>(a.q, b, a.W, i, h, a.H, D);
          const T* krow = row_of<T>(a.k, b, L, j, h, a.H, D);
          const T* vrow = row_of<T>(a.v, b, L, j, h, a.H, D);
          const TG* grow = row_of<TG>(a.dout, b, a.W, i, h, a.H, D);
          float qk = 0.f, uk = 0.f, qr = 0.f, dp = 0.f;
          for (int x = 0; x < D; ++x) {
            const float qx = ldf(qrow + x), kx = ldf(krow + x);
            qk = fmaf(qx, kx, qk);
            uk = fmaf(bu[x], kx, uk);
            qr = fmaf(qx, rd[x], qr);
            dp = fmaf(ldf(grow + x), ldf(vrow + x), dp);
          }
          const long long row = (static_cast<long long>(b) * a.H + h) * a.W + i;
          const float p = expf(a.scale * ((qk + uk) + (qr + vr)) - a.lse[row]);
          g = a.scale * p * (dp - a.delta[row]);
        }
        const int ni = min(32, a.W - i0);
        for (int t = 0; t < ni; ++t) {
          const float gt = __shfl_sync(0xffffffffu, g, t);
          const T* qrow = row_of<T>(a.q, b, a.W, i0 + t, h, a.H, D);
#pragma unroll
          for (int c = 0; c < kMaxDPerLane; ++c) {
            const int x = lane + 32 * c;
            if (x < D) ar[c] = fmaf(gt, ldf(qrow + x) + bv[x], ar[c]);
          }
        }
      }
    }
  }
#pragma unroll
  for (int c = 0; c < kMaxDPerLane; ++c) {
    const int x = lane + 32 * c;
    if (x < D) out[x] = ar[c];
  }
}

// du, dv_bias from the partials: one warp per (head, column) -- grid
// (H, 2D / 8), 8 warps a block -- lanes over the partials in a fixed order,
// then a fixed shuffle tree.
// du, dv_bias from the partials part [n_part][H][2][D] (d(q+u) columns, then
// d(q+v)): a block takes 32 adjacent columns; warp w adds partials w,
// w + 32, ... of its lane's column (coalesced rows), then the 32 warp sums
// are added in warp order, so the order is fixed.
__global__ void bwd_bias_kernel(const float* __restrict__ part, int n_part, int H, int D, float* __restrict__ du,
                                float* __restrict__ dvb) {
  grid_dep_wait();  // launched behind the kernel that writes the partials
  __shared__ float red[32][32];
  const int lane = threadIdx.x & 31, wp = threadIdx.x >> 5;
  const int ncol = H * 2 * D;
  const int col = blockIdx.x * 32 + lane;
  float s = 0.f;
  if (col < ncol) {
#pragma unroll 4
    for (int q = wp; q < n_part; q += 32) s += part[static_cast<long long>(q) * ncol + col];
  }
  red[wp][lane] = s;
  __syncthreads();
  if (wp == 0 && col < ncol) {
    float t = 0.f;
#pragma unroll
    for (int k = 0; k < 32; ++k) t += red[k][lane];
    const int h = col / (2 * D), x = col % (2 * D);
    if (x < D)
      du[h * D + x] = t;
    else
      dvb[h * D + x - D] = t;
  }
}

template <typename T, typename TG>
cudaError_t launch_typed(BwdArgs a, float* du, float* dvb, cudaStream_t stream) {
  const int nb = (a.W + kWarps - 1) / kWarps;
  bwd_delta_kernel<TG><<<dim3(nb, a.H, a.B), kThreads, 0, stream>>>(a);
  bwd_dq_kernel<T, TG><<<dim3(nb, a.H, a.B), kThreads, sizeof(float) * (kWarps * 5 * a.D), stream>>>(a);
  bwd_dkdv_kernel<T, TG><<<dim3(nb, a.H, a.B), kThreads, sizeof(float) * (kWarps * 2 + 2) * a.D, stream>>>(a);
  bwd_dr_kernel<T, TG><<<dim3((a.n_r + kWarps - 1) / kWarps, a.H), kThreads, sizeof(float) * (kWarps + 2) * a.D,
                         stream>>>(a);
  bwd_bias_kernel<<<(a.H * 2 * a.D + 31) / 32, 1024, 0, stream>>>(a.part, a.B * nb, a.H, a.D, du,
                                                                   dvb);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_bias(const float* part, int n_part, int H, int D, float* du, float* dvb,
                            cudaStream_t stream) {
  return launch_dependent(bwd_bias_kernel, dim3((H * 2 * D + 31) / 32), dim3(1024), 0, stream, part, n_part, H, D,
                          du, dvb);
}

size_t relattn_bwd_simt_scratch_bytes(int B, int W, int H, int D) {
  const size_t nb = (static_cast<size_t>(W) + kWarps - 1) / kWarps;
  return sizeof(float) * (static_cast<size_t>(B) * H * W + static_cast<size_t>(B) * nb * H * 2 * D);
}

cudaError_t launch_relattn_bwd_simt(const void* q, const void* k, const void* v, const void* r,
                                    const float* bias_u, const float* bias_v, const void* o, const float* lse,
                                    const void* dout, float* dq, float* dk, float* dv, float* dr, float* du,
                                    float* dvb, int B, int W, int M, int H, int D, int n_r, float scale, bool bf16,
                                    bool go_bf16, bool vec16, void* scratch, cudaStream_t stream) {
  BwdArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.r = r;
  a.bias_u = bias_u;
  a.bias_v = bias_v;
  a.o = o;
  a.lse = lse;
  a.dout = dout;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.dr = dr;
  a.delta = static_cast<float*>(scratch);
  a.part = a.delta + static_cast<size_t>(B) * H * W;
  a.B = B;
  a.W = W;
  a.M = M;
  a.H = H;
  a.D = D;
  a.n_r = n_r;
  a.scale = scale;
  a.vec16 = vec16;
  if (bf16)
    return go_bf16 ? launch_typed<__nv_bfloat16, __nv_bfloat16>(a, du, dvb, stream)
                   : launch_typed<__nv_bfloat16, float>(a, du, dvb, stream);
  return go_bf16 ? launch_typed<float, __nv_bfloat16>(a, du, dvb, stream)
                 : launch_typed<float, float>(a, du, dvb, stream);
}

}  // namespace txl
