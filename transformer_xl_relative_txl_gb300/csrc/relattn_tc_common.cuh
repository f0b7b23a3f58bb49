// Device helpers shared by the tensor-core relative-attention kernels: the
// per-lane distance-window shift, mixed-precision adds, warp-level waits and
// arrivals, and the persistent work-unit decoding.
#pragma once

#include <cstdint>

#include "txl_device.cuh"

namespace txl {

constexpr int kTileRows = 128;  // query rows per unit (TMEM lanes)
constexpr int kStepKeys = 64;   // keys per step, distances per ring tile

// A (batch, head, 128-query tile) unit, or a chunk of one: key steps
// [t0, t0 + nks) of the tile's visible range.
struct Unit {
  int b, h, i0, nks;
  int t0;
};

// Units are ordered longest query tile first; u in [0, nqt * B * H).
__host__ __device__ __forceinline__ Unit decode_unit(int u, int B, int H, int W, int M, int nqt) {
  const int BH = B * H;
  const int qt = nqt - 1 - u / BH;
  const int bh = u % BH;
  Unit r;
  r.b = bh / H;
  r.h = bh % H;
  r.i0 = qt * kTileRows;
  const int kmax = min(M + r.i0 + kTileRows - 1, M + W - 1);
  r.nks = kmax / kStepKeys + 1;
  r.t0 = 0;
  return r;
}

// Work item it of a launch whose units are split into nsplit chunks of
// their key steps (chunk c of unit it / nsplit: steps [c*n/nsplit,
// (c+1)*n/nsplit)); nsplit never exceeds a unit's step count.
__host__ __device__ __forceinline__ Unit decode_item(int it, int nsplit, int B, int H, int W, int M, int nqt) {
  Unit r = decode_unit(it / nsplit, B, H, W, M, nqt);
  if (nsplit > 1) {
    const int c = it % nsplit;
    const int lo = (c * r.nks) / nsplit, hi = ((c + 1) * r.nks) / nsplit;
    r.t0 = lo;
    r.nks = hi - lo;
  }
  return r;
}

// Unit of round r for CTA c of P: units are sorted longest first and dealt
// in a snake order (c, then 2P-1-c, then 2P+c, ...), which pairs long units
// with short ones.  Returns a value >= n_units once the CTA has no more (and
// every later round is then past the end as well).
__device__ __forceinline__ int sched_unit(int r, int c, int P) {
  return r * P + ((r & 1) ? P - 1 - c : c);
}

// Unit of round r for CTA c: from a host-made table when there is one (row c
// of `stride` unit indices, -1 past the CTA's last unit), else the snake
// order.  Returns n_units once the CTA has no more.
__device__ __forceinline__ int unit_at(const int* sched, int stride, int r, int c, int P, int n_units) {
  if (sched == nullptr) return sched_unit(r, c, P);
  if (r >= stride) return n_units;
  const int u = __ldg(sched + c * stride + r);
  return u < 0 ? n_units : u;
}

__device__ __forceinline__ uint32_t byte_perm(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// fp32 + bf16 (low or high half of a packed pair), one rounding.
__device__ __forceinline__ float add_bf16lo(uint32_t pk, float s) {
  float r;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tadd.rn.f32.bf16 %0, lo, %2;\n\t}"
      : "=f"(r) : "r"(pk), "f"(s));
  return r;
}
__device__ __forceinline__ float add_bf16hi(uint32_t pk, float s) {
  float r;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tadd.rn.f32.bf16 %0, hi, %2;\n\t}"
      : "=f"(r) : "r"(pk), "f"(s));
  return r;
}

__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Per-lane window shift on bf16 pairs.  lo, hi hold the window X[0..63]
// packed two per register (X[2i] in the low half); on return out[j] packs
// (Y[2j], Y[2j+1]) with Y[k] = X[lane + 1 + k], k = 0..31.  Whole registers
// move by a five-stage select network on (lane + 1) / 2; the odd half-register
// remainder is one byte permute.
__device__ __forceinline__ void window_shift_packed(const uint32_t (&lo)[16], const uint32_t (&hi)[16], int lane,
                                                    uint32_t (&out)[16]) {
  uint32_t R[32];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    R[i] = lo[i];
    R[16 + i] = hi[i];
  }
  const int sh = lane + 1;
  const int q = sh >> 1;
  const bool b16 = q & 16, b8 = q & 8, b4 = q & 4, b2 = q & 2, b1 = q & 1;
#pragma unroll
  for (int j = 0; j <= 15; ++j) R[j] = b16 ? R[j + 16] : R[j];
#pragma unroll
  for (int j = 0; j <= 23; ++j) R[j] = b8 ? R[j + 8] : R[j];
#pragma unroll
  for (int j = 0; j <= 19; ++j) R[j] = b4 ? R[j + 4] : R[j];
#pragma unroll
  for (int j = 0; j <= 17; ++j) R[j] = b2 ? R[j + 2] : R[j];
#pragma unroll
  for (int j = 0; j <= 16; ++j) R[j] = b1 ? R[j + 1] : R[j];
  const uint32_t sel = (sh & 1) ? 0x5432u : 0x3210u;
#pragma unroll
  for (int j = 0; j < 16; ++j) out[j] = byte_perm(R[j], R[j + 1], sel);
}

// 32 fp32 values -> 16 bf16 pairs (round to nearest even).
__device__ __forceinline__ void pack32(const uint32_t (&x)[32], uint32_t (&out)[16]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) out[i] = pack_bf16x2(__uint_as_float(x[2 * i]), __uint_as_float(x[2 * i + 1]));
}

// Window shift of an fp32 window held in two 32-column TMEM loads.
__device__ __forceinline__ void window_shift(const uint32_t (&x0)[32], const uint32_t (&x1)[32], int lane,
                                             uint32_t (&out)[16]) {
  uint32_t lo[16], hi[16];
  pack32(x0, lo);
  pack32(x1, hi);
  window_shift_packed(lo, hi, lane, out);
}

// x[k] = s[k] + (distance term of column k), the distance value of column k
// sitting at shifted-window position 31 - k.
__device__ __forceinline__ void add_window(const uint32_t (&sraw)[32], const uint32_t (&bd)[16], float* x) {
#pragma unroll
  for (int k = 0; k < 32; ++k) {
    const int i = 31 - k;
    x[k] = (i & 1) ? add_bf16hi(bd[i >> 1], __uint_as_float(sraw[k])) : add_bf16lo(bd[i >> 1], __uint_as_float(sraw[k]));
  }
}

// The backward's per-pair terms for 32 key columns of one query row (lane
// `lane` of lane quadrant `quad`; columns [32 half, 32 half + 32) of a 64-key
// step).  TMEM holds the step's unscaled content scores at column colS, the
// dout . v_j products at colDP and the 192-distance window (q+v) . r_d at
// colWin.  The window is shifted into key order as in the forward, then
//   p = 2^(s scale log2(e) - lse2)   (lse2: the row's lse in log2 units)
//   g = scale p (dout . v_j - delta)
// where visible(c) is false for masked columns c (p = g = 0 there).
//
// step_grads_half_at takes the TMEM columns of the two 32-column window
// chunks (positions w0 and w0 + 32, w0 = 32 quad + (half ? 0 : 32)) as
// arguments, for windows that are not contiguous in TMEM.
template <typename Vis>
__device__ __forceinline__ void step_grads_half_at(uint32_t tmem, uint32_t colS, uint32_t colDP, uint32_t colW0,
                                                   uint32_t colW1, int quad, int half, int lane, float lse2,
                                                   float delta, float scale, float scale_log2e, Vis visible,
                                                   float (&g)[32], float (&p)[32]) {
  const uint32_t lb = tmem + (static_cast<uint32_t>(quad * 32) << 16);
  uint32_t bd[16], sx[32], dpv[32];
  {
    uint32_t xlo[32], xhi[32];
    tmem_ld32(lb + colW0, xlo);
    tmem_ld32(lb + colW1, xhi);
    tmem_ld32(lb + colS + 32 * half, sx);
    tmem_ld32(lb + colDP + 32 * half, dpv);
    tmem_wait_ld(xlo);
    tmem_wait_ld(xhi);
    tmem_wait_ld(sx);
    tmem_wait_ld(dpv);
    uint32_t plo[16], phi[16];
    pack32(xlo, plo);
    pack32(xhi, phi);
    window_shift_packed(plo, phi, lane, bd);
  }
  add_window(sx, bd, p);
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    const float e = visible(32 * half + c) ? ex2(fmaf(p[c], scale_log2e, -lse2)) : 0.f;
    p[c] = e;
    g[c] = scale * e * (__uint_as_float(dpv[c]) - delta);
  }
}

template <typename Vis>
__device__ __forceinline__ void step_grads_half(uint32_t tmem, uint32_t colS, uint32_t colDP, uint32_t colWin,
                                                int quad, int half, int lane, float lse2, float delta, float scale,
                                                float scale_log2e, Vis visible, float (&g)[32], float (&p)[32]) {
  // key columns 0-31 use window positions [32 quad + 32, 32 quad + 96),
  // columns 32-63 [32 quad, 32 quad + 64)
  const uint32_t w0 = colWin + 32 * quad + (half ? 0 : 32);
  step_grads_half_at(tmem, colS, colDP, w0, w0 + 32, quad, half, lane, lse2, delta, scale, scale_log2e, visible, g,
                     p);
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, uint64_t ns, volatile int* abort) {
  const bool got = mbar_wait(bar, parity, ns, abort);
  return __all_sync(0xffffffffu, got);
}

// Elected-lane arrive after every lane's tcgen05 accesses are complete.
__device__ __forceinline__ void warp_arrive_tc(uint64_t* bar) {
  tc_fence_before();
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

// Elected-lane arrive after every lane's shared-memory writes are made
// visible to the async proxy (the tensor core reads them next).
__device__ __forceinline__ void warp_arrive_smem(uint64_t* bar) {
  fence_proxy_async_smem();
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

// Elected-lane arrive after every lane's generic accesses.
__device__ __forceinline__ void warp_arrive(uint64_t* bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

}  // namespace txl
