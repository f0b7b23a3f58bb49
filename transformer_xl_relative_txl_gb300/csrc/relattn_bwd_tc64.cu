// Backward of the relative attention on the tensor cores: bf16 q, k, v, r,
// o and dout, D = 64, fp32 accumulation and gradients.
//
// The gradients (see relattn_bwd.cu for the formulas and the stop-gradient)
// come from two kernels that each rebuild the scores of the forward:
//
//   dq kernel, one CTA per 128-query tile of a (batch, head), 64-key steps:
//     S = (q+u) K^T, dP = dout V^T and the 192-distance window (q+v) R^T of
//     the step (three MMAs); each thread owns one query row (TMEM lane) and
//     forms p = exp(s - lse), g = scale p (dP - Delta), with the distance
//     term shifted into key order as in the forward.  g goes to shared
//     memory twice: in key order (G, the A operand of d(q+u) += G K) and
//     skewed into distance order (Gs: row i, column d = M+i-j).  A distance
//     slot of 64 rows receives its last values two steps after its first;
//     then d(q+v) += Gs R and dr += Gs^T (q+v) (an M = 64 MMA) run on it, and
//     the slot's dr rows are staged in shared memory and added to the output
//     by one TMA bulk reduction (fp32 vector atomics for a slot that starts
//     below distance 0).
//   dk/dv kernel, one CTA per 64 segment keys of a (batch, head), looping
//     over the 128-query tiles that see them: the same three MMAs and the
//     same p, g; then dV += P^T dout and dK += G^T (q+u) with P and G read
//     as MN-major A operands (M = 64 keys).
//
// Both kernels are synchronous: thread 0 issues the TMA loads (double
// buffered, one step ahead) and the MMAs; all 128 threads wait on the MMA
// barriers.  Every wait is bounded; a timeout raises the device status word
// and the CTA drains its own copies and MMAs before it exits.
//
// TMEM (512 columns): S [0, 64), dP [64, 128), distance window [128, 320)
// (reused for the dr slot result, M = 64 layout), d(q+u) or dV [320, 384),
// d(q+v) or dK [384, 448).  An M = 64 result keeps its row r in lane
// 32 (r / 16) + r % 16.
#include <cuda.h>
#include <cuda_bf16.h>

#include <cstdint>

#include "pdl.cuh"
#include "relattn_tc_common.cuh"
#include "txl_device.cuh"
#include "txl_internal.h"

namespace txl {
namespace {

constexpr int D = 64;
constexpr int BM = 128;     // query rows per tile
constexpr int BN = 64;      // keys per step / block
constexpr int kWin = 192;   // distance rows of a step's window
constexpr int kTile = BM * 128;          // 128 rows x 64 bf16
constexpr int kKTile = BN * 128;         // 64 rows x 64 bf16
constexpr int kWinTile = kWin * 128;     // 192 rows x 64 bf16
constexpr uint32_t kColS = 0, kColDP = 64, kColWin = 128, kColA = 320, kColB = 384, kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;

// dq kernel shared memory
constexpr int kQOffQu = 0;
constexpr int kQOffQv = kQOffQu + kTile;
constexpr int kQOffDO = kQOffQv + kTile;
constexpr int kQOffK = kQOffDO + kTile;          // 2 stages
constexpr int kQOffV = kQOffK + 2 * kKTile;      // 2 stages
constexpr int kQOffR = kQOffV + 2 * kKTile;      // 2 stages
constexpr int kQOffG = kQOffR + 2 * kWinTile;    // G in key order (also the raw q tile at the start)
constexpr int kQOffGs = kQOffG + kTile;          // 4 distance slots
constexpr int kQOffDr = kQOffGs + 4 * kTile;     // a finished slot's dr rows: 2 boxes [64][32] fp32, 128B-swizzled
constexpr int kQOffBar = kQOffDr + BN * D * 4;
constexpr int kQOffBias = kQOffBar + 256;        // u, then v of the head (fp32)
constexpr int kQSmem = kQOffBias + 2 * 64 * 4 + 1024;
static_assert(kQSmem <= 232448, "shared memory budget");

// dk/dv kernel shared memory
constexpr int kKOffK = 0;
constexpr int kKOffV = kKOffK + kKTile;
constexpr int kKOffQu = kKOffV + kKTile;         // 2 buffers
constexpr int kKOffQv = kKOffQu + 2 * kTile;     // 2 buffers
constexpr int kKOffQ = kKOffQv + 2 * kTile;      // raw q, 2 stages
constexpr int kKOffDO = kKOffQ + 2 * kTile;      // 2 stages
constexpr int kKOffR = kKOffDO + 2 * kTile;      // 2 stages
constexpr int kKOffP = kKOffR + 2 * kWinTile;
constexpr int kKOffG = kKOffP + kTile;
constexpr int kKOffBar = kKOffG + kTile;
constexpr int kKOffBias = kKOffBar + 256;        // per item parity: u, then v of the item's head (fp32)
constexpr int kKSmem = kKOffBias + 2 * 2 * 64 * 4 + 1024;
static_assert(kKSmem <= 232448, "shared memory budget");

struct BwdParams {
  const float* bias_u;
  const float* bias_v;
  const float* lse;         // [B, H, W]
  const __nv_bfloat16* o;   // [B, W, H, D]
  const __nv_bfloat16* dout;
  float* dq;                // [B, W, H, D]
  float* dk;                // [B, W, H, D]
  float* dv;
  float* dr;                // [n_r, H, D], zeroed before the dq kernel
  float* delta;             // [B, H, W] scratch: written by the dq kernel, read by the dk/dv kernel
  float* part;              // [B * nqt][H][2][D] scratch: per-tile sums of d(q+u), d(q+v)
  int B, W, M, H, n_r, nqt;
  float scale, scale_log2e;
  unsigned int* status;
  unsigned long long wait_ns;
  int inject_stall;  // test hook: the dq kernel's issuer loads nothing past the first two steps
};

struct QBars {
  uint64_t q, kv[2], r[2], m1, m2[2], gready, fin, fin2;
  uint32_t tmem_base;
  int abort;
};
struct KBars {
  uint64_t kv, in[2], m1, m2, fin;
  uint32_t tmem_base;
  int abort;
};

// Byte offset of bf16 element (row, col) in a 128B-swizzled tile of 64-column rows.
__device__ __forceinline__ uint32_t swz(int row, int col) {
  return static_cast<uint32_t>((row >> 3) * 1024 + (row & 7) * 128 + ((((col >> 3) ^ (row & 7))) << 4) +
                               ((col & 7) << 1));
}

// Chunks [4 half, 4 half + 4) (head dims 32 half .. 32 half + 31) of row a
// of (q+u) and (q+v); bu, bv: the head's u and v staged in shared memory.
__device__ __forceinline__ void build_qu_qv_half(const uint8_t* sQ, uint8_t* sQu, uint8_t* sQv, int a, int half,
                                                 const float* bu, const float* bv) {
#pragma unroll
  for (int cc = 0; cc < 4; ++cc) {
    const int c = 4 * half + cc;
    const uint32_t off = (a >> 3) * 1024 + (a & 7) * 128 + ((c ^ (a & 7)) << 4);
    const uint4 raw = *reinterpret_cast<const uint4*>(sQ + off);
    const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
    const float4 u0 = *reinterpret_cast<const float4*>(bu + 8 * c);
    const float4 u1 = *reinterpret_cast<const float4*>(bu + 8 * c + 4);
    const float4 v0 = *reinterpret_cast<const float4*>(bv + 8 * c);
    const float4 v1 = *reinterpret_cast<const float4*>(bv + 8 * c + 4);
    const float ub[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
    const float vb[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    uint32_t qu[4], qv[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float x0 = bf16_lo(w4[e]), x1 = bf16_hi(w4[e]);
      qu[e] = pack_bf16x2(x0 + ub[2 * e], x1 + ub[2 * e + 1]);
      qv[e] = pack_bf16x2(x0 + vb[2 * e], x1 + vb[2 * e + 1]);
    }
    *reinterpret_cast<uint4*>(sQu + off) = make_uint4(qu[0], qu[1], qu[2], qu[3]);
    *reinterpret_cast<uint4*>(sQv + off) = make_uint4(qv[0], qv[1], qv[2], qv[3]);
  }
}

// dst[0..3] += (x0..x3) (fp32 bit patterns), one vector reduction in L2 with
// no value returned.
__device__ __forceinline__ void red_add_v4(float* dst, uint32_t x0, uint32_t x1, uint32_t x2, uint32_t x3) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "r"(x0), "r"(x1), "r"(x2), "r"(x3)
               : "memory");
}

// Delta_i = dout_i . o_i over the 64 bf16 of each row.
__device__ __forceinline__ float row_delta(const __nv_bfloat16* o, const __nv_bfloat16* g) {
  float s0 = 0.f, s1 = 0.f;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint4 a = __ldg(reinterpret_cast<const uint4*>(o) + c);
    const uint4 b = __ldg(reinterpret_cast<const uint4*>(g) + c);
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      s0 = fmaf(bf16_lo(aw[e]), bf16_lo(bw[e]), s0);
      s1 = fmaf(bf16_hi(aw[e]), bf16_hi(bw[e]), s1);
    }
  }
  return s0 + s1;
}

// ============================================================================
// dq kernel: 8 warps, two per TMEM lane quadrant (key columns 0-31 and
// 32-63 of the same rows).  Per step t, after the gradients of step t are in
// shared memory, thread 0 issues the step's d(q+u) / slot MMAs and right
// behind them the score MMAs of step t+1; the dr rows of the finished slot
// are flushed while those run.
// ============================================================================
constexpr int kQThreads = 256;
constexpr int kIssuer2 = 128;  // lane 0 of warp 4: the dq kernel's gradient / slot MMAs
// The dq kernel adds warp 8, whose lane 0 issues the loads and the score MMAs
// outside the pair warps' barriers.
constexpr int kDqIssuer = kQThreads;
constexpr int kDqThreads = kQThreads + 32;
constexpr uint32_t kColDr = 448;  // the finished slot's dr rows (M = 64 layout)

// Columns [32 half, 32 half + 32) of row a of a 128B-swizzled [128 x 64] bf16 tile.
__device__ __forceinline__ void store_row_half(uint8_t* tile, int a, int half, const float (&x)[32]) {
  uint8_t* row = tile + (a >> 3) * 1024 + (a & 7) * 128;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint32_t w0 = pack_bf16x2(x[8 * c], x[8 * c + 1]), w1 = pack_bf16x2(x[8 * c + 2], x[8 * c + 3]);
    const uint32_t w2 = pack_bf16x2(x[8 * c + 4], x[8 * c + 5]), w3 = pack_bf16x2(x[8 * c + 6], x[8 * c + 7]);
    *reinterpret_cast<uint4*>(row + (((4 * half + c) ^ (a & 7)) << 4)) = make_uint4(w0, w1, w2, w3);
  }
}

__global__ void __launch_bounds__(kDqThreads, 1)
    bwd_dq_tc64_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_rw,
                       const __grid_constant__ CUtensorMap tm_do, const __grid_constant__ CUtensorMap tm_dr,
                       const BwdParams p) {
  grid_dep_wait();  // launched behind the previous kernel on the stream: it has completed from here on
  grid_dep_launch_dependents();  // the dk/dv kernel's CTAs may take SMs this launch no longer needs
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  uint8_t* sQu = smem + kQOffQu;
  uint8_t* sQv = smem + kQOffQv;
  uint8_t* sDO = smem + kQOffDO;
  uint8_t* sK = smem + kQOffK;
  uint8_t* sV = smem + kQOffV;
  uint8_t* sR = smem + kQOffR;
  uint8_t* sG = smem + kQOffG;
  uint8_t* sGs = smem + kQOffGs;
  QBars* bars = reinterpret_cast<QBars*>(smem + kQOffBar);
  float* sBias = reinterpret_cast<float*>(smem + kQOffBias);
  uint8_t* sDr = smem + kQOffDr;
  volatile int* abort = &bars->abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quad = warp & 3, half = warp >> 2;
  const int a = quad * 32 + lane;  // this thread's row of the tile
  const uint64_t wait_ns = p.wait_ns;

  const Unit w = decode_unit(blockIdx.x, p.B, p.H, p.W, p.M, p.nqt);
  const int T = w.nks;
  const int i = w.i0 + a;  // query row
  const int L = p.M + p.W;

  // Window of step t: distance rows [wb(t), wb(t) + 192), wb = M + i0 - 64 t - 64.
  auto wbase = [&](int t) { return p.M + w.i0 - BN * t - BN; };
  uint32_t n_ld[2] = {0, 0};  // loads issued per stage (the issuer)
  auto issue_step_loads = [&](int t) {
    const int s = t & 1;
    mbar_arrive_expect_tx(&bars->kv[s], 2 * kKTile);
    tma_load_4d(sK + s * kKTile, &tm_k, &bars->kv[s], 0, w.h, BN * t, w.b);
    tma_load_4d(sV + s * kKTile, &tm_v, &bars->kv[s], 0, w.h, BN * t, w.b);
    mbar_arrive_expect_tx(&bars->r[s], kWinTile);
    tma_load_3d(sR + s * kWinTile, &tm_rw, &bars->r[s], 0, w.h, wbase(t));
    ++n_ld[s];
  };
  // The issuer starts the unit's loads first thing (it owns their barriers);
  // the block barrier below makes its initialisation visible to the waiters.
  if (tid == kDqIssuer) {
    mbar_init(&bars->q, 1);
    mbar_init(&bars->kv[0], 1);
    mbar_init(&bars->kv[1], 1);
    mbar_init(&bars->r[0], 1);
    mbar_init(&bars->r[1], 1);
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_rw);
    tma_prefetch_desc(&tm_do);
    tma_prefetch_desc(&tm_dr);
    mbar_arrive_expect_tx(&bars->q, 2 * kTile);
    tma_load_4d(sG, &tm_q, &bars->q, 0, w.h, w.i0, w.b);  // raw q, into the G tile for now
    tma_load_4d(sDO, &tm_do, &bars->q, 0, w.h, w.i0, w.b);
    issue_step_loads(0);
    if (T > 1) issue_step_loads(1);
  } else if (tid == 0) {
    mbar_init(&bars->m1, 1);
    mbar_init(&bars->m2[0], 1);
    mbar_init(&bars->m2[1], 1);
    mbar_init(&bars->gready, 1);
    mbar_init(&bars->fin, 1);
    mbar_init(&bars->fin2, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (tid < 2 * D) sBias[tid] = tid < D ? p.bias_u[w.h * D + tid] : p.bias_v[w.h * D + tid - D];
  // Per-row constants: lse (log2 domain) and Delta.
  const long long row_id = (static_cast<long long>(w.b) * p.H + w.h) * p.W + i;
  float lse2 = INFINITY, delta = 0.f;  // rows past W: every p is 0
  const bool pair = tid < kQThreads;  // warps 0-7
  if (pair && i < p.W) {
    lse2 = p.lse[row_id] * kLog2e;
    const long long off = ((static_cast<long long>(w.b) * p.W + i) * p.H + w.h) * D;
    delta = row_delta(p.o + off, p.dout + off);
    if (half == 0) p.delta[row_id] = delta;
  }
  // Distance slots start at zero: a slot entry no step writes is a pair
  // that does not exist.
  for (int x = tid; x < 4 * kTile / 16; x += kDqThreads)
    reinterpret_cast<uint4*>(sGs)[x] = make_uint4(0u, 0u, 0u, 0u);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  bool ok = true;
  if (pair) {
    ok = mbar_wait(&bars->q, 0, wait_ns, abort);
    if (ok) build_qu_qv_half(sG, sQu, sQv, a, half, sBias, sBias + D);
    else report_timeout(abort, p.status);
    fence_proxy_async_smem();
  }
  ok = __syncthreads_and(ok) != 0;

  constexpr uint32_t id64 = idesc_bf16(128, 64, false, false);
  constexpr uint32_t id192 = idesc_bf16(128, 192, false, false);
  constexpr uint32_t idMN = idesc_bf16(128, 64, false, true);   // B MN-major
  constexpr uint32_t idT = idesc_bf16(64, 64, true, true);      // A and B MN-major, M = 64
  const uint64_t dQu = sdesc_sw128(smem_u32(sQu), 16, 1024);
  const uint64_t dQv = sdesc_sw128(smem_u32(sQv), 16, 1024);
  const uint64_t dDO = sdesc_sw128(smem_u32(sDO), 16, 1024);
  const uint64_t dG = sdesc_sw128(smem_u32(sG), 16, 1024);
  const uint64_t dQvMN = sdesc_sw128(smem_u32(sQv), 8192, 1024);
  int n_slot = 0;     // distance slots issued (the slot issuer, kIssuer2)

  // The issuer: the score MMAs of step t (S, dP, distance window).
  auto score_mmas = [&](int t) -> bool {
    const int s = t & 1;
    if (!mbar_wait(&bars->kv[s], (t >> 1) & 1, wait_ns, abort) ||
        !mbar_wait(&bars->r[s], (t >> 1) & 1, wait_ns, abort))
      return false;
    tc_fence_after();
    const uint64_t dK = sdesc_sw128(smem_u32(sK + s * kKTile), 16, 1024);
    const uint64_t dV = sdesc_sw128(smem_u32(sV + s * kKTile), 16, 1024);
    const uint64_t dR = sdesc_sw128(smem_u32(sR + s * kWinTile), 16, 1024);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) mma_ss(tmem + kColS, dQu + 2 * kk, dK + 2 * kk, id64, kk > 0);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) mma_ss(tmem + kColDP, dDO + 2 * kk, dV + 2 * kk, id64, kk > 0);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) mma_ss(tmem + kColWin, dQv + 2 * kk, dR + 2 * kk, id192, kk > 0);
    tc_commit(&bars->m1);
    return true;
  };
  // kIssuer2: d(q+v) += Gs R and dr_slot = Gs^T (q+v) for distance slot tau,
  // whose R rows are rows [64 r_row, 64 r_row + 64) of window stage rs.
  auto slot_mmas = [&](int tau, int rs, int r_row) {
    const int gi = (tau + 2) & 3;
    const uint64_t dGs = sdesc_sw128(smem_u32(sGs + gi * kTile), 16, 1024);
    const uint64_t dGsT = sdesc_sw128(smem_u32(sGs + gi * kTile), 8192, 1024);
    const uint64_t dRs = sdesc_sw128(smem_u32(sR + rs * kWinTile + r_row * kKTile), 8192, 1024);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) mma_ss(tmem + kColB, dGs + 2 * kk, dRs + 128 * kk, idMN, n_slot > 0 || kk > 0);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) mma_ss(tmem + kColDr, dGsT + 128 * kk, dQvMN + 128 * kk, idT, kk > 0);
    ++n_slot;
  };
  // Everyone: the dr rows of slot tau (TMEM, M = 64 layout: row 16 quad +
  // lane in lanes 0-15 of each quadrant; this warp takes head dims
  // [32 half, 32 half + 32)), distance rows d0 .. d0 + 63.  A slot that starts
  // at d0 >= 0 is staged in sDr, box `half` holding dims [32 half, +32) as 64
  // rows of 128 bytes with 16-byte chunk c of row r at chunk c ^ (r & 7) (the
  // TMA's 128-byte swizzle: two lanes a bank group), for two TMA reductions
  // that thread 0 issues after the next block barrier; rows past the tensor
  // are dropped by the TMA, and rows from M+W on hold zeros (no query row
  // reaches them).  A slot that straddles distance 0 adds its rows d >= 0
  // with vector atomics.  Returns whether reductions are pending.
  auto stage_dr = [&](int tau) -> bool {
    const int d0 = p.M + w.i0 - BN * tau - BN;
    if (d0 + BN <= 0) return false;
    uint32_t v[32];
    tmem_ld32(tmem + (static_cast<uint32_t>(quad * 32) << 16) + kColDr + 32 * half, v);
    tmem_wait_ld(v);
    const int rr = 16 * quad + lane;
    const int d = d0 + rr;
    if (d0 < 0) {
      if (lane < 16 && d >= 0 && d < L) {
        float* dst = p.dr + (static_cast<long long>(d) * p.H + w.h) * D + 32 * half;
#pragma unroll
        for (int e = 0; e < 8; ++e) red_add_v4(dst + 4 * e, v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
      }
      return false;
    }
    if (lane < 16) {
      uint8_t* row = sDr + half * (BN * 128) + rr * 128;
#pragma unroll
      for (int e = 0; e < 8; ++e)
        *reinterpret_cast<uint4*>(row + ((e ^ (rr & 7)) << 4)) = make_uint4(v[4 * e], v[4 * e + 1], v[4 * e + 2],
                                                                             v[4 * e + 3]);
    }
    fence_proxy_async_smem();
    return true;
  };
  int dr_d0 = -1;  // distance row of the staged slot awaiting its reduction (-1: none)
  // Thread 0, after a block barrier that follows the staging: the reduction.
  auto issue_dr = [&]() {
    if (dr_d0 >= 0) {
      tma_reduce_add_3d(&tm_dr, sDr, 0, w.h, dr_d0);
      tma_reduce_add_3d(&tm_dr, sDr + BN * 128, 32, w.h, dr_d0);
      bulk_commit_group();
    }
    dr_d0 = -1;
  };
  auto flush_dr = [&](int tau) {
    if (stage_dr(tau)) dr_d0 = p.M + w.i0 - BN * tau - BN;
  };

  // Barrier phases cannot be skipped: the score MMAs of step t+1 wait for
  // the pairs of step t (gready), the loads of step t+2 for step t's
  // gradient MMAs (m2), and each of those is what lets the next phase of the
  // same barrier happen.
  if (tid == kDqIssuer) {
    // ============================ issuer ==================================
    if (ok) ok = score_mmas(0);
    for (int t = 0; t < T && ok; ++t) {
      if (t + 1 < T) {
        // the pairs of step t have read S, dP and the window
        if (!(ok = mbar_wait(&bars->gready, t & 1, wait_ns, abort))) break;
        tc_fence_after();
        if (!(ok = score_mmas(t + 1))) break;
      }
      if (t + 2 < T && !p.inject_stall) {
        // step t's gradient MMAs have read K and the window of stage t & 1
        if (!(ok = mbar_wait(&bars->m2[t & 1], (t >> 1) & 1, wait_ns, abort))) break;
        issue_step_loads(t + 2);
      }
    }
    if (!ok) report_timeout(abort, p.status);
    // Let this thread's copies and MMAs finish before the memory is released.
    for (int s = 0; s < 2; ++s)
      if (n_ld[s] > 0) mbar_wait_own(&bars->kv[s], (n_ld[s] - 1) & 1, wait_ns);
    for (int s = 0; s < 2; ++s)
      if (n_ld[s] > 0) mbar_wait_own(&bars->r[s], (n_ld[s] - 1) & 1, wait_ns);
    mbar_wait_own(&bars->q, 0, wait_ns);
    tc_commit(&bars->fin);
    mbar_wait_own(&bars->fin, 0, wait_ns);
  } else if (pair) {
    // ============================ pairs ===================================
    // m2 commits c = 0, 1, ...: one per step, then the last two slots; commit
    // c lands on m2[c & 1] with parity (c >> 1) & 1.
    for (int t = 0; t < T && ok; ++t) {
      const int s = t & 1;
      // (1) the step's gradients into G (key order) and the slots; thread 0
      // hands the slot staged at the end of the last step to the TMA.
      ok = mbar_wait(&bars->m1, t & 1, wait_ns, abort);
      if (!named_bar_and(1, kQThreads, ok)) {
        ok = false;
        break;
      }
      if (tid == 0) issue_dr();
      tc_fence_after();
      {
        float g[32], pr[32];
        const int lim = p.M + i - BN * t;  // key column c visible iff c <= lim
        step_grads_half(tmem, kColS, kColDP, kColWin, quad, half, lane, lse2, delta, p.scale, p.scale_log2e,
                        [&](int c) { return c <= lim; }, g, pr);
        store_row_half(sG, a, half, g);
        // Skewed copy: key column c of step t sits at window position
        // z = 64 + a - c, i.e. in distance slot t - z / 64, column z % 64.
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int z = 64 + a - (32 * half + c);
          const int gi = (t - (z >> 6) + 2) & 3;
          *reinterpret_cast<__nv_bfloat16*>(sGs + gi * kTile + swz(a, z & 63)) = __float2bfloat16_rn(g[c]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      named_bar_sync(1, kQThreads);
      // (2) the issuer goes on with the next step's score MMAs; kIssuer2
      // issues d(q+u) += G K and the slot step t finished (t-2).
      if (tid == 0) {
        mbar_arrive(&bars->gready);
      } else if (tid == kIssuer2) {
        tc_fence_after();
        const uint64_t dKmn = sdesc_sw128(smem_u32(sK + s * kKTile), 8192, 1024);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) mma_ss(tmem + kColA, dG + 2 * kk, dKmn + 128 * kk, idMN, t > 0 || kk > 0);
        slot_mmas(t - 2, s, 2);
        tc_commit(&bars->m2[t & 1]);
      }
      // (3) flush the slot's dr rows; the slot's buffer is free again and
      // becomes slot t+2.  sDr is free once the last reduction has read it.
      if (tid == 0) bulk_wait_group_read0();
      ok = mbar_wait(&bars->m2[t & 1], (t >> 1) & 1, wait_ns, abort);
      if (!named_bar_and(1, kQThreads, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      flush_dr(t - 2);
      {
        uint4* nxt = reinterpret_cast<uint4*>(sGs + (t & 3) * kTile);
        for (int x = tid; x < kTile / 16; x += kQThreads) nxt[x] = make_uint4(0u, 0u, 0u, 0u);
      }
      tc_fence_before();
    }
    // The last two slots are finished once the last step has written them.
    for (int k = 0; k < 2 && ok; ++k) {
      const int tau = T - 2 + k, c = T + k;
      named_bar_sync(1, kQThreads);
      if (tid == kIssuer2) {
        tc_fence_after();
        slot_mmas(tau, (T - 1) & 1, T - 1 - tau);
        tc_commit(&bars->m2[c & 1]);
      }
      if (tid == 0) {
        issue_dr();
        bulk_wait_group_read0();
      }
      ok = mbar_wait(&bars->m2[c & 1], (c >> 1) & 1, wait_ns, abort);
      if (!named_bar_and(1, kQThreads, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      flush_dr(tau);
      tc_fence_before();
    }

    if (ok) {
      // dq = d(q+u) + d(q+v) for this row's 32 head dims; the tile's column
      // sums of both go to the bias partials through shared memory
      // (XOR-staggered columns).
      named_bar_sync(1, kQThreads);  // the slot buffers are free for the column sums
      if (tid == 0) issue_dr();
      uint32_t u[32], v[32];
      const uint32_t lb = tmem + (static_cast<uint32_t>(quad * 32) << 16);
      tmem_ld32(lb + kColA + 32 * half, u);
      tmem_ld32(lb + kColB + 32 * half, v);
      tmem_wait_ld(u);
      tmem_wait_ld(v);
      if (i < p.W) {
        float4* dst = reinterpret_cast<float4*>(p.dq + ((static_cast<long long>(w.b) * p.W + i) * p.H + w.h) * D +
                                                32 * half);
#pragma unroll
        for (int e = 0; e < 8; ++e)
          dst[e] = make_float4(__uint_as_float(u[4 * e]) + __uint_as_float(v[4 * e]),
                               __uint_as_float(u[4 * e + 1]) + __uint_as_float(v[4 * e + 1]),
                               __uint_as_float(u[4 * e + 2]) + __uint_as_float(v[4 * e + 2]),
                               __uint_as_float(u[4 * e + 3]) + __uint_as_float(v[4 * e + 3]));
      }
      // red[x][row ^ (x & 31)]: column x of the row sums (x < 64: d(q+u)).
      float* red = reinterpret_cast<float*>(sGs);
#pragma unroll
      for (int x = 0; x < 32; ++x) {
        red[(32 * half + x) * BM + (a ^ x)] = __uint_as_float(u[x]);
        red[(64 + 32 * half + x) * BM + (a ^ x)] = __uint_as_float(v[x]);
      }
      named_bar_sync(1, kQThreads);
      if (tid < 2 * D) {
        float sum = 0.f;
        for (int r = 0; r < BM; ++r) sum += red[tid * BM + (r ^ (tid & 31))];
        const int qt = w.i0 / BM;
        p.part[((static_cast<long long>(w.b) * p.nqt + qt) * p.H + w.h) * 2 * D + tid] = sum;
      }
    }
    if (!ok && tid == 0) report_timeout(abort, p.status);
    // Let this CTA's own reductions and gradient MMAs finish before the
    // memory is released.
    if (tid == 0) bulk_wait_group0();
    if (tid == kIssuer2) {
      tc_commit(&bars->fin2);
      mbar_wait_own(&bars->fin2, 0, wait_ns);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// ============================================================================
// dk / dv kernel: 8 warps as in the dq kernel, persistent.  An item is a
// block of 64 segment keys of a (batch, head) with the query tiles that see
// them; items are ordered longest first (the key block varies slowest) and
// dealt to the CTAs in a snake order.  A CTA walks one stream of query tiles
// across its items, so its barriers, TMEM and load pipeline carry from item
// to item: the next item's keys and values load as soon as the last tile's
// score MMAs have read the current ones, and its first score MMAs are
// issued behind the last tile's gradient MMAs.  (q+u), (q+v) of the next
// tile are built while the current tile's gradient MMAs run.
// ============================================================================
struct KItem {
  int b, h, jj0, qt0, nt;  // keys jj0 .. jj0+63; query tiles qt0 .. qt0+nt-1
};

__device__ __forceinline__ KItem kitem(int it, int B, int H, int nqt) {
  const int BH = B * H;
  const int bh = it % BH;
  KItem r;
  r.b = bh / H;
  r.h = bh % H;
  r.jj0 = (it / BH) * BN;
  r.qt0 = r.jj0 / BM;  // first query tile with a row i >= jj0
  r.nt = nqt - r.qt0;
  return r;
}

// Position in a CTA's tile stream: its k-th item and that item's s-th tile.
struct KPos {
  int k, s;
  bool valid;
  KItem w;
};

__global__ void __launch_bounds__(kQThreads, 1)
    bwd_dkdv_tc64_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_rw,
                         const __grid_constant__ CUtensorMap tm_do, const BwdParams p, int n_items) {
  grid_dep_wait();  // launched behind the dq kernel: the per-row Delta it writes
  grid_dep_launch_dependents();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  uint8_t* sK = smem + kKOffK;
  uint8_t* sV = smem + kKOffV;
  uint8_t* sQu = smem + kKOffQu;  // 2 buffers
  uint8_t* sQv = smem + kKOffQv;  // 2 buffers
  uint8_t* sQ = smem + kKOffQ;
  uint8_t* sDO = smem + kKOffDO;
  uint8_t* sR = smem + kKOffR;
  uint8_t* sP = smem + kKOffP;
  uint8_t* sG = smem + kKOffG;
  KBars* bars = reinterpret_cast<KBars*>(smem + kKOffBar);
  float* sBias = reinterpret_cast<float*>(smem + kKOffBias);  // [item parity][u, v][64]
  volatile int* abort = &bars->abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quad = warp & 3, half = warp >> 2;
  const int a = quad * 32 + lane;
  const uint64_t wait_ns = p.wait_ns;
  const int P = gridDim.x;

  auto pos_of = [&](int k) {  // tile 0 of the CTA's k-th item
    KPos t;
    const int it = sched_unit(k, blockIdx.x, P);
    t.k = k;
    t.s = 0;
    t.valid = it < n_items;
    if (t.valid) t.w = kitem(it, p.B, p.H, p.nqt);
    return t;
  };
  auto next_pos = [&](const KPos& t) {
    if (!t.valid) return t;
    if (t.s + 1 < t.w.nt) {
      KPos r = t;
      ++r.s;
      return r;
    }
    return pos_of(t.k + 1);
  };
  // u, v of an item's head into its bias buffer (threads 0-127)
  auto stage_bias = [&](const KPos& t) {
    if (t.valid && tid < 2 * D)
      sBias[(t.k & 1) * 2 * D + tid] = tid < D ? p.bias_u[t.w.h * D + tid] : p.bias_v[t.w.h * D + tid - D];
  };

  KPos cur = pos_of(0);
  KPos nx1 = next_pos(cur);
  KPos nx2 = next_pos(nx1);
  if (tid == 0) {
    mbar_init(&bars->kv, 1);
    mbar_init(&bars->in[0], 1);
    mbar_init(&bars->in[1], 1);
    mbar_init(&bars->m1, 1);
    mbar_init(&bars->m2, 1);
    mbar_init(&bars->fin, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  stage_bias(cur);
  if (nx1.valid && nx1.k != cur.k) stage_bias(nx1);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  uint32_t n_ld[2] = {0, 0};  // tile loads issued per stage (thread 0)
  uint32_t n_kv = 0;          // key/value loads issued (thread 0)
  auto issue_tile_loads = [&](const KPos& t, int st) {
    const int i0 = (t.w.qt0 + t.s) * BM;
    mbar_arrive_expect_tx(&bars->in[st], 2 * kTile + kWinTile);
    tma_load_4d(sQ + st * kTile, &tm_q, &bars->in[st], 0, t.w.h, i0, t.w.b);
    tma_load_4d(sDO + st * kTile, &tm_do, &bars->in[st], 0, t.w.h, i0, t.w.b);
    tma_load_3d(sR + st * kWinTile, &tm_rw, &bars->in[st], 0, t.w.h, i0 - t.w.jj0 - BN);
    ++n_ld[st];
  };
  auto issue_kv_loads = [&](const KItem& w) {
    mbar_arrive_expect_tx(&bars->kv, 2 * kKTile);
    tma_load_4d(sK, &tm_k, &bars->kv, 0, w.h, p.M + w.jj0, w.b);
    tma_load_4d(sV, &tm_v, &bars->kv, 0, w.h, p.M + w.jj0, w.b);
    ++n_kv;
  };
  if (tid == 0 && cur.valid) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_rw);
    tma_prefetch_desc(&tm_do);
    issue_kv_loads(cur.w);
    issue_tile_loads(cur, 0);
    if (nx1.valid) issue_tile_loads(nx1, 1);
  }

  constexpr uint32_t id64 = idesc_bf16(128, 64, false, false);
  constexpr uint32_t id192 = idesc_bf16(128, 192, false, false);
  constexpr uint32_t idT = idesc_bf16(64, 64, true, true);
  const uint64_t dK = sdesc_sw128(smem_u32(sK), 16, 1024);
  const uint64_t dV = sdesc_sw128(smem_u32(sV), 16, 1024);
  const uint64_t dPT = sdesc_sw128(smem_u32(sP), 8192, 1024);
  const uint64_t dGT = sdesc_sw128(smem_u32(sG), 8192, 1024);

  // Thread 0: the score MMAs of stream tile g at t (its (q+u), (q+v) in
  // buffer g & 1); an item's first tile waits for the item's keys and values.
  auto score_mmas = [&](const KPos& t, int g) -> bool {
    const int st = g & 1;
    if (t.s == 0 && !mbar_wait(&bars->kv, t.k & 1, wait_ns, abort)) return false;
    tc_fence_after();
    const uint64_t dQu = sdesc_sw128(smem_u32(sQu + st * kTile), 16, 1024);
    const uint64_t dQv = sdesc_sw128(smem_u32(sQv + st * kTile), 16, 1024);
    const uint64_t dDO = sdesc_sw128(smem_u32(sDO + st * kTile), 16, 1024);
    const uint64_t dR = sdesc_sw128(smem_u32(sR + st * kWinTile), 16, 1024);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) mma_ss(tmem + kColS, dQu + 2 * kk, dK + 2 * kk, id64, kk > 0);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) mma_ss(tmem + kColDP, dDO + 2 * kk, dV + 2 * kk, id64, kk > 0);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) mma_ss(tmem + kColWin, dQv + 2 * kk, dR + 2 * kk, id192, kk > 0);
    tc_commit(&bars->m1);
    return true;
  };
  // Everyone: this warp's half of (q+u), (q+v) of stream tile g at t, from its raw q.
  auto build = [&](const KPos& t, int g) -> bool {
    const int st = g & 1;
    if (!mbar_wait(&bars->in[st], (g >> 1) & 1, wait_ns, abort)) return false;
    const float* bu = sBias + (t.k & 1) * 2 * D;
    build_qu_qv_half(sQ + st * kTile, sQu + st * kTile, sQv + st * kTile, a, half, bu, bu + D);
    return true;
  };
  // lse (log2 domain) and Delta of this thread's row in tile t; rows past W
  // get lse = +inf, so every p is 0.  Loaded one tile ahead.
  auto row_consts = [&](const KPos& t, float& l2, float& dl) {
    l2 = INFINITY;
    dl = 0.f;
    if (!t.valid) return;
    const int i = (t.w.qt0 + t.s) * BM + a;
    if (i < p.W) {
      const long long row_id = (static_cast<long long>(t.w.b) * p.H + t.w.h) * p.W + i;
      l2 = p.lse[row_id] * kLog2e;
      dl = p.delta[row_id];
    }
  };

  bool ok = true;
  if (cur.valid) {
    ok = build(cur, 0);
    if (!ok) report_timeout(abort, p.status);
  }
  fence_proxy_async_smem();
  ok = __syncthreads_and(ok) != 0;
  if (tid == 0 && ok && cur.valid && !score_mmas(cur, 0)) report_timeout(abort, p.status);

  float lse_next, delta_next;
  row_consts(cur, lse_next, delta_next);
  for (int g = 0; cur.valid && ok; ++g) {
    const int st = g & 1;
    const KItem& w = cur.w;
    const int i = (w.qt0 + cur.s) * BM + a;
    const float lse2 = lse_next, delta = delta_next;
    row_consts(nx1, lse_next, delta_next);
    const bool last = cur.s + 1 == w.nt;  // the item's last tile
    // (1) everyone: p and g of the tile's rows against the key block; then
    // the next tile's (q+u), (q+v).  The tile's score MMAs are done, so on
    // the item's last tile thread 0 loads the next item's keys and values.
    ok = mbar_wait(&bars->m1, g & 1, wait_ns, abort);
    if (!__syncthreads_and(ok)) {
      ok = false;
      break;
    }
    tc_fence_after();
    if (tid == 0 && last && nx1.valid) issue_kv_loads(nx1.w);
    {
      float gr[32], pr[32];
      // key jj0 + c is visible to row i iff jj0 + c <= i and it exists
      const int lim = min(i - w.jj0, p.W - 1 - w.jj0);
      step_grads_half(tmem, kColS, kColDP, kColWin, quad, half, lane, lse2, delta, p.scale, p.scale_log2e,
                      [&](int c) { return c <= lim; }, gr, pr);
      store_row_half(sP, a, half, pr);
      store_row_half(sG, a, half, gr);
    }
    if (nx1.valid && !build(nx1, g + 1)) ok = false;
    fence_proxy_async_smem();
    tc_fence_before();
    if (!__syncthreads_and(ok)) {
      ok = false;
      break;
    }
    // (2) thread 0: dV += P^T dout, dK += G^T (q+u)  (M = 64 keys, K = 128
    // queries); then the next tile's score MMAs.
    if (tid == 0) {
      tc_fence_after();
      const uint64_t dDOmn = sdesc_sw128(smem_u32(sDO + st * kTile), 8192, 1024);
      const uint64_t dQuMN = sdesc_sw128(smem_u32(sQu + st * kTile), 8192, 1024);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_ss(tmem + kColA, dPT + 128 * kk, dDOmn + 128 * kk, idT, cur.s > 0 || kk > 0);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_ss(tmem + kColB, dGT + 128 * kk, dQuMN + 128 * kk, idT, cur.s > 0 || kk > 0);
      tc_commit(&bars->m2);
      if (nx1.valid && !score_mmas(nx1, g + 1)) report_timeout(abort, p.status);
    }
    // (3) everyone: the tile's MMAs are done; thread 0 refills its stage
    // with tile g+2, whose item's u, v go to that item's bias buffer (read
    // by its build after the next block barrier).  After an item's last
    // tile its dV and dK go out.
    ok = mbar_wait(&bars->m2, g & 1, wait_ns, abort);
    if (!__syncthreads_and(ok)) {
      ok = false;
      break;
    }
    if (tid == 0 && nx2.valid) issue_tile_loads(nx2, st);
    if (nx2.valid && nx2.s == 0) stage_bias(nx2);
    if (last) {
      // Rows of the M = 64 results: lanes 0-15 of each quadrant, row 16 quad + lane.
      tc_fence_after();
      uint32_t vv[32], kv[32];
      const uint32_t lb = tmem + (static_cast<uint32_t>(quad * 32) << 16);
      tmem_ld32(lb + kColA + 32 * half, vv);
      tmem_ld32(lb + kColB + 32 * half, kv);
      tmem_wait_ld(vv);
      tmem_wait_ld(kv);
      const int jj = w.jj0 + 16 * quad + lane;
      if (lane < 16 && jj < p.W) {
        const long long off = ((static_cast<long long>(w.b) * p.W + jj) * p.H + w.h) * D + 32 * half;
        float4* dvp = reinterpret_cast<float4*>(p.dv + off);
        float4* dkp = reinterpret_cast<float4*>(p.dk + off);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          dvp[e] = make_float4(__uint_as_float(vv[4 * e]), __uint_as_float(vv[4 * e + 1]),
                               __uint_as_float(vv[4 * e + 2]), __uint_as_float(vv[4 * e + 3]));
          dkp[e] = make_float4(__uint_as_float(kv[4 * e]), __uint_as_float(kv[4 * e + 1]),
                               __uint_as_float(kv[4 * e + 2]), __uint_as_float(kv[4 * e + 3]));
        }
      }
      tc_fence_before();
    }
    cur = nx1;
    nx1 = nx2;
    nx2 = next_pos(nx2);
  }
  // Let this CTA's own copies and MMAs finish before the memory is released.
  if (tid == 0) {
    if (n_kv > 0) mbar_wait_own(&bars->kv, (n_kv - 1) & 1, wait_ns);
    for (int s2 = 0; s2 < 2; ++s2)
      if (n_ld[s2] > 0) mbar_wait_own(&bars->in[s2], (n_ld[s2] - 1) & 1, wait_ns);
    tc_commit(&bars->fin);
    mbar_wait_own(&bars->fin, 0, wait_ns);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

int num_sms() {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

}  // namespace

size_t relattn_bwd_tc64_scratch_bytes(int B, int W, int H) {
  const size_t nqt = (static_cast<size_t>(W) + BM - 1) / BM;
  return sizeof(float) * (static_cast<size_t>(B) * H * W + static_cast<size_t>(B) * nqt * H * 2 * D);
}

cudaError_t launch_relattn_bwd_tc64(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                    const CUtensorMap& tm_rw, const CUtensorMap& tm_do, const CUtensorMap& tm_dr,
                                    const float* bias_u,
                                    const float* bias_v, const float* lse, const void* o, const void* dout,
                                    float* dq, float* dk, float* dv, float* dr, float* du, float* dvb, int B,
                                    int W, int M, int H, int n_r, float scale, void* scratch, const WaitCtl& wc,
                                    cudaStream_t stream) {
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(bwd_dq_tc64_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kQSmem)) !=
      cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(bwd_dkdv_tc64_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kKSmem)) !=
      cudaSuccess)
    return e;
  BwdParams p;
  p.bias_u = bias_u;
  p.bias_v = bias_v;
  p.lse = lse;
  p.o = static_cast<const __nv_bfloat16*>(o);
  p.dout = static_cast<const __nv_bfloat16*>(dout);
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.dr = dr;
  p.delta = static_cast<float*>(scratch);
  p.nqt = (W + BM - 1) / BM;
  p.part = p.delta + static_cast<size_t>(B) * H * W;
  p.B = B;
  p.W = W;
  p.M = M;
  p.H = H;
  p.n_r = n_r;
  p.scale = scale;
  p.scale_log2e = scale * kLog2e;
  p.status = wc.status;
  p.wait_ns = wc.limit_ns;
  p.inject_stall = wc.inject_stall;
  if ((e = cudaMemsetAsync(dr, 0, sizeof(float) * static_cast<size_t>(n_r) * H * D, stream)) != cudaSuccess)
    return e;
  const int units = p.nqt * B * H;
  if ((e = launch_dependent(bwd_dq_tc64_kernel, dim3(units), dim3(kDqThreads), kQSmem, stream, tm_q, tm_k, tm_v,
                            tm_rw, tm_do, tm_dr, p)) != cudaSuccess)
    return e;
  const int n_items = (W + BN - 1) / BN * B * H;
  const int grid = n_items < num_sms() ? n_items : num_sms();
  if ((e = launch_dependent(bwd_dkdv_tc64_kernel, dim3(grid), dim3(kQThreads), kKSmem, stream, tm_q, tm_k, tm_v,
                            tm_rw, tm_do, p, n_items)) != cudaSuccess)
    return e;
  return launch_bwd_bias(p.part, B * p.nqt, H, D, du, dvb, stream);
}

}  // namespace txl
