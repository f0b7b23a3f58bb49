// Backward of the relative attention on the tensor cores with the pair terms
// materialised, for head dimension D = 64 or 128: bf16 q, k, v, r, o and
// dout, fp32 accumulation and gradients.
//
// The formulas and the stop-gradient are those of relattn_bwd.cu ("Transformer-
// XL, explained", method step 2 and the symbol SG(.)):
//   p_ij = exp(s_ij - lse_i),  g_ij = scale p_ij (dout_i . v_j - Delta_i)
//   dq_i = sum_j g_ij k_j + sum_j g_ij r_{M+i-j}
//   dk_j = sum_i g_ij (q_i+u),  dv_j = sum_i p_ij dout_i   (segment keys j)
//   dr_d = sum_{b,i} g_{i, M+i-d} (q_i+v),  du = sum_{b,i} sum_j g_ij k_j,
//   dbias_v = sum_{b,i} sum_j g_ij r_{M+i-j}
//
// At D = 128 the fused design of relattn_bwd_tc64.cu does not fit (the
// tiles of both score operands and the gradient accumulators exceed the
// shared and tensor memory); at D = 64 this design is the faster one.  The
// work is split in three:
//   1. bwd_pairs_kernel, one CTA per (batch, head, 128-query tile) or half of
//      one's key steps, 64-key steps: S = (q+u) K^T, dP = dout V^T and the
//      step's 64 new distances of the 192-distance window (q+v) R^T on the
//      tensor cores (K = D), then per pair p and g with the distance term
//      shifted into key order as in the forward.  It writes, in bf16,
//      G [bh][i][j] and P [bh][i][j] (key order; P only for steps with
//      segment keys), GS [bh][i][d] (the same g in distance order,
//      d = M+i-j), and (q+u), (q+v) as the MMAs saw them.
//   2. bgemm_kernel, this library's tcgen05 GEMM arranged for the products
//      (M = 128 rows of a tile, N = D, fp32 accumulators in TMEM, fp32
//      results), all four in one launch whose CTAs take tiles from a counter:
//      dq = G K + GS r per (batch, head), the two parts in two accumulators of
//      one tile, whose epilogue also writes each part's column sums over the
//      tile's rows (the bias gradients' partials); dk = G^T (q+u) and
//      dv = P^T dout over the segment keys (G and P read as MN-major A
//      operands); dr = sum_b GS^T (q+v) per head (the k loop runs over every
//      sequence's queries).
//   3. bwd_bias_kernel adds the partials in a fixed order into du, dv_bias.
// The batch runs in chunks of sequences whose scratch fits a cap (1 GiB by
// default); dr accumulates over the chunks.  Every result is deterministic.
// Every wait is bounded; a timed-out wait raises the device status word and
// the CTA unwinds.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <atomic>
#include <cstdint>
#include <algorithm>
#include <initializer_list>
#include <queue>
#include <vector>

#include "pdl.cuh"
#include "relattn_tc_common.cuh"
#include "txl_device.cuh"
#include "txl_internal.h"

namespace txl {
namespace {

constexpr int BM = 128;  // query rows per tile
constexpr int BN = 64;   // keys per step
constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------------------
// 1. Score rebuild
// ---------------------------------------------------------------------------
// Shared memory: an operand tile of head dimension D is D / 64 tiles of 64
// columns (128-byte rows, 128-byte swizzle), one after the other.  Inputs of
// a step (64 keys, 64 values, 64 new distance rows) in a ring of stages
// (three at D = 64, two at D = 128).  G and P
// of a step leave through 128 x 64 staging tiles and TMA stores, GS (the same
// g in distance order) through row-contiguous stores read from the G tile.
//
// TMEM: S and dP of a step in two buffers (columns 0-127, 128-255), and the
// 192-distance window as three of four 64-column slots (256-511).  The window
// of step t + 1 is the window of step t moved by 64 distances, so a step
// computes only its 64 new distances, into the slot the step before it no
// longer reads; the MMAs of step t + 1 then run while step t's pairs are
// computed.
constexpr int kHalfQ = BM * 128;   // 128 rows x 64 bf16: 16 KB
constexpr int kHalfK = BN * 128;   // 64 rows: 8 KB
template <int D>
struct PairCfg {
  static constexpr int NH = D / 64;                          // 64-column tiles of an operand
  static constexpr int kSOffQu = 0;
  static constexpr int kSOffQv = kSOffQu + NH * kHalfQ;
  static constexpr int kSOffDO = kSOffQv + NH * kHalfQ;
  static constexpr int kSOffIn = kSOffDO + NH * kHalfQ;     // stage s: K, V, R tiles (NH x 8 KB each)
  static constexpr int kInStage = 3 * NH * kHalfK;
  static constexpr int NS = D == 64 ? 3 : 2;                // input stages (loads run NS steps ahead)
  static constexpr int kSOffG = kSOffIn + NS * kInStage;    // G staging: 128 rows x 64 keys
  static constexpr int kSOffP = kSOffG + BM * BN * 2;       // P staging
  static constexpr int kSOffBar = kSOffP + BM * BN * 2;
  static constexpr int kSOffBias = kSOffBar + 256;          // u, then v of the head (fp32)
  static constexpr int kSSmem = kSOffBias + 2 * D * 4 + 1024;
  static_assert(D == 64 || D == 128, "head dimension");
  static_assert(kSSmem <= 232448, "shared memory budget");
};
constexpr uint32_t kColWin = 256, kSTmemCols = 512;
constexpr int kPairThreads = 256;            // warps 0-7
constexpr int kSThreads = kPairThreads + 96;  // + the load, MMA and store warps

struct ScoreParams {
  const float* bias_u;
  const float* bias_v;
  const float* lse;         // [B, H, W]
  const __nv_bfloat16* o;   // [B, W, H, D]
  const __nv_bfloat16* dout;
  __nv_bfloat16* GS;        // [B*H][W][LP], column d = distance
  __nv_bfloat16* Qu;        // [B, W, H, D]: q + u, rounded as the MMAs see it
  __nv_bfloat16* Qv;        // [B, W, H, D]: q + v
  int B, W, M, H, nqt, LP;
  float scale, scale_log2e;
  unsigned int* status;
  unsigned long long wait_ns;
  int inject_stall;  // test hook: the load thread loads nothing past the first two steps
  unsigned int* gemm_ctr;  // the products' tile counter, zeroed here for the launch that follows
  int split_qt;            // the last split_qt query tiles run as two CTAs each (halves of the key steps)
};

// CTA u's work: a (sequence, head, 128-query tile) unit, or one half of its
// key steps.  Whole units come first, longest first; then the halves of the
// units of the last split_qt query tiles (the longest), longest first.  The
// pair terms of different key steps are independent, so a unit's steps can
// run in two CTAs; each rebuilds the distance window at its first step.
__host__ __device__ __forceinline__ Unit pair_item(int u, const ScoreParams& p) {
  const int BH = p.B * p.H;
  const int n_whole = (p.nqt - p.split_qt) * BH;
  int qt, bh, part = -1;
  if (u < n_whole) {
    qt = p.nqt - p.split_qt - 1 - u / BH;
    bh = u % BH;
  } else {
    u -= n_whole;
    const int k = u / BH;  // 0 .. 2 split_qt - 1
    qt = p.nqt - 1 - (k >> 1);
    part = k & 1;
    bh = u % BH;
  }
  Unit r;
  r.b = bh / p.H;
  r.h = bh % p.H;
  r.i0 = qt * BM;
  const int n = min(p.M + r.i0 + BM - 1, p.M + p.W - 1) / BN + 1;
  r.t0 = part == 1 ? n / 2 : 0;
  r.nks = part < 0 ? n : part == 0 ? n / 2 : n - n / 2;
  return r;
}

struct SBars {
  uint64_t q, in[3], x, m1[2], done[2], sfree, fin;
  uint64_t ifree[3];  // input stage s read by the MMAs of its step (one phase per use)
  uint32_t tmem_base;
  int abort;
};

// Row a of (q+u) and (q+v) for head dims [D/2 half, D/2 half + D/2) (the
// warp half's share), from the raw q tile staged in the same layout as the
// operand tiles; also written to gqu / gqv (the share's dims of the row,
// 16-byte aligned) unless null.
template <int D>
__device__ __forceinline__ void build_half(const uint8_t* sQ, uint8_t* sQu, uint8_t* sQv, int a, int half,
                                           const float* bu, const float* bv, __nv_bfloat16* gqu,
                                           __nv_bfloat16* gqv) {
  constexpr int CH = D / 16;  // 16-byte chunks (8 dims) of the share
#pragma unroll
  for (int c = 0; c < CH; ++c) {
    const int gc = half * CH + c;  // chunk of the row: dims 8 gc .. 8 gc + 7
    const uint32_t off =
        (gc >> 3) * kHalfQ + (a >> 3) * 1024 + (a & 7) * 128 + ((((gc & 7) ^ (a & 7))) << 4);
    const uint4 raw = *reinterpret_cast<const uint4*>(sQ + off);
    const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
    const float* ub = bu + 8 * gc;
    const float* vb = bv + 8 * gc;
    uint32_t qu[4], qv[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float x0 = bf16_lo(w4[e]), x1 = bf16_hi(w4[e]);
      qu[e] = pack_bf16x2(x0 + ub[2 * e], x1 + ub[2 * e + 1]);
      qv[e] = pack_bf16x2(x0 + vb[2 * e], x1 + vb[2 * e + 1]);
    }
    const uint4 xu = make_uint4(qu[0], qu[1], qu[2], qu[3]), xv = make_uint4(qv[0], qv[1], qv[2], qv[3]);
    *reinterpret_cast<uint4*>(sQu + off) = xu;
    *reinterpret_cast<uint4*>(sQv + off) = xv;
    if (gqu != nullptr) {
      reinterpret_cast<uint4*>(gqu)[c] = xu;
      reinterpret_cast<uint4*>(gqv)[c] = xv;
    }
  }
}

// Zeros of row[lo, hi) (bf16; row 16-byte aligned).
__device__ __forceinline__ void zero_bf16(__nv_bfloat16* row, int lo, int hi) {
  int d = lo;
  for (; d < hi && (d & 7) != 0; ++d) row[d] = __float2bfloat16_rn(0.f);
  for (; d + 8 <= hi; d += 8) *reinterpret_cast<uint4*>(row + d) = make_uint4(0u, 0u, 0u, 0u);
  for (; d < hi; ++d) row[d] = __float2bfloat16_rn(0.f);
}

// 32 values of row a, keys [32 half, 32 half + 32) of a 128 x 64 tile staged
// for a 128-byte-swizzled TMA store (64 bf16 per row).
__device__ __forceinline__ void stage_row32(uint8_t* tile, int a, int half, const float (&x)[32]) {
  uint8_t* rowp = tile + (a >> 3) * 1024 + (a & 7) * 128;
#pragma unroll
  for (int c = 0; c < 4; ++c)
    *reinterpret_cast<uint4*>(rowp + (((4 * half + c) ^ (a & 7)) << 4)) =
        make_uint4(pack_bf16x2(x[8 * c], x[8 * c + 1]), pack_bf16x2(x[8 * c + 2], x[8 * c + 3]),
                   pack_bf16x2(x[8 * c + 4], x[8 * c + 5]), pack_bf16x2(x[8 * c + 6], x[8 * c + 7]));
}

__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}

// Warps 0-7 compute the pairs, two per TMEM lane quadrant (key columns 0-31
// and 32-63 of the same rows), each on its own: a step's barrier takes one
// arrival per warp.  One thread of warp 8 issues the loads (NS steps ahead),
// one of warp 9 the MMAs (one step ahead of the pairs), one of warp 10 the
// G / P stores, each waiting only on what it needs.
template <int D>
__global__ void __launch_bounds__(kSThreads, 1)
    bwd_pairs_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_r,
                     const __grid_constant__ CUtensorMap tm_do, const __grid_constant__ CUtensorMap tm_g,
                     const __grid_constant__ CUtensorMap tm_p, const ScoreParams p) {
  using C = PairCfg<D>;
  constexpr int NH = C::NH;
  grid_dep_wait();  // launched behind the previous kernel on the stream: it has completed from here on
  grid_dep_launch_dependents();  // the products' CTAs may take SMs this launch no longer needs
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  uint8_t* sQu = smem + C::kSOffQu;
  uint8_t* sQv = smem + C::kSOffQv;
  uint8_t* sDO = smem + C::kSOffDO;
  uint8_t* sIn = smem + C::kSOffIn;
  uint8_t* sG = smem + C::kSOffG;
  uint8_t* sP = smem + C::kSOffP;
  SBars* bars = reinterpret_cast<SBars*>(smem + C::kSOffBar);
  float* sBias = reinterpret_cast<float*>(smem + C::kSOffBias);
  volatile int* abort = &bars->abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quad = warp & 3, half = warp >> 2;
  const int a = quad * 32 + lane;  // this thread's row of the tile
  const uint64_t wait_ns = p.wait_ns;

  const Unit w = pair_item(blockIdx.x, p);
  const int T = w.nks;   // steps of this CTA: key steps t0 + t, t = 0 .. T-1
  const int t0 = w.t0;
  const int i = w.i0 + a;  // query row
  const int z = w.b * p.H + w.h;
  // first distance of the window of local step t: M + i0 - 64 (t0 + t) - 64
  auto wbase = [&](int t) { return p.M + w.i0 - BN * (t0 + t) - BN; };

  if (tid == 0) {
    if (blockIdx.x == 0) *p.gemm_ctr = 0u;  // read by the next launch on the stream only
    mbar_init(&bars->q, 1);
    for (int x = 0; x < C::NS; ++x) {
      mbar_init(&bars->in[x], 1);
      mbar_init(&bars->ifree[x], 1);
    }
    mbar_init(&bars->x, 1);
    mbar_init(&bars->m1[0], 1);
    mbar_init(&bars->m1[1], 1);
    mbar_init(&bars->done[0], kPairThreads / 32);  // one arrival per pair warp
    mbar_init(&bars->done[1], kPairThreads / 32);
    mbar_init(&bars->sfree, 1);
    mbar_init(&bars->fin, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&bars->tmem_base, kSTmemCols);
    tmem_relinquish();
  }
  if (tid < 2 * D) sBias[tid] = tid < D ? p.bias_u[w.h * D + tid] : p.bias_v[w.h * D + tid - D];
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  // 64 distance rows from `d0` (every 64-dim tile of them) into NH x 8 KB.
  auto load_r64 = [&](uint8_t* dst, uint64_t* bar, int d0) {
#pragma unroll
    for (int hh = 0; hh < NH; ++hh) tma_load_3d(dst + hh * kHalfK, &tm_r, bar, 64 * hh, w.h, d0);
  };
  // Inputs of local step t into stage t & 1: keys and values [64 (t0 + t),
  // + 64) and the window's new distances [wb(t), wb(t) + 64).
  constexpr int NS = C::NS;
  uint32_t n_in[3] = {0, 0, 0};  // loads issued per stage (the load thread)
  auto load_in = [&](int t) {
    const int s = t % NS;
    uint8_t* st = sIn + s * C::kInStage;
    mbar_arrive_expect_tx(&bars->in[s], C::kInStage);
#pragma unroll
    for (int hh = 0; hh < NH; ++hh) {
      tma_load_4d(st + hh * kHalfK, &tm_k, &bars->in[s], 64 * hh, w.h, BN * (t0 + t), w.b);
      tma_load_4d(st + (NH + hh) * kHalfK, &tm_v, &bars->in[s], 64 * hh, w.h, BN * (t0 + t), w.b);
    }
    load_r64(st + 2 * NH * kHalfK, &bars->in[s], wbase(t));
    if (s == 0) ++n_in[0];  // constant indices keep the counts in registers
    else if (s == 1) ++n_in[1];
    else ++n_in[2];
  };
  // one thread of each of warps 8-10: loads, MMAs, stores
  const bool loader = tid == kPairThreads, mma_thread = tid == kPairThreads + 32,
             storer = tid == kPairThreads + 64;
  if (loader) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_r);
    tma_prefetch_desc(&tm_do);
    tma_prefetch_desc(&tm_g);
    tma_prefetch_desc(&tm_p);
    // the raw q tile goes to stage 1 until (q+u), (q+v) are built
    mbar_arrive_expect_tx(&bars->q, 2 * NH * kHalfQ);
#pragma unroll
    for (int hh = 0; hh < NH; ++hh) {
      tma_load_4d(sIn + C::kInStage + hh * kHalfQ, &tm_q, &bars->q, 64 * hh, w.h, w.i0, w.b);
      tma_load_4d(sDO + hh * kHalfQ, &tm_do, &bars->q, 64 * hh, w.h, w.i0, w.b);
    }
    load_in(0);
    if (NS == 3 && T > 2 && !p.inject_stall) load_in(2);  // stage 2 is free from the start
    // the rest of step 0's window (distances wb(0) + 64 ... + 192) into the
    // staging tiles, which are free until step 0's pairs are written
    mbar_arrive_expect_tx(&bars->x, 2 * NH * kHalfK);
    load_r64(sG, &bars->x, wbase(0) + 64);
    load_r64(sP, &bars->x, wbase(0) + 128);
  }

  // Per-row constants: lse (log2 domain) and Delta = dout . o.
  float lse2 = INFINITY, delta = 0.f;  // rows past W: every p is 0
  if (tid < kPairThreads && i < p.W) {
    const long long row_id = (static_cast<long long>(w.b) * p.H + w.h) * p.W + i;
    lse2 = p.lse[row_id] * kLog2e;
    const long long off = ((static_cast<long long>(w.b) * p.W + i) * p.H + w.h) * D;
    const uint4* po = reinterpret_cast<const uint4*>(p.o + off);
    const uint4* pg = reinterpret_cast<const uint4*>(p.dout + off);
    float s0 = 0.f, s1 = 0.f;
#pragma unroll 4
    for (int c = 0; c < D / 8; ++c) {
      const uint4 x = __ldg(po + c), y = __ldg(pg + c);
      const uint32_t xw[4] = {x.x, x.y, x.z, x.w}, yw[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        s0 = fmaf(bf16_lo(xw[e]), bf16_lo(yw[e]), s0);
        s1 = fmaf(bf16_hi(xw[e]), bf16_hi(yw[e]), s1);
      }
    }
    delta = s0 + s1;
  }
  bool ok = true;
  if (tid < kPairThreads) {
    // (q+u) and (q+v) from the raw q tile; rows past W are not written out
    ok = mbar_wait(&bars->q, 0, wait_ns, abort);
    if (ok) {
      __nv_bfloat16 *gqu = nullptr, *gqv = nullptr;
      if (i < p.W && t0 == 0) {  // one CTA of a split unit writes them
        const size_t off = ((static_cast<size_t>(w.b) * p.W + i) * p.H + w.h) * D + (D / 2) * half;
        gqu = p.Qu + off;
        gqv = p.Qv + off;
      }
      build_half<D>(sIn + C::kInStage, sQu, sQv, a, half, sBias, sBias + D, gqu, gqv);
    } else {
      report_timeout(abort, p.status);
    }
    fence_proxy_async_smem();
  }
  ok = __syncthreads_and(ok) != 0;

  constexpr uint32_t id64 = idesc_bf16(128, 64, false, false);
  const uint64_t dQu = sdesc_sw128(smem_u32(sQu), 16, 1024);
  const uint64_t dQv = sdesc_sw128(smem_u32(sQv), 16, 1024);
  const uint64_t dDO = sdesc_sw128(smem_u32(sDO), 16, 1024);
  // TMEM column of window position `pos` (a multiple of 32) at step t
  auto win_col = [&](int pos, int t) -> uint32_t {
    return kColWin + 64 * (((pos >> 6) - t) & 3) + (pos & 63);
  };
  // (q+v) against a 64-row distance tile, into the window slot of block k at step t
  auto win_mma = [&](const uint8_t* rtile, int k, int t) {
    const uint64_t dR = sdesc_sw128(smem_u32(rtile), 16, 1024);
    const uint32_t col = win_col(64 * k, t);
#pragma unroll
    for (int kk = 0; kk < 4 * NH; ++kk) {
      const uint64_t off = (kk >> 2) * (kHalfQ >> 4) + (kk & 3) * 2;
      mma_ss(tmem + col, dQv + off, dR + (kk >> 2) * (kHalfK >> 4) + (kk & 3) * 2, id64, kk > 0);
    }
  };
  // Thread 0: the MMAs of step t (K = D as D / 64 tiles of 64 columns of
  // every operand): S and dP into buffer t & 1, the window's new distances.
  auto score_mmas = [&](int t) -> bool {
    const int s = t & 1;       // S / dP buffer
    const int si = t % NS;     // input stage
    if (!mbar_wait(&bars->in[si], (t / NS) & 1, wait_ns, abort)) return false;
    if (t == 0 && !mbar_wait(&bars->x, 0, wait_ns, abort)) return false;
    tc_fence_after();
    const uint8_t* st = sIn + si * C::kInStage;
    const uint64_t dK = sdesc_sw128(smem_u32(st), 16, 1024);
    const uint64_t dV = sdesc_sw128(smem_u32(st + NH * kHalfK), 16, 1024);
    const uint32_t colS = 128 * s, colDP = 128 * s + 64;
#pragma unroll
    for (int kk = 0; kk < 4 * NH; ++kk) {
      const uint64_t qa = (kk >> 2) * (kHalfQ >> 4) + (kk & 3) * 2;
      const uint64_t ka = (kk >> 2) * (kHalfK >> 4) + (kk & 3) * 2;
      mma_ss(tmem + colS, dQu + qa, dK + ka, id64, kk > 0);
      mma_ss(tmem + colDP, dDO + qa, dV + ka, id64, kk > 0);
    }
    win_mma(st + 2 * NH * kHalfK, 0, t);
    if (t == 0) {
      win_mma(sG, 1, 0);
      win_mma(sP, 2, 0);
    }
    tc_commit(&bars->m1[s]);
    tc_commit(&bars->ifree[si]);
    return true;
  };

  // Barrier phases cannot be skipped: the MMAs of step t + 2 wait for the
  // pairs of step t (done), the pairs of step t + 1 for the staging of step t
  // (sfree), the loads of step t + NS for the MMAs of step t (ifree), and
  // each of those is what lets the next phase of the same barrier happen.
  if (loader) {
    // ============================ loads ===================================
    if (ok && T > 1) load_in(1);  // the raw q has been read: stage 1 is free
    for (int t = 0; t + NS < T && ok && !p.inject_stall; ++t) {
      // step t's MMAs have read stage t % NS: refill it for step t + NS
      // (the next phase of ifree[t % NS] needs that load, so none is skipped)
      if (!(ok = mbar_wait(&bars->ifree[t % NS], (t / NS) & 1, wait_ns, abort))) break;
      load_in(t + NS);
    }
    if (!ok) report_timeout(abort, p.status);
    // Let this CTA's own copies finish before the memory is released.
#pragma unroll
    for (int x = 0; x < NS; ++x)
      if (n_in[x] > 0) mbar_wait_own(&bars->in[x], (n_in[x] - 1) & 1, wait_ns);
    mbar_wait_own(&bars->x, 0, wait_ns);
    mbar_wait_own(&bars->q, 0, wait_ns);
  } else if (mma_thread) {
    // ============================ MMAs ====================================
    if (ok) ok = score_mmas(0) && (T < 2 || score_mmas(1));
    for (int t = 0; t + 2 < T && ok; ++t) {
      // step t's pairs have read its S / dP buffer and its oldest window slot
      if (!(ok = mbar_wait(&bars->done[t & 1], (t >> 1) & 1, wait_ns, abort))) break;
      tc_fence_after();
      ok = score_mmas(t + 2);
    }
    if (!ok) report_timeout(abort, p.status);
    tc_commit(&bars->fin);
    mbar_wait_own(&bars->fin, 0, wait_ns);
  } else if (storer) {
    // ============================ G / P stores ============================
    for (int t = 0; t < T && ok; ++t) {
      if (!(ok = mbar_wait(&bars->done[t & 1], (t >> 1) & 1, wait_ns, abort))) break;
      tma_store_3d(&tm_g, sG, BN * (t0 + t), w.i0, z);
      // P is read by the dv product only, over the segment's keys (>= M)
      if (BN * (t0 + t) + BN > p.M) tma_store_3d(&tm_p, sP, BN * (t0 + t), w.i0, z);
      bulk_commit_group();
      bulk_wait_group_read0();
      mbar_arrive(&bars->sfree);
    }
    if (!ok) report_timeout(abort, p.status);
    bulk_wait_group0();
  } else if (tid < kPairThreads) {
    // ============================ pairs ===================================
    const size_t row = (static_cast<size_t>(z) * p.W + i) * p.LP;
    if (i < p.W && t0 == 0) {
      // GS past the row's last distance M + i: the products read up to 191
      // columns beyond it (a 128-row tile plus a 64-deep k block), which must
      // hold zeros.  Key order needs none: every step writes all 64 columns.
      const int L = p.M + p.W, lo = p.M + i + 1, hi = min(L, lo + 191), mid = min(hi, lo + 96);
      zero_bf16(p.GS + row, half ? mid : lo, half ? hi : mid);
    }
    const int i_warp = w.i0 + quad * 32;  // first query row of this warp
    for (int t = 0; t < T && ok; ++t) {
      const int s = t & 1;
      if (!warp_wait(&bars->m1[s], (t >> 1) & 1, wait_ns, abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float g[32], pr[32];
      const int lim = p.M + i - BN * (t0 + t);  // key column c of the step visible iff c <= lim
      const int w0 = 32 * quad + (half ? 0 : 32);
      const uint32_t cw0 = win_col(w0, t), cw1 = win_col(w0 + 32, t);
      if (__all_sync(0xffffffffu, lim >= 32 * half + 31)) {  // no masked column in the warp's 32
        step_grads_half_at(tmem, 128 * s, 128 * s + 64, cw0, cw1, quad, half, lane, lse2, delta, p.scale,
                           p.scale_log2e, [](int) { return true; }, g, pr);
      } else {
        step_grads_half_at(tmem, 128 * s, 128 * s + 64, cw0, cw1, quad, half, lane, lse2, delta, p.scale,
                           p.scale_log2e, [&](int c) { return c <= lim; }, g, pr);
      }
      // step t-1's G and P stores have read the staging tiles
      if (t > 0 && !mbar_wait(&bars->sfree, (t - 1) & 1, wait_ns, abort)) report_timeout(abort, p.status);
      stage_row32(sG, a, half, g);
      if (BN * (t0 + t) + BN > p.M) stage_row32(sP, a, half, pr);  // a step of memory keys only: no P
      __syncwarp();
      // this warp has read step t's TMEM columns and staged its pairs; the
      // warps do not wait for one another.  The GS pass below reads only the
      // rows this warp staged, so the MMAs of step t + 2 and the stores of the
      // staging tiles need not wait for it (the next staging does, in order).
      fence_proxy_async_smem();  // the G and P staging is read by the TMA stores next
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->done[s]);
      // GS: row r of the warp holds distances D0_r - 31 ... D0_r, with
      // D0_r = M + i_warp + r - 64 (t0 + t) - 32 half, i.e. keys 32 half + 31 ... 32 half
      // of the staged G row; one row per pass, a distance per lane (64
      // contiguous bytes per store instruction).
      {
        const int d_lane = p.M + i_warp - BN * (t0 + t) - 32 * half - 31 + lane;
        const int key = 32 * half + 31 - lane;  // staged column this lane reads
        const int chunk = key >> 3;
        // rows [r_lo, r_hi) of the warp exist and have d >= 0 for this lane
        const int r_lo = max(0, -d_lane), r_hi = min(32, p.W - i_warp);
        uint16_t* gs = reinterpret_cast<uint16_t*>(p.GS) + (static_cast<size_t>(z) * p.W + i_warp) * p.LP + d_lane;
        const uint8_t* src = sG + quad * 32 * 128 + (key & 7) * 2;
        // the lane's column in each swizzle phase k = row & 7
        uint32_t col[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) col[k] = static_cast<uint32_t>((chunk ^ k) << 4);
        uint16_t val[32];
#pragma unroll
        for (int r = 0; r < 32; ++r)
          val[r] = *reinterpret_cast<const uint16_t*>(src + (r >> 3) * 1024 + (r & 7) * 128 + col[r & 7]);
#pragma unroll
        for (int r = 0; r < 32; ++r)
          if (r >= r_lo && r < r_hi) gs[static_cast<size_t>(r) * (p.LP + 1)] = val[r];
      }
    }
    if (!ok && lane == 0) report_timeout(abort, p.status);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kSTmemCols);
  }
}

// ---------------------------------------------------------------------------
// 2. The gradient products
// ---------------------------------------------------------------------------
// One persistent launch runs all four products, one CTA per SM, 192 threads:
// warp 0 loads (TMA), warp 1 issues the MMAs (M = 128, N = D, K = 16, into
// one of two TMEM accumulator slots), warps 2-5 move the fp32 accumulator
// rows to global memory.  A stage holds 64 k of A (a 128 x 64 K-major tile,
// or two 64 k x 64 row MN-major tiles) and of B (D / 64 tiles of 64 k x 64
// columns, N-major).
//
// The tiles of the four products differ in length by up to 48 times (a DR
// tile streams every sequence's queries, a DK tile near the end of the
// segment two k blocks), and the products do not depend on one another, so
// the CTAs take tiles from a device counter, longest kinds first: a CTA that
// finishes early takes the next tile, and the launch ends within about one
// short tile of the average load.  Which CTA runs a tile does not change its
// arithmetic: every output element is written by exactly one tile.
enum BMode { kModeDQ = 0, kModeDK = 1, kModeDV = 2, kModeDR = 3 };
constexpr int kGATile = 128 * 128;  // 16 KB
constexpr int kGBBlock = 64 * 128;  // 8 KB
constexpr int kGTq = 8;  // slots of the tile-index queue from the loader to the MMA and epilogue warps
constexpr int kGThreads = 192;
template <int D>
struct GemmCfg {
  static constexpr int NH = D / 64;
  static constexpr int kGStage = kGATile + NH * kGBBlock;
  static constexpr int kGStages = D == 128 ? 6 : 8;  // at most kGMaxStages
  static constexpr int kGOffEpi = kGStages * kGStage;          // DQ: 4 epilogue warps x 32 x 32 fp32 (column sums)
  static constexpr int kGOffRed = kGOffEpi + 4 * 32 * 32 * 4;  // DQ: [4 warps][2 parts][128] warp sums
  static constexpr int kGOffBar = kGOffRed + 4 * 2 * 128 * 4;
  static constexpr int kGSmem = kGOffBar + 512 + 1024;
  static_assert(kGSmem <= 232448, "shared memory budget");
  // TMEM: two accumulator slots of 2 D columns; a DQ tile fills its slot
  // with both of its parts (key, distance), the other products use the
  // first D.
  static constexpr uint32_t kGAccCols = 2 * D;
  static constexpr uint32_t kGTmemCols = 2 * kGAccCols;
};

struct GemmArgs {
  int B, W, M, H, L;
  int BH, nmt, nmtL, nkbW;  // row blocks of 128 queries, of 128 distances; 64-deep blocks of the W queries
  int nDR, nDQ;             // tiles of the DR and DQ kinds; DK and DV follow, interleaved
  int ks, nmtK;             // DK, DV: tiles start at key column M - ks (ks = M % 8), nmtK row blocks
  int LP;                   // row length of G and P
  const __nv_bfloat16* G;   // DK, DV epilogue: G, P [B*H][W][LP], q+u and dout [B, W, H, D]
  const __nv_bfloat16* P;
  const __nv_bfloat16* qu;
  const __nv_bfloat16* dout;
  int total;                // all tiles
  float* dq;
  float* dk;
  float* dv;
  float* dr;
  float* part;     // per (sequence, row block) column sums of both dq parts, [B*nmt][H][2][D]
  int accumulate;  // add to dr (a later chunk of sequences) instead of storing
  unsigned int* ctr;  // tile counter: zero when the launch starts
  unsigned int* status;
  unsigned long long wait_ns;
};

struct GTile {
  int mode, z, m0, kb0, nkb;
  int nkb_c;  // DQ: k blocks of the key part (the distance part follows, as many)
};

// Tile u of the launch, in the order the counter hands them out: DR tiles
// (rows = distances d of a head, k = (sequence, query) pairs with i >= d - M,
// where GS is not zero), then DQ tiles (rows = queries of a sequence and head;
// k runs over the keys [0, M + m0 + 128) with A = G, B = k into the slot's
// first accumulator, then over the same distances with A = GS, B = r into its
// second; G and GS are zero past each row's last visible key), then DK and DV
// tiles in turn (rows = segment keys m; k = queries i from m0 on, since key
// M + m is visible to queries i >= m only).  A DK or DV tile reads G or P from
// key column M + m0, which a tensor copy needs on a 16-byte boundary, so the
// tiles start at m0 = 128 n - ks (M + m0 a multiple of 8; rows m < 0, memory
// keys, are not written), and the k loop starts at query 128 n: the query
// tile before it has G and P only up to its own last key step.  The pairs it
// leaves out, queries i in [m, 128 n) of the tile's first ks keys, are added
// by the epilogue.  Each kind runs longest first.
__host__ __device__ __forceinline__ GTile gtile(const GemmArgs& p, int u) {
  GTile r;
  r.nkb_c = 0;
  if (u < p.nDR) {
    r.mode = kModeDR;
    r.m0 = (u / p.H) * 128;
    r.z = u % p.H;
    r.kb0 = max(0, r.m0 - p.M) / 64;
    r.nkb = p.B * (p.nkbW - r.kb0);
    return r;
  }
  u -= p.nDR;
  if (u < p.nDQ) {
    r.mode = kModeDQ;
    r.m0 = (p.nmt - 1 - u / p.BH) * 128;
    r.z = u % p.BH;
    r.kb0 = 0;
    r.nkb_c = (min(p.L, p.M + r.m0 + 128) + 63) / 64;
    r.nkb = 2 * r.nkb_c;
    return r;
  }
  u -= p.nDQ;
  r.mode = (u & 1) ? kModeDV : kModeDK;
  u >>= 1;
  r.m0 = (u / p.BH) * 128 - p.ks;
  r.z = u % p.BH;
  r.kb0 = 2 * (u / p.BH);
  r.nkb = p.nkbW - r.kb0;
  return r;
}

// The products' tile counts for nb sequences (the fields gtile reads, and
// the total); false if the count overflows an int.
bool product_geometry(GemmArgs& g, int nb, int W, int M, int H) {
  g.B = nb;
  g.W = W;
  g.M = M;
  g.H = H;
  g.L = M + W;
  g.BH = nb * H;
  g.nmt = (W + 127) / 128;
  g.nmtL = (g.L + 127) / 128;
  g.nkbW = (W + 63) / 64;
  g.nDR = H * g.nmtL;
  g.nDQ = g.BH * g.nmt;
  g.ks = M % 8;
  g.nmtK = (W + g.ks + 127) / 128;
  const long long total = static_cast<long long>(g.nDR) + g.nDQ + 2LL * g.BH * g.nmtK;
  g.total = static_cast<int>(total);
  return total <= 0x7FFFFFFFLL;
}

constexpr int kGMaxStages = 8;
struct GBars {
  uint64_t full[kGMaxStages], empty[kGMaxStages];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t tq_full[kGTq], tq_empty[kGTq];
  uint64_t done;
  uint32_t tmem_base;
  int abort;
  int tq[kGTq];
};
static_assert(sizeof(GBars) <= 512, "barrier block");

// Tensor maps (all bf16, 128-byte swizzle, zero fill):
//   a_g, a_gs: G and GS {L, W, B*H} box {64, 128, 1} (DQ, K-major);
//   b_k: k {D, H, L, B} box {64, 1, 64, 1}; b_r: r {D, H, n_r} box {64, 1, 64};
//   m_g, m_p, m_gs: G, P, GS box {64, 64, 1} (DK, DV, DR: MN-major A);
//   b_qu, b_do, b_qv: q+u, dout, q+v {D, H, W, B} box {64, 1, 64, 1}.
struct GMaps {
  CUtensorMap a_g, a_gs, b_k, b_r, m_g, m_p, m_gs, b_qu, b_do, b_qv;
};

// Queue slot n % kGTq of the tile-index queue: the loader writes tile indices
// in the order it takes them; the MMA thread and each epilogue warp read
// every one, the last (>= total) telling them to stop.
__device__ __forceinline__ int tq_read(GBars* bars, uint32_t n) { return *reinterpret_cast<volatile int*>(&bars->tq[n % kGTq]); }

template <int D>
__global__ void __launch_bounds__(kGThreads, 1)
    bgemm_kernel(const __grid_constant__ GMaps maps, const GemmArgs p) {
  using GC = GemmCfg<D>;
  constexpr int NH = GC::NH;
  constexpr int kGStage = GC::kGStage, kGOffEpi = GC::kGOffEpi, kGOffRed = GC::kGOffRed;
  constexpr uint32_t kGAccCols = GC::kGAccCols, kGTmemCols = GC::kGTmemCols;
  grid_dep_wait();  // launched behind the pair kernel: its pair terms and the zeroed counter
  grid_dep_launch_dependents();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  GBars* bars = reinterpret_cast<GBars*>(smem + GC::kGOffBar);
  volatile int* abort = &bars->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int S = GC::kGStages;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&bars->acc_full[a], 1);
      mbar_init(&bars->acc_empty[a], 4);
    }
    for (int q = 0; q < kGTq; ++q) {
      mbar_init(&bars->tq_full[q], 1);
      mbar_init(&bars->tq_empty[q], 5);  // the MMA thread and the four epilogue warps
    }
    mbar_init(&bars->done, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, kGTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const uint64_t wait_ns = p.wait_ns;

  if (warp == 0) {
    // ============================ TMA producer ============================
    if (lane == 0) {
      tma_prefetch_desc(&maps.a_g);
      tma_prefetch_desc(&maps.a_gs);
      tma_prefetch_desc(&maps.m_gs);
      tma_prefetch_desc(&maps.b_qv);
      uint32_t it = 0, n = 0;
      bool ok = true;
      unsigned int next = atomicAdd(p.ctr, 1u);
      while (ok) {
        const int u = static_cast<int>(min(next, static_cast<unsigned int>(p.total)));
        // hand the tile index on; the slot is free once its last reader is done
        if (!(ok = mbar_wait(&bars->tq_empty[n % kGTq], ((n / kGTq) & 1) ^ 1, wait_ns, abort))) break;
        bars->tq[n % kGTq] = u;
        mbar_arrive(&bars->tq_full[n % kGTq]);
        ++n;
        if (u >= p.total) break;
        next = atomicAdd(p.ctr, 1u);  // the tile after this one, fetched while this one loads
        const GTile g = gtile(p, u);
        const int b = g.mode == kModeDR ? 0 : g.z / p.H, h = g.mode == kModeDR ? g.z : g.z % p.H;
        const int nq = p.nkbW - g.kb0;  // DR: k blocks per sequence
        const CUtensorMap* ma = g.mode == kModeDK ? &maps.m_g : g.mode == kModeDV ? &maps.m_p : &maps.m_gs;
        const CUtensorMap* mb = g.mode == kModeDK ? &maps.b_qu : g.mode == kModeDV ? &maps.b_do : &maps.b_qv;
        for (int kk = 0; kk < g.nkb; ++kk, ++it) {
          const int s = static_cast<int>(it % S);
          if (!(ok = mbar_wait(&bars->empty[s], ((it / S) & 1) ^ 1, wait_ns, abort))) break;
          uint8_t* st = smem + s * kGStage;
          uint8_t* sb = st + kGATile;
          uint64_t* bar = &bars->full[s];
          mbar_arrive_expect_tx(bar, kGStage);
          if (g.mode == kModeDQ) {
            const bool dist = kk >= g.nkb_c;  // the distance part
            const int k0 = 64 * (dist ? kk - g.nkb_c : kk);
            if (!dist) {
              tma_load_3d(st, &maps.a_g, bar, k0, g.m0, g.z);
#pragma unroll
              for (int j = 0; j < NH; ++j) tma_load_4d(sb + j * kGBBlock, &maps.b_k, bar, 64 * j, h, k0, b);
            } else {
              tma_load_3d(st, &maps.a_gs, bar, k0, g.m0, g.z);
#pragma unroll
              for (int j = 0; j < NH; ++j) tma_load_3d(sb + j * kGBBlock, &maps.b_r, bar, 64 * j, h, k0);
            }
          } else {
            int bb = b, k0 = 64 * (g.kb0 + kk), x0 = g.m0, zz = g.z;
            if (g.mode == kModeDR) {
              bb = kk / nq;
              k0 = 64 * (g.kb0 + kk % nq);
              zz = bb * p.H + h;
            } else {
              x0 = p.M + g.m0;  // key columns of G and P
            }
            tma_load_3d(st, ma, bar, x0, k0, zz);
            tma_load_3d(st + kGATile / 2, ma, bar, x0 + 64, k0, zz);
#pragma unroll
            for (int j = 0; j < NH; ++j) tma_load_4d(sb + j * kGBBlock, mb, bar, 64 * j, h, k0, bb);
          }
        }
      }
      if (!ok) report_timeout(abort, p.status);
      for (int s = 0; s < S && static_cast<uint32_t>(s) < it; ++s) {
        const uint32_t last = s + ((it - 1 - s) / S) * S;
        mbar_wait_own(&bars->full[s], (last / S) & 1, wait_ns);
      }
    }
  } else if (warp == 1) {
    // ============================ MMA issuer ==============================
    if (lane == 0) {
      // A K-major for DQ (rows = queries, k = keys or distances), MN-major for
      // the others (A is G, P or GS read transposed)
      constexpr uint32_t idesc_k = idesc_bf16(128, D, false, true);
      constexpr uint32_t idesc_mn = idesc_bf16(128, D, true, true);
      const uint32_t base = smem_u32(smem);
      uint32_t it = 0, tl = 0;
      bool ok = true;
      for (uint32_t n = 0; ok; ++n, ++tl) {
        if (!(ok = mbar_wait(&bars->tq_full[n % kGTq], (n / kGTq) & 1, wait_ns, abort))) break;
        const int u = tq_read(bars, n);
        mbar_arrive(&bars->tq_empty[n % kGTq]);
        if (u >= p.total) break;
        const GTile g = gtile(p, u);
        const bool amn = g.mode != kModeDQ;
        const uint32_t acc = tl & 1;
        if (tl >= 2 && !(ok = mbar_wait(&bars->acc_empty[acc], ((tl >> 1) - 1) & 1, wait_ns, abort))) break;
        tc_fence_after();
        const uint32_t d0 = tmem + acc * kGAccCols;
        for (int kk = 0; kk < g.nkb; ++kk, ++it) {
          const int s = static_cast<int>(it % S);
          if (!(ok = mbar_wait(&bars->full[s], (it / S) & 1, wait_ns, abort))) break;
          tc_fence_after();
          const uint32_t st = base + s * kGStage;
          // K-major A: 8-row groups 1024 bytes apart, 32 bytes per 16 k.
          // MN-major A and B: 64-wide blocks 8 KB apart, 8-k-row groups 1024
          // bytes apart, 16 k rows = 2 KB.
          const uint64_t da = amn ? sdesc_sw128(st, kGATile / 2, 1024) : sdesc_sw128(st, 16, 1024);
          const uint64_t db = sdesc_sw128(st + kGATile, kGBBlock, 1024);
          // DQ: the key part into the slot's first D columns, the distance
          // part into the next D
          const bool second = g.mode == kModeDQ && kk >= g.nkb_c;
          const uint32_t d = d0 + (second ? D : 0);
          const int kl = second ? kk - g.nkb_c : kk;  // k block within the part
          const uint32_t idesc = amn ? idesc_mn : idesc_k;
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_ss(d, da + (amn ? k * 128 : k * 2), db + k * 128, idesc, (kl > 0 || k > 0) ? 1u : 0u);
          tc_commit(&bars->empty[s]);
        }
        if (!ok) break;
        tc_commit(&bars->acc_full[acc]);
      }
      if (!ok) report_timeout(abort, p.status);
      tc_commit(&bars->done);
      mbar_wait_own(&bars->done, 0, wait_ns);
    }
  } else {
    // ============================ epilogue ===============================
    // The four epilogue warps take every wait together (named barrier 2 over
    // their 128 threads returns the AND of the four outcomes), so they leave
    // the loop together and the DQ tiles' barriers always see all four.
    const int quad = warp & 3;
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    bool ok = true;
    for (uint32_t n = 0, tl = 0;; ++n, ++tl) {
      ok = named_bar_and(2, 128, warp_wait(&bars->tq_full[n % kGTq], (n / kGTq) & 1, wait_ns, abort));
      if (!ok) break;
      const int u = tq_read(bars, n);
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->tq_empty[n % kGTq]);
      if (u >= p.total) break;
      const GTile g = gtile(p, u);
      const uint32_t acc = tl & 1;
      const uint32_t acc_col = tmem + lane_base + acc * kGAccCols;
      const int row = g.m0 + 32 * quad + lane;
      ok = named_bar_and(2, 128, warp_wait(&bars->acc_full[acc], (tl >> 1) & 1, wait_ns, abort));
      if (!ok) break;
      tc_fence_after();
      if (g.mode == kModeDQ) {
        // dq = key part + distance part; the column sums of each part over
        // the tile's rows (this warp's 32 through its staging tile, then the
        // four warps in order) go to the bias partials.
        float* swp = reinterpret_cast<float*>(smem + kGOffEpi) + quad * 32 * 32;
        float* wred = reinterpret_cast<float*>(smem + kGOffRed);
        const int b = g.z / p.H, h = g.z % p.H;
        float* dst = row < p.W ? p.dq + ((static_cast<size_t>(b) * p.W + row) * p.H + h) * D : nullptr;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t vc[32], vd[32];
          tmem_ld32(acc_col + 32 * c, vc);
          tmem_ld32(acc_col + D + 32 * c, vd);
          tmem_wait_ld(vc);
          tmem_wait_ld(vd);
          if (c == D / 32 - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->acc_empty[acc]);
          }
          if (dst != nullptr) {
            float4* o4 = reinterpret_cast<float4*>(dst + 32 * c);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              o4[j] = make_float4(__uint_as_float(vc[4 * j]) + __uint_as_float(vd[4 * j]),
                                  __uint_as_float(vc[4 * j + 1]) + __uint_as_float(vd[4 * j + 1]),
                                  __uint_as_float(vc[4 * j + 2]) + __uint_as_float(vd[4 * j + 2]),
                                  __uint_as_float(vc[4 * j + 3]) + __uint_as_float(vd[4 * j + 3]));
          }
#pragma unroll
          for (int part = 0; part < 2; ++part) {
            const uint32_t(&v)[32] = part == 0 ? vc : vd;
            __syncwarp();  // the last pass has read the staging tile
            // row `lane` of the warp: 16-byte chunk j at chunk j ^ (lane & 7)
#pragma unroll
            for (int j = 0; j < 8; ++j)
              reinterpret_cast<float4*>(swp + lane * 32)[j ^ (lane & 7)] =
                  make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                              __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
            __syncwarp();
            float sum = 0.f;  // column `lane` of the chunk over the warp's rows, in row order
#pragma unroll 8
            for (int r = 0; r < 32; ++r) sum += swp[r * 32 + ((((lane >> 2) ^ (r & 7))) << 2) + (lane & 3)];
            wred[(quad * 2 + part) * 128 + 32 * c + lane] = sum;
          }
        }
        named_bar_sync(2, 128);
        {
          const int et = threadIdx.x - 64;  // epilogue thread 0 .. 127: one column of each part
          float* pp = p.part + ((static_cast<size_t>(b) * p.nmt + g.m0 / 128) * p.H + h) * 2 * D;
          if (et < D) {
#pragma unroll
            for (int part = 0; part < 2; ++part)
              pp[part * D + et] = ((wred[(0 * 2 + part) * 128 + et] + wred[(1 * 2 + part) * 128 + et]) +
                                   wred[(2 * 2 + part) * 128 + et]) +
                                  wred[(3 * 2 + part) * 128 + et];
          }
        }
        named_bar_sync(2, 128);  // the sums are read before the next DQ tile writes them
        continue;
      }
      float* dst = nullptr;
      const bool add = g.mode == kModeDR && p.accumulate;
      if (g.mode == kModeDR) {
        if (row < p.L) dst = p.dr + (static_cast<size_t>(row) * p.H + g.z) * D;
      } else if (row >= 0 && row < p.W) {
        const int b = g.z / p.H, h = g.z % p.H;
        dst = (g.mode == kModeDK ? p.dk : p.dv) + ((static_cast<size_t>(b) * p.W + row) * p.H + h) * D;
      }
      // the first ks keys of a tile after the first: queries [row, m0 + ks)
      const int tri_end = g.mode != kModeDR && g.m0 > 0 && row < g.m0 + p.ks ? min(g.m0 + p.ks, p.W) : 0;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(acc_col + 32 * c, v);
        tmem_wait_ld(v);
        if (c == D / 32 - 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->acc_empty[acc]);
        }
        if (dst != nullptr && row < tri_end) {
          // DK: sum_i G[i][M+row] (q+u)_i; DV: sum_i P[i][M+row] dout_i, in query order
          const int b = g.z / p.H, h = g.z % p.H;
          const __nv_bfloat16* X = (g.mode == kModeDK ? p.G : p.P) + static_cast<size_t>(g.z) * p.W * p.LP + p.M + row;
          const __nv_bfloat16* Y = g.mode == kModeDK ? p.qu : p.dout;
          for (int i = row; i < tri_end; ++i) {
            const float x = __bfloat162float(X[static_cast<size_t>(i) * p.LP]);
            const uint4* yr = reinterpret_cast<const uint4*>(Y + ((static_cast<size_t>(b) * p.W + i) * p.H + h) * D + 32 * c);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              const uint4 y = yr[q4];
              const uint32_t yw[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int j = 8 * q4 + 2 * e;
                v[j] = __float_as_uint(fmaf(x, bf16_lo(yw[e]), __uint_as_float(v[j])));
                v[j + 1] = __float_as_uint(fmaf(x, bf16_hi(yw[e]), __uint_as_float(v[j + 1])));
              }
            }
          }
        }
        if (dst != nullptr) {
          float4* o4 = reinterpret_cast<float4*>(dst + 32 * c);
          if (add) {
            // each (distance, head) row belongs to one tile: a plain read-add-write
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float4 x = o4[j];
              o4[j] = make_float4(x.x + __uint_as_float(v[4 * j]), x.y + __uint_as_float(v[4 * j + 1]),
                                  x.z + __uint_as_float(v[4 * j + 2]), x.w + __uint_as_float(v[4 * j + 3]));
            }
          } else {
#pragma unroll
            for (int j = 0; j < 8; ++j)
              o4[j] = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                  __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
          }
        }
      }
    }
    if (!ok) report_timeout(abort, p.status);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kGTmemCols);
  }
}

int num_sms() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  int n = cached[dev].load();
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cached[dev].store(n);
  }
  return n;
}

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

struct PairScratch {
  __nv_bfloat16 *G, *P, *GS, *Qu, *Qv;
  float* part;
  unsigned int* ctr;  // the products' tile counter
  size_t bytes;
};

// Scratch of one chunk of Bc sequences, then the bias partials of all chunks.
PairScratch carve(void* base, int Bc, int W, int M, int H, int D, size_t n_part) {
  const size_t L = static_cast<size_t>(M) + W, LP = (L + 63) / 64 * 64;
  const size_t bh = static_cast<size_t>(Bc) * H, bwhd = static_cast<size_t>(Bc) * W * H * D;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += round256(bytes);
    return static_cast<char*>(base) + at;
  };
  PairScratch s;
  s.G = reinterpret_cast<__nv_bfloat16*>(take(bh * W * LP * 2));
  s.P = reinterpret_cast<__nv_bfloat16*>(take(bh * W * LP * 2));
  s.GS = reinterpret_cast<__nv_bfloat16*>(take(bh * W * LP * 2));
  s.Qu = reinterpret_cast<__nv_bfloat16*>(take(bwhd * 2));
  s.Qv = reinterpret_cast<__nv_bfloat16*>(take(bwhd * 2));
  s.part = reinterpret_cast<float*>(take(n_part * H * 2 * D * 4));
  s.ctr = reinterpret_cast<unsigned int*>(take(sizeof(unsigned int)));
  s.bytes = off;
  return s;
}

// Sequences per chunk: as many as keep one chunk's scratch within the cap
// (at least one).  Later chunks reuse the scratch; dr accumulates over them.
std::atomic<size_t> g_chunk_cap{size_t(1) << 30};

int chunk_seqs(int B, int W, int M, int H, int D) {
  const size_t one = carve(nullptr, 1, W, M, H, D, 0).bytes;
  const size_t c = g_chunk_cap.load() / (one == 0 ? 1 : one);
  return static_cast<int>(std::max<size_t>(1, std::min<size_t>(c, static_cast<size_t>(B))));
}

// How many of the longest query tiles the pair kernel runs as two CTAs per
// unit (0-2).  CTAs start in launch order on whichever SM frees first, so the
// launch is list scheduling over the SMs; its length is modelled with a CTA
// costing its key steps plus 3 (the start and end of a CTA: about 6.7 us
// against 2.25 us a step at the wide workload, B=8 H=8 W=M=768), and the
// count with the shortest modelled launch is taken.  At wide, splitting the
// last tile's 24-step units turns 384 CTAs of 14-24 steps into 448 and the
// modelled length from 146 to 133 us.
int pair_split_tiles(int nqt, int bh, int W, int M, int sms) {
  if (bh <= 0 || sms <= 0 || static_cast<long long>(nqt + 2) * bh > 200000) return 0;
  auto steps = [&](int qt) { return std::min(M + qt * BM + BM - 1, M + W - 1) / BN + 1; };
  std::vector<long long> load(static_cast<size_t>(sms));
  auto span = [&](int k) {
    std::fill(load.begin(), load.end(), 0LL);
    std::priority_queue<long long, std::vector<long long>, std::greater<long long>> heap(load.begin(), load.end());
    auto put = [&](long long c) {
      const long long l = heap.top();
      heap.pop();
      heap.push(l + c);
    };
    for (int qt = nqt - k - 1; qt >= 0; --qt)
      for (int x = 0; x < bh; ++x) put(3 + steps(qt));
    for (int j = 0; j < 2 * k; ++j) {
      const int n = steps(nqt - 1 - (j >> 1));
      for (int x = 0; x < bh; ++x) put(3 + ((j & 1) ? n - n / 2 : n / 2));
    }
    long long m = 0;
    while (!heap.empty()) {
      m = std::max(m, heap.top());
      heap.pop();
    }
    return m;
  };
  int best = 0;
  long long best_span = span(0);
  for (int k = 1; k <= std::min(nqt, 2); ++k) {
    if (steps(nqt - k) < 4) break;  // halves of at least two steps
    const long long v = span(k);
    if (v < best_span) {
      best_span = v;
      best = k;
    }
  }
  return best;
}

// Bias partials: one per (sequence, 128-row block) of every chunk.
size_t total_parts(int B, int W) { return static_cast<size_t>(B) * ((W + 127) / 128); }

template <int D>
cudaError_t launch_products(const GMaps& maps, GemmArgs p, cudaStream_t stream) {
  constexpr int kGSmem = GemmCfg<D>::kGSmem;
  static std::atomic<bool> attr_done[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_done[dev].load()) {
    if ((e = cudaFuncSetAttribute(bgemm_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, kGSmem)) !=
        cudaSuccess)
      return e;
    attr_done[dev].store(true);
  }
  const int grid = std::min(p.total, num_sms());
  return launch_dependent(bgemm_kernel<D>, dim3(grid), dim3(kGThreads), kGSmem, stream, maps, p);
}

}  // namespace

int relattn_bwd_pairs_split_tiles(int nqt, int bh, int W, int M, int sms) {
  return pair_split_tiles(nqt, bh, W, M, sms);
}

int relattn_bwd_pairs_work(int B, int W, int M, int H, int split_qt, int* n_ctas, int* n_tiles, int* ctas,
                           int cap_ctas, int* tiles, int cap_tiles) {
  if (B < 0 || W < 0 || M < 0 || H < 0 || n_ctas == nullptr || n_tiles == nullptr) return -1;
  ScoreParams p{};
  p.B = B;
  p.W = W;
  p.M = M;
  p.H = H;
  p.nqt = (W + BM - 1) / BM;
  if (split_qt < 0 || split_qt > std::min(p.nqt, 2)) return -1;
  p.split_qt = split_qt;
  GemmArgs g{};
  const long long units = static_cast<long long>(p.nqt + split_qt) * B * H;
  if (units > 0x7FFFFFFFLL || !product_geometry(g, B, W, M, H)) return -1;
  *n_ctas = static_cast<int>(units);
  *n_tiles = g.total;
  if ((ctas != nullptr && cap_ctas < *n_ctas) || (tiles != nullptr && cap_tiles < *n_tiles)) return -2;
  for (int u = 0; ctas != nullptr && u < *n_ctas; ++u) {
    const Unit w = pair_item(u, p);
    const int row[5] = {w.b, w.h, w.i0, w.t0, w.nks};
    std::copy(row, row + 5, ctas + 5 * static_cast<size_t>(u));
  }
  for (int u = 0; tiles != nullptr && u < *n_tiles; ++u) {
    const GTile t = gtile(g, u);
    const int row[6] = {t.mode, t.z, t.m0, t.kb0, t.nkb, t.nkb_c};
    std::copy(row, row + 6, tiles + 6 * static_cast<size_t>(u));
  }
  return 0;
}

void relattn_bwd_pairs_set_chunk_bytes(size_t bytes) { g_chunk_cap.store(bytes == 0 ? size_t(1) << 30 : bytes); }

size_t relattn_bwd_pairs_scratch_bytes(int B, int W, int M, int H, int D) {
  const int Bc = chunk_seqs(B, W, M, H, D);
  return carve(nullptr, Bc, W, M, H, D, total_parts(B, W)).bytes;
}

bool relattn_bwd_pairs_supported(int W, int M, int D) { return W > 0 && M >= 0 && (D == 64 || D == 128); }

namespace {

template <int D>
cudaError_t launch_pairs(PFN_cuTensorMapEncodeTiled_v12000 encode, const void* q, const void* k, const void* v,
                         const void* r, const float* bias_u, const float* bias_v, const float* lse, const void* o,
                         const void* dout, float* dq, float* dk, float* dv, float* dr, float* du, float* dvb, int B,
                         int W, int M, int H, int n_r, float scale, void* scratch, const WaitCtl& wc,
                         cudaStream_t stream) {
  if (encode == nullptr || !relattn_bwd_pairs_supported(W, M, D)) return cudaErrorInvalidValue;
  constexpr int kSSmem = PairCfg<D>::kSSmem;
  const int L = M + W, LP = (L + 63) / 64 * 64;
  const int Bc = chunk_seqs(B, W, M, H, D);
  const PairScratch sc = carve(scratch, Bc, W, M, H, D, total_parts(B, W));
  const cuuint64_t hd2 = static_cast<cuuint64_t>(H) * D * 2;
  bool ok = true;
  auto enc = [&](CUtensorMap* m, const void* base, int rank, std::initializer_list<cuuint64_t> dims,
                 std::initializer_list<cuuint64_t> strides, std::initializer_list<cuuint32_t> box) {
    cuuint64_t dd[4];
    cuuint64_t ss[3];
    cuuint32_t bb[4];
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    int n = 0;
    for (cuuint64_t x : dims) dd[n++] = x;
    n = 0;
    for (cuuint64_t x : strides) ss[n++] = x;
    n = 0;
    for (cuuint32_t x : box) bb[n++] = x;
    ok = ok && encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dd, ss, bb, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  };
  const cuuint64_t d_ = D, h_ = H, w_ = W, l_ = L;
  const cuuint64_t lp2 = static_cast<cuuint64_t>(LP) * 2;
  // r and the chunk's scratch do not move between chunks
  GMaps gm;  // the products' maps
  CUtensorMap tpk;
  enc(&gm.b_r, r, 3, {d_, h_, static_cast<cuuint64_t>(n_r)}, {d_ * 2, hd2}, {64, 1, 64});
  auto enc_scratch = [&](int nb) {
    const cuuint64_t bh_ = static_cast<cuuint64_t>(nb) * H, b_ = nb;
    // G, P, GS: [nb*H][W][LP] bf16 (columns past L zero-filled); q+u, q+v: [nb, W, H, D]
    enc(&gm.a_g, sc.G, 3, {l_, w_, bh_}, {lp2, w_ * lp2}, {64, 128, 1});
    enc(&gm.a_gs, sc.GS, 3, {l_, w_, bh_}, {lp2, w_ * lp2}, {64, 128, 1});
    enc(&tpk, sc.P, 3, {l_, w_, bh_}, {lp2, w_ * lp2}, {64, 128, 1});
    enc(&gm.m_g, sc.G, 3, {l_, w_, bh_}, {lp2, w_ * lp2}, {64, 64, 1});
    enc(&gm.m_p, sc.P, 3, {l_, w_, bh_}, {lp2, w_ * lp2}, {64, 64, 1});
    enc(&gm.m_gs, sc.GS, 3, {l_, w_, bh_}, {lp2, w_ * lp2}, {64, 64, 1});
    enc(&gm.b_qu, sc.Qu, 4, {d_, h_, w_, b_}, {d_ * 2, hd2, w_ * hd2}, {64, 1, 64, 1});
    enc(&gm.b_qv, sc.Qv, 4, {d_, h_, w_, b_}, {d_ * 2, hd2, w_ * hd2}, {64, 1, 64, 1});
  };

  cudaError_t e;
  {
    static std::atomic<bool> attr_done[64];
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_done[dev].load()) {
      if ((e = cudaFuncSetAttribute(bwd_pairs_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSSmem)) !=
          cudaSuccess)
        return e;
      attr_done[dev].store(true);
    }
  }
  const size_t seg = static_cast<size_t>(W) * H * D;      // one sequence of q, o, dout, dq, dk, dv
  const size_t mem = static_cast<size_t>(L) * H * D;      // one sequence of k, v
  const int nmt = (W + 127) / 128;
  int last_nb = -1;
  for (int b0 = 0; b0 < B; b0 += Bc) {
    const int nb = std::min(Bc, B - b0);
    const __nv_bfloat16* qb = static_cast<const __nv_bfloat16*>(q) + b0 * seg;
    const __nv_bfloat16* kb = static_cast<const __nv_bfloat16*>(k) + b0 * mem;
    const __nv_bfloat16* vb = static_cast<const __nv_bfloat16*>(v) + b0 * mem;
    const __nv_bfloat16* ob = static_cast<const __nv_bfloat16*>(o) + b0 * seg;
    const __nv_bfloat16* gb = static_cast<const __nv_bfloat16*>(dout) + b0 * seg;
    const cuuint64_t b_ = nb;
    CUtensorMap tq, tdo128, tv;
    enc(&tq, qb, 4, {d_, h_, w_, b_}, {d_ * 2, hd2, w_ * hd2}, {64, 1, 128, 1});
    enc(&tdo128, gb, 4, {d_, h_, w_, b_}, {d_ * 2, hd2, w_ * hd2}, {64, 1, 128, 1});
    enc(&gm.b_k, kb, 4, {d_, h_, l_, b_}, {d_ * 2, hd2, l_ * hd2}, {64, 1, 64, 1});
    enc(&tv, vb, 4, {d_, h_, l_, b_}, {d_ * 2, hd2, l_ * hd2}, {64, 1, 64, 1});
    enc(&gm.b_do, gb, 4, {d_, h_, w_, b_}, {d_ * 2, hd2, w_ * hd2}, {64, 1, 64, 1});
    if (nb != last_nb) {
      enc_scratch(nb);
      last_nb = nb;
    }
    if (!ok) return cudaErrorInvalidValue;
    // 1. pair terms -> G, P, GS, q+u, q+v
    ScoreParams p;
    p.bias_u = bias_u;
    p.bias_v = bias_v;
    p.lse = lse + static_cast<size_t>(b0) * H * W;
    p.o = ob;
    p.dout = gb;
    p.GS = sc.GS;
    p.Qu = sc.Qu;
    p.Qv = sc.Qv;
    p.B = nb;
    p.W = W;
    p.M = M;
    p.H = H;
    p.nqt = (W + BM - 1) / BM;
    p.LP = LP;
    p.scale = scale;
    p.scale_log2e = scale * kLog2e;
    p.status = wc.status;
    p.wait_ns = wc.limit_ns;
    p.inject_stall = b0 == 0 ? wc.inject_stall : 0;
    p.gemm_ctr = sc.ctr;
    p.split_qt = pair_split_tiles(p.nqt, nb * H, W, M, num_sms());
    const long long units = static_cast<long long>(p.nqt + p.split_qt) * nb * H;
    if (units > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    if ((e = launch_dependent(bwd_pairs_kernel<D>, dim3(static_cast<unsigned>(units)), dim3(kSThreads), kSSmem,
                              stream, tq, gm.b_k, tv, gm.b_r, tdo128, gm.a_g, tpk, p)) != cudaSuccess)
      return e;
    // 2. the products, one launch: DR, DQ, DK and DV tiles from the counter
    // that the pair kernel has just zeroed
    GemmArgs g;
    if (!product_geometry(g, nb, W, M, H)) return cudaErrorInvalidValue;
    g.LP = LP;
    g.G = sc.G;
    g.P = sc.P;
    g.qu = sc.Qu;
    g.dout = gb;
    g.dq = dq + b0 * seg;
    g.dk = dk + b0 * seg;
    g.dv = dv + b0 * seg;
    g.dr = dr;
    g.part = sc.part + static_cast<size_t>(b0) * nmt * H * 2 * D;
    g.accumulate = b0 > 0;
    g.ctr = sc.ctr;
    g.status = wc.status;
    g.wait_ns = wc.limit_ns;
    if ((e = launch_products<D>(gm, g, stream)) != cudaSuccess) return e;
  }
  if (n_r > L &&
      (e = cudaMemsetAsync(dr + static_cast<size_t>(L) * H * D, 0, static_cast<size_t>(n_r - L) * H * D * 4,
                           stream)) != cudaSuccess)
    return e;
  const size_t n_part = total_parts(B, W);
  if (n_part > 0x7FFFFFFF) return cudaErrorInvalidValue;
  return launch_bwd_bias(sc.part, static_cast<int>(n_part), H, D, du, dvb, stream);
}

}  // namespace

cudaError_t launch_relattn_bwd_pairs(PFN_cuTensorMapEncodeTiled_v12000 encode, const void* q, const void* k,
                                     const void* v, const void* r, const float* bias_u, const float* bias_v,
                                     const float* lse, const void* o, const void* dout, float* dq, float* dk,
                                     float* dv, float* dr, float* du, float* dvb, int B, int W, int M, int H, int D,
                                     int n_r, float scale, void* scratch, const WaitCtl& wc, cudaStream_t stream) {
  if (D == 64)
    return launch_pairs<64>(encode, q, k, v, r, bias_u, bias_v, lse, o, dout, dq, dk, dv, dr, du, dvb, B, W, M, H,
                            n_r, scale, scratch, wc, stream);
  if (D == 128)
    return launch_pairs<128>(encode, q, k, v, r, bias_u, bias_v, lse, o, dout, dq, dk, dv, dr, du, dvb, B, W, M, H,
                             n_r, scale, scratch, wc, stream);
  return cudaErrorInvalidValue;
}

}  // namespace txl
