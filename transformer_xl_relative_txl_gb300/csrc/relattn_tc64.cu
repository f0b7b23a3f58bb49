// bf16 relative-position attention on the sm_103a tensor cores, head dimension
// 64 (tcgen05 + TMEM + TMA, fp32 accumulation).
//
//   s[i,j] = scale * ((q_i + u) . k_j + (q_i + v) . r_{M+i-j}),   j <= M+i
//   o_i = softmax(s[i,.]) V
//
// Same operation, tiling and distance indexing as the general kernel in
// relattn_tc.cu ("Transformer-XL, explained", method steps 3-5: keys and
// values over [memory ; segment], the four-term relative score grouped by its
// query-side factor, the distance term computed once per distance in a ring
// of 64-distance tiles and shifted into place per row by an index).  What
// differs is how the work is spread at D = 64, where the per-element softmax
// work, not the tensor core, bounds the kernel:
//
//   * The two softmax warps that share a TMEM lane quadrant take alternate
//     64-key steps instead of halves of every step.  Each warp owns a whole
//     step (one 96-distance window per 64 columns, no per-step exchange of
//     row maxima) and its own output accumulator, O0 for even steps and O1
//     for odd ones; the warps of a unit's last step merge the two with their
//     running maxima and sums while the other parity starts the next unit.
//     Each warp has two steps' time for one step, which hides the latency of
//     its dependent chains behind the other warp.
//   * The distance ring has four slots: the tile that step t adds reuses the
//     slot of tile t-4, last read by step t-2, so the distance MMAs run a
//     full step ahead of the softmax instead of waiting on its previous step.
//     The ring continues across units, so the next unit's first tiles are
//     computed while this unit's last step runs.
//   * A softmax warp reads everything a step needs from TMEM (S and the
//     distance window) in one batch and signals it with a single arrival
//     (one barrier per step modulo 4); the content-MMA issuer reuses the S
//     buffer and the distance-MMA issuer a ring slot once the steps that
//     read them have signalled.
//     The TMEM for the fourth slot comes from keeping P in shared memory
//     (both PV operands are then shared-memory descriptors).
//   * (q+u) and (q+v) are double-buffered in shared memory (128B-swizzled
//     K-major tiles) and the next unit's pair is built right after each
//     warp's first step of the current unit, half of the head dimensions by
//     each step parity, so no unit boundary waits for it.
//   * bf16 output is staged in the epilogue warp's idle P quadrant and
//     written by a TMA store.
//
// TMEM (512 columns): O0 [0,64) O1 [64,128) S0 [128,192) S1 [192,256)
// distance ring [256,512).
//
// Warps: 0-7 softmax (warp w: lane quadrant w%4, step parity w/4); 8 TMA
// loader; 9 content-score MMA issuer (owns the TMEM allocation); 10 PV MMA
// issuer; 11 distance-score MMA issuer.  A tcgen05.mma costs tens of cycles
// to issue and each barrier wait or commit more under load, so the three MMA
// streams get their own threads; their waits overlap and each commits its own
// MMAs.  Persistent CTAs walk (batch, head, 128-query tile) units longest
// first, dealt to the CTAs in a snake order.  Every wait is bounded; a wait
// that runs out raises a CTA abort flag and the device status word, every
// role unwinds (the loader and the issuers wait for their own operations in
// flight) and the TMEM is freed before exit.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <queue>
#include <tuple>
#include <type_traits>
#include <vector>

#include "pdl.cuh"
#include "relattn_tc_common.cuh"
#include "txl_device.cuh"
#include "txl_internal.h"

namespace txl {
namespace {

constexpr int BM = kTileRows;
constexpr int BN = kStepKeys;
constexpr int D = 64;
constexpr int kLoaderWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kPvWarp = 10;
constexpr int kQrWarp = 11;
constexpr int kThreads = 384;  // 3 warpgroups: 2 softmax, 1 producer (loader, three MMA issuers)
// Register split (launch: 168 per thread, 384 x 168 = 64512): softmax
// warpgroups 224, producer warpgroup 56; 2*128*224 + 128*56 = 64512, and per
// scheduler 224 + 224 + 56 = 504 <= 512 per thread-slot.
constexpr uint32_t kRegsSoftmax = 224;
constexpr uint32_t kRegsProducer = 56;
static_assert(2 * 128 * kRegsSoftmax + 128 * kRegsProducer <= kThreads * 168, "register split");
constexpr uint32_t kColO = 0;    // O0, O1: 64 columns each
constexpr uint32_t kColS = 128;  // S0, S1: 64 columns each
constexpr uint32_t kColG = 256;  // distance ring: 4 slots of 64 columns
constexpr int kSlots = 4;
static_assert(kSlots == 4, "ring slot counters and barrier init assume four slots");
constexpr uint32_t kTmemCols = 512;
constexpr float kLazy = 8.0f;  // log2 headroom before a running max moves

constexpr int kRowTile = BN * 128;  // 64 rows x 64 bf16 (8 KB)
constexpr int kQTile = BM * 128;    // 128 rows x 64 bf16 (16 KB)
constexpr int NK = 4, NV = 4, NR = 4;  // K, V, R tile stages
static_assert(NK == NV, "K and V tiles share the loader's stage logic");
constexpr int kOffQ = 0;                        // raw q tile of the next unit (TMA)
constexpr int kOffQu = kOffQ + kQTile;          // (q+u): 2 buffers
constexpr int kOffQv = kOffQu + 2 * kQTile;     // (q+v): 2 buffers
constexpr int kOffK = kOffQv + 2 * kQTile;
constexpr int kOffV = kOffK + NK * kRowTile;
constexpr int kOffR = kOffV + NV * kRowTile;
constexpr int kOffP = kOffR + NR * kRowTile;    // P (bf16): 2 buffers, same layout as (q+u)
constexpr int kOffRed = kOffP + 2 * kQTile;     // [unit parity][m, l][row] handed to the epilogue
constexpr int kOffBias = kOffRed + 2 * 2 * BM * 4;  // per softmax warp: 32 dims of u, then of v (fp32)
constexpr int kOffBar = kOffBias + 8 * 64 * 4;
constexpr int kSmemBytes = kOffBar + 512 + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct Params {
  const float* bias_u;
  const float* bias_v;
  void* o;
  float* lse;
  int B, W, M, H;
  int nqt, n_units;  // n_units: work items (units x nsplit)
  int nsplit;        // > 1: key steps split into chunks; partial results go to part_o / part_lse
  float* part_o;     // [item][128 rows][D] fp32, o of the chunk (normalised by its own sum)
  float* part_lse;   // [item][128 rows] fp32, log2-domain lse of the chunk (-inf: no visible key)
  int* part_cnt;     // [unit][4 quadrants] chunks finished; zero between launches
  float scale_log2e;  // |scale| * log2(e)
  float qsign;        // sign of scale, folded into (q+u), (q+v)
  unsigned int* status;
  unsigned long long wait_ns;
  int inject_stall;
  const int* sched;   // host-made unit table [grid][sched_stride] (-1 ends a row); nullptr: snake order
  int sched_stride;
  int roll_src0;  // >= 0: memory roll of k, v rows [roll_src0, M+W) by the last query tile's units
  // ring_cap > 0: keys and values come from two places -- memory row m
  // (m < M) is row (ring_start + m) % ring_cap of the ring maps tm_k / tm_v,
  // segment row x is row x of tm_ks / tm_vs.  ring_start, ring_cap and M are
  // multiples of 64, so a key tile never wraps or straddles the two.
  int ring_cap, ring_start;
  int ring_append;  // ring: also store the segment's k, v tiles into ring rows (start + M + x) % cap
};

struct Bars {
  uint64_t fullK[NK], emptyK[NK], fullV[NV], emptyV[NV], fullR[NR], emptyR[NR];
  uint64_t q_full, q_empty;
  uint64_t q_ready, s_full[2], p_full[2], pv_done[2], o_full, o_free;
  uint64_t sread[4];  // step g's S and distance window have been read (index g % 4, phase g / 4)
  uint64_t mma_final, pv_final, qr_final;
  uint64_t lbar[4];   // per quadrant: the non-owning warp's (m, l) of a unit is in `red`
  uint64_t lfree[4];  // per quadrant: the epilogue has read it
  int vq[4][5];       // loader: queued V tiles (key row, batch, head, roll, unit ordinal), by V count % 4
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Bars) <= 512, "barrier block too large");

template <bool O_BF16, bool SPLIT, bool RING>
__global__ void __launch_bounds__(kThreads, 1)
    relattn_tc64_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_r,
                        const __grid_constant__ CUtensorMap tm_o, const __grid_constant__ CUtensorMap tm_km,
                        const __grid_constant__ CUtensorMap tm_vm, const __grid_constant__ CUtensorMap tm_ks,
                        const __grid_constant__ CUtensorMap tm_vs, const Params p) {
  // Launched behind the previous kernel on the stream, which has completed from
  // here on.  No early trigger: the next persistent launch starts its CTAs when
  // this one completes (placed early, they timed slower back to back).
  grid_dep_wait();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  uint8_t* sQ = smem + kOffQ;
  uint8_t* sQu = smem + kOffQu;
  uint8_t* sQv = smem + kOffQv;
  uint8_t* sK = smem + kOffK;
  uint8_t* sV = smem + kOffV;
  uint8_t* sR = smem + kOffR;
  uint8_t* sP = smem + kOffP;
  float* red = reinterpret_cast<float*>(smem + kOffRed);
  float* sbias = reinterpret_cast<float*>(smem + kOffBias);
  Bars* bars = reinterpret_cast<Bars*>(smem + kOffBar);
  volatile int* abort = &bars->abort;
  const int kSplit = SPLIT ? p.nsplit : 1;  // chunks per unit

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < 4; ++s) {
      mbar_init(&bars->fullK[s], 1);
      mbar_init(&bars->emptyK[s], 1);
      mbar_init(&bars->fullV[s], 1);
      mbar_init(&bars->emptyV[s], 1);
      mbar_init(&bars->fullR[s], 1);
      mbar_init(&bars->emptyR[s], 1);
      mbar_init(&bars->lbar[s], 32);
      mbar_init(&bars->lfree[s], 1);
      mbar_init(&bars->sread[s], 4);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->s_full[s], 2);  // content and distance MMAs of a step
      mbar_init(&bars->p_full[s], 4);
      mbar_init(&bars->pv_done[s], 1);
    }
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 8);
    mbar_init(&bars->q_ready, 8);
    mbar_init(&bars->o_full, 1);
    mbar_init(&bars->o_free, 4);
    mbar_init(&bars->mma_final, 1);
    mbar_init(&bars->pv_final, 1);
    mbar_init(&bars->qr_final, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const uint64_t wait_ns = p.wait_ns;

  if (warp == kLoaderWarp) {
    // ============================ TMA loader ===============================
    setmaxnreg_dec<kRegsProducer>();
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_r);
      uint32_t nQ = 0, nK = 0, nV = 0, nR = 0;
      bool ok = true, stop = false;
      // Memory roll: the unit of the last query tile of each (batch, head)
      // loads every key and value row once.  A K or V tile whose rows lie in
      // the kept range is stored from its stage to the memory output just
      // before the stage is refilled (its MMA has consumed it by then), or at
      // the end.  Per K and per V stage: destination row of the pending store
      // (-1: none), batch and head (kept apart for K and V: a K stage is
      // refilled before the V stage of the same index).
      int pk_row[NK], pk_b[NK], pk_h[NK], pv_row[NK], pv_b[NK], pv_h[NK];
#pragma unroll
      for (int s = 0; s < NK; ++s) pk_row[s] = pv_row[s] = -1;
      auto flush_store = [&](int* prow, const int* pb, const int* ph, int s, const CUtensorMap* map,
                             uint8_t* stage) {
        if (prow[s] >= 0) {
          tma_store_4d(map, stage, 0, ph[s], prow[s], pb[s]);
          bulk_commit_group();
          bulk_wait_group_read0();  // the stage is refilled next
          prow[s] = -1;
        }
      };
      auto acquire = [&](uint64_t* empty, uint64_t* full, uint32_t n, int ns, int bytes) -> bool {
        const int s = static_cast<int>(n % ns);
        if (!mbar_wait(&empty[s], ((n / ns) & 1) ^ 1, wait_ns, abort)) return false;
        mbar_arrive_expect_tx(&full[s], bytes);
        return true;
      };
      // The raw q tile of a unit is loaded one unit ahead: the softmax warps
      // build (q+u), (q+v) from it during the unit before.
      auto load_q = [&](int u) -> bool {
        if (!mbar_wait(&bars->q_empty, (nQ & 1) ^ 1, wait_ns, abort)) return false;
        mbar_arrive_expect_tx(&bars->q_full, kQTile);
        const Unit w = decode_item(u, kSplit, p.B, p.H, p.W, p.M, p.nqt);
        tma_load_4d(sQ, &tm_q, &bars->q_full, 0, w.h, w.i0, w.b);
        ++nQ;
        return true;
      };
      // K or V tile of key row kr (a multiple of 64) of batch b, head h into
      // the next stage of its stream; rl: the unit keeps these rows (roll).
      auto load_kv = [&](uint64_t* empty, uint64_t* full, uint8_t* dst, uint32_t& n, const CUtensorMap* map, int kr,
                         int b, int h, bool rl, int* prow, int* pb, int* ph, const CUtensorMap* rmap,
                         const CUtensorMap* smap) -> bool {
        const int s = static_cast<int>(n % NK);
        if (!mbar_wait(&empty[s], ((n / NK) & 1) ^ 1, wait_ns, abort)) return false;
        flush_store(prow, pb, ph, s, rmap, dst + s * kRowTile);
        mbar_arrive_expect_tx(&full[s], kRowTile);
        if constexpr (RING) {
          if (kr < p.M)  // start + kr < 2 cap: one conditional wrap
            tma_load_4d(dst + s * kRowTile, map, &full[s], 0, h,
                        p.ring_start + kr - (p.ring_start + kr >= p.ring_cap ? p.ring_cap : 0), b);
          else
            tma_load_4d(dst + s * kRowTile, smap, &full[s], 0, h, kr - p.M, b);
        } else {
          tma_load_4d(dst + s * kRowTile, map, &full[s], 0, h, kr, b);
        }
        if constexpr (RING)
          prow[s] = (rl && kr >= p.M)  // start + kr < start + M + W <= 2 cap
                        ? p.ring_start + kr - (p.ring_start + kr >= p.ring_cap ? p.ring_cap : 0)
                        : -1;
        else
          prow[s] = (rl && kr >= p.roll_src0) ? kr - p.roll_src0 : -1;
        pb[s] = b;
        ph[s] = h;
        ++n;
        return true;
      };
      // V tiles trail the K and R tiles by kVLag tiles.  A V stage is freed
      // only when the P.V MMA of its step completes, after that step's
      // softmax, while a K stage is free as soon as its score MMA is done; in
      // one issue order K(t), R(t+1), V(t), every K load would wait behind
      // the V stage of step t-4 and land just in time (the score issuer then
      // waits for it).  With V(t-2) after K(t), K and R run up to their full
      // stage depth ahead, and V(t) still lands two steps before its P.V.
      // Only the plain instantiation trails, the one where the gain was
      // measured; with split key ranges (about one item per CTA, whose first
      // P.V would wait longer for V) and with ring memory the two orders time
      // the same within the noise, so those keep V(t) right after K(t).
      // Queued V tiles wait in bars->vq (this thread only).  Before the raw
      // q of the unit after next is loaded, every queued V of a unit two or
      // more back goes out: that load waits for the (q+u), (q+v) build of the
      // next unit, which waits for the epilogue of the unit before, which
      // needs all of that unit's V tiles (a unit of one step would otherwise
      // hold them behind the load).
      constexpr uint32_t kVLag = (SPLIT || RING) ? 0 : 2;
      uint32_t nVq = 0;  // V tiles queued; nVq - nV of them not yet issued
      auto issue_v = [&]() -> bool {
        const int* e = bars->vq[nV % 4];
        return load_kv(bars->emptyV, bars->fullV, sV, nV, &tm_v, e[0], e[1], e[2], e[3] != 0, pv_row, pv_b, pv_h,
                       RING ? &tm_v : &tm_vm, &tm_vs);
      };
      if (const int u0 = unit_at(p.sched, p.sched_stride, 0, blockIdx.x, gridDim.x, p.n_units); u0 < p.n_units)
        ok = load_q(u0);
      for (int rd = 0;; ++rd) {
        const int u = unit_at(p.sched, p.sched_stride, rd, blockIdx.x, gridDim.x, p.n_units);
        if (!ok || stop || u >= p.n_units) break;
        const int un_next = unit_at(p.sched, p.sched_stride, rd + 1, blockIdx.x, gridDim.x, p.n_units);
        const Unit w = decode_item(u, kSplit, p.B, p.H, p.W, p.M, p.nqt);
        while (ok && nV < nVq && bars->vq[nV % 4][4] <= rd - 2) ok = issue_v();
        if (!ok) break;
        if (un_next < p.n_units && !(ok = load_q(un_next))) break;
        auto load_r = [&](int d0) -> bool {
          if (!acquire(bars->emptyR, bars->fullR, nR, NR, kRowTile)) return false;
          tma_load_3d(sR + (nR % NR) * kRowTile, &tm_r, &bars->fullR[nR % NR], 0, w.h, d0);
          ++nR;
          return true;
        };
        // last query tile: the roll (or, for a ring, the append of the
        // segment's rows into ring rows (start + M + x) % cap, which no unit
        // of this launch reads)
        const bool rolls = (RING ? p.ring_append != 0 : p.roll_src0 >= 0) && w.i0 + BM >= p.W;
        // distance tiles -2 and -1 of the item's first step
        ok = load_r(p.M + w.i0 - BN * (w.t0 - 1)) && load_r(p.M + w.i0 - BN * w.t0);
        for (int t = 0; ok && t < w.nks; ++t) {
          if (p.inject_stall && t == 1) {  // test hook: starve the consumers
            stop = true;
            break;
          }
          const int kr = (w.t0 + t) * BN;  // first key row of the tile
          ok = load_kv(bars->emptyK, bars->fullK, sK, nK, &tm_k, kr, w.b, w.h, rolls, pk_row, pk_b, pk_h,
                       RING ? &tm_k : &tm_km, &tm_ks) &&
               load_r(p.M + w.i0 - BN * (w.t0 + t + 1));
          if (ok) {
            int* e = bars->vq[nVq % 4];
            e[0] = kr;
            e[1] = w.b;
            e[2] = w.h;
            e[3] = rolls;
            e[4] = rd;
            ++nVq;
            if (nVq - nV > kVLag) ok = issue_v();
          }
        }
      }
      while (ok && !stop && nV < nVq) ok = issue_v();  // the last kVLag V tiles
      if (!ok) report_timeout(abort, p.status);
      auto drain = [&](uint64_t* full, uint32_t n, int ns) {
        for (int s = 0; s < ns && static_cast<uint32_t>(s) < n; ++s) {
          const uint32_t last = s + ((n - 1 - s) / ns) * ns;
          mbar_wait_own(&full[s], (last / ns) & 1, wait_ns);
        }
      };
      drain(&bars->q_full, nQ, 1);
      drain(bars->fullK, nK, NK);
      drain(bars->fullV, nV, NV);
      drain(bars->fullR, nR, NR);
      // Roll stores still pending: each waits for the MMAs that read its
      // stage's last tile (the stage's data stays until then), then stores.
      if (ok && !stop) {
        for (int s = 0; s < NK; ++s) {
          const uint32_t last = static_cast<uint32_t>(s) + ((nK - 1 - s) / NK) * NK;  // nK == nV
          if (pk_row[s] >= 0 && mbar_wait(&bars->emptyK[s], (last / NK) & 1, wait_ns, abort))
            flush_store(pk_row, pk_b, pk_h, s, RING ? &tm_k : &tm_km, sK + s * kRowTile);
          if (pv_row[s] >= 0 && mbar_wait(&bars->emptyV[s], (last / NV) & 1, wait_ns, abort))
            flush_store(pv_row, pv_b, pv_h, s, RING ? &tm_v : &tm_vm, sV + s * kRowTile);
        }
      }
      bulk_wait_group0();  // every roll store is complete before the CTA exits
    }
  } else if (warp == kMmaWarp) {
    // ===================== content-score MMA issuer ========================
    setmaxnreg_dec<kRegsProducer>();
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16(128, BN, false, false);
      const uint64_t dQu = sdesc_sw128(smem_u32(sQu), 16, 1024);
      const uint64_t dK = sdesc_sw128(smem_u32(sK), 16, 1024);
      constexpr uint32_t kTile16 = kRowTile >> 4;
      uint32_t nK = 0, gt = 0, un = 0;
      bool ok = true;
      for (int rd = 0;; ++rd) {
        const int u = unit_at(p.sched, p.sched_stride, rd, blockIdx.x, gridDim.x, p.n_units);
        if (!ok || u >= p.n_units) break;
        const Unit w = decode_item(u, kSplit, p.B, p.H, p.W, p.M, p.nqt);
        if (!(ok = mbar_wait(&bars->q_ready, un & 1, wait_ns, abort))) break;
        tc_fence_after();
        const uint32_t g0 = gt;
        for (int t = 0; t < w.nks; ++t) {
          const uint32_t g = g0 + t, sb = g & 1;
          // S buffer sb was last read by step g-2.
          if (g >= 2 && !(ok = mbar_wait(&bars->sread[(g - 2) & 3], ((g - 2) >> 2) & 1, wait_ns, abort))) break;
          const int sk = nK % NK;
          if (!(ok = mbar_wait(&bars->fullK[sk], (nK / NK) & 1, wait_ns, abort))) break;
          tc_fence_after();
          const uint64_t dk = dK + sk * kTile16;
          const uint32_t sd = tmem + kColS + sb * BN;
          const uint64_t dq = dQu + (un & 1) * (kQTile >> 4);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) mma_ss(sd, dq + kk * 2, dk + kk * 2, idS, kk > 0);
          tc_commit(&bars->emptyK[sk]);
          tc_commit(&bars->s_full[sb]);
          ++nK;
        }
        if (!ok) break;
        gt = g0 + w.nks;
        ++un;
      }
      if (!ok) report_timeout(abort, p.status);
      tc_commit(&bars->mma_final);
      mbar_wait_own(&bars->mma_final, 0, wait_ns);
    }
  } else if (warp == kQrWarp) {
    // ==================== distance-score MMA issuer ========================
    setmaxnreg_dec<kRegsProducer>();
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16(128, BN, false, false);
      const uint64_t dQv = sdesc_sw128(smem_u32(sQv), 16, 1024);
      const uint64_t dR = sdesc_sw128(smem_u32(sR), 16, 1024);
      constexpr uint32_t kTile16 = kRowTile >> 4;
      uint32_t nR = 0, gt = 0, un = 0;
      // Last global step that reads the tile now in each ring slot (-1: none).
      int last0 = -1, last1 = -1, last2 = -1, last3 = -1;
      int rb = 0;  // ring slot of the first distance tile (-2) of the unit
      bool ok = true;
      for (int rd = 0;; ++rd) {
        const int u = unit_at(p.sched, p.sched_stride, rd, blockIdx.x, gridDim.x, p.n_units);
        if (!ok || u >= p.n_units) break;
        const Unit w = decode_item(u, kSplit, p.B, p.H, p.W, p.M, p.nqt);
        if (!(ok = mbar_wait(&bars->q_ready, un & 1, wait_ns, abort))) break;
        tc_fence_after();
        const uint32_t g0 = gt;
        const uint64_t dq = dQv + (un & 1) * (kQTile >> 4);
        for (int t = 0; ok && t < w.nks; ++t) {
          const uint32_t sb = (g0 + t) & 1;
          for (int e = (t == 0 ? -2 : t); e <= t; ++e) {
            const int slot = (rb + e + 2) & (kSlots - 1);
            // The slot's previous tile is free once every step up to its
            // last reader L has read: steps of one parity read in order, so
            // waiting for steps L and L-1 covers both parities.  (Four
            // barriers by step % 4 keep these waits from aliasing: step L+3
            // cannot have read before this tile exists.)
            const int L = slot == 0 ? last0 : (slot == 1 ? last1 : (slot == 2 ? last2 : last3));
            if (L >= 0 && !(ok = mbar_wait(&bars->sread[L & 3], (L >> 2) & 1, wait_ns, abort))) break;
            if (L >= 1 && !(ok = mbar_wait(&bars->sread[(L - 1) & 3], ((L - 1) >> 2) & 1, wait_ns, abort))) break;
            const int sr = nR % NR;
            if (!(ok = mbar_wait(&bars->fullR[sr], (nR / NR) & 1, wait_ns, abort))) break;
            tc_fence_after();
            const uint64_t dr = dR + sr * kTile16;
            const uint32_t gd = tmem + kColG + slot * BN;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) mma_ss(gd, dq + kk * 2, dr + kk * 2, idS, kk > 0);
            tc_commit(&bars->emptyR[sr]);
            ++nR;
            const int lr = static_cast<int>(g0) + min(e + 2, w.nks - 1);  // tile e's last reader
            last0 = slot == 0 ? lr : last0;
            last1 = slot == 1 ? lr : last1;
            last2 = slot == 2 ? lr : last2;
            last3 = slot == 3 ? lr : last3;
          }
          if (!ok) break;
          tc_commit(&bars->s_full[sb]);
        }
        if (!ok) break;
        gt = g0 + w.nks;
        ++un;
        rb = (rb + w.nks + 2) & (kSlots - 1);
      }
      if (!ok) report_timeout(abort, p.status);
      tc_commit(&bars->qr_final);
      mbar_wait_own(&bars->qr_final, 0, wait_ns);
    }
  } else if (warp == kPvWarp) {
    // ============================ PV issuer ================================
    setmaxnreg_dec<kRegsProducer>();
    if (lane == 0) {
      constexpr uint32_t idO = idesc_bf16(128, D, false, true);
      const uint64_t dV = sdesc_sw128(smem_u32(sV), BN * 128, 1024);
      const uint64_t dP = sdesc_sw128(smem_u32(sP), 16, 1024);
      constexpr uint32_t kTile16 = kRowTile >> 4;
      uint32_t nV = 0, g = 0, un = 0;
      bool ok = true;
      for (int rd = 0;; ++rd) {
        const int u = unit_at(p.sched, p.sched_stride, rd, blockIdx.x, gridDim.x, p.n_units);
        if (!ok || u >= p.n_units) break;
        const Unit w = decode_item(u, kSplit, p.B, p.H, p.W, p.M, p.nqt);
        for (int t = 0; t < w.nks; ++t, ++g) {
          if (!(ok = mbar_wait(&bars->p_full[g & 1], (g >> 1) & 1, wait_ns, abort))) break;
          const int sv = nV % NV;
          if (!(ok = mbar_wait(&bars->fullV[sv], (nV / NV) & 1, wait_ns, abort))) break;
          // The first PV into each accumulator of a unit overwrites it: the
          // previous unit's epilogue must have read both.
          if (t < 2 && un > 0 && !(ok = mbar_wait(&bars->o_free, (un - 1) & 1, wait_ns, abort))) break;
          tc_fence_after();
          const uint64_t dv = dV + sv * kTile16;
          const uint64_t dp = dP + (g & 1) * (kQTile >> 4);
          const uint32_t od = tmem + kColO + (g & 1) * D;
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            mma_ss(od, dp + kk * 2, dv + ((kk * 16 * 128) >> 4), idO, t >= 2 || kk > 0);
          tc_commit(&bars->emptyV[sv]);
          tc_commit(&bars->pv_done[g & 1]);
          ++nV;
        }
        if (!ok) break;
        tc_commit(&bars->o_full);
        ++un;
      }
      if (!ok) report_timeout(abort, p.status);
      tc_commit(&bars->pv_final);
      mbar_wait_own(&bars->pv_final, 0, wait_ns);
    }
  } else {
    // ============================ softmax warps ============================
    setmaxnreg_inc<kRegsSoftmax>();
    const int par = warp >> 2;  // step parity taken by this warp
    const int quad = warp & 3;  // TMEM lane quadrant
    const int a = quad * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const float sl2 = p.scale_log2e;
    uint32_t gt = 0, un = 0, nQ = 0;
    int rb = 0;  // ring slot of the unit's distance tile -2 (continues across units)
    bool store_pending = false;  // lane 0 has a TMA store out of this warp's P quadrant
    bool ok = true;

    // (q + u), (q + v) of unit w into buffer `buf` (128B-swizzled K-major
    // tiles): this warp's row, head dimensions [32 par, 32 par + 32).
    // bu_l, bv_l: this lane's dims 32 par + lane of the unit's u and v (loaded
    // ahead by the caller, so their latency overlaps other work).
    auto build_q = [&](const Unit& w, int buf, float bu_l, float bv_l) -> bool {
      // This warp's 32 dims of u and v, staged once for broadcast reads.
      float* sb_w = sbias + warp * 64;
      sb_w[lane] = bu_l;
      sb_w[32 + lane] = bv_l;
      __syncwarp();
      if (!warp_wait(&bars->q_full, nQ & 1, wait_ns, abort)) return false;
      uint4 raw[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c = 4 * par + j;
        raw[j] = *reinterpret_cast<const uint4*>(sQ + (a / 8) * 1024 + (a % 8) * 128 + ((c ^ (a % 8)) * 16));
      }
      warp_arrive(&bars->q_empty);
      ++nQ;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c = 4 * par + j;
        const int off = buf * kQTile + (a / 8) * 1024 + (a % 8) * 128 + ((c ^ (a % 8)) * 16);
        const uint32_t w4[4] = {raw[j].x, raw[j].y, raw[j].z, raw[j].w};
        const float4 u0 = *reinterpret_cast<const float4*>(sb_w + 8 * j);
        const float4 u1 = *reinterpret_cast<const float4*>(sb_w + 8 * j + 4);
        const float4 v0 = *reinterpret_cast<const float4*>(sb_w + 32 + 8 * j);
        const float4 v1 = *reinterpret_cast<const float4*>(sb_w + 32 + 8 * j + 4);
        const float ub[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
        const float vb[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        uint32_t qu[4], qv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float x0 = bf16_lo(w4[e]), x1 = bf16_hi(w4[e]);
          qu[e] = pack_bf16x2((x0 + ub[2 * e]) * p.qsign, (x1 + ub[2 * e + 1]) * p.qsign);
          qv[e] = pack_bf16x2((x0 + vb[2 * e]) * p.qsign, (x1 + vb[2 * e + 1]) * p.qsign);
        }
        *reinterpret_cast<uint4*>(sQu + off) = make_uint4(qu[0], qu[1], qu[2], qu[3]);
        *reinterpret_cast<uint4*>(sQv + off) = make_uint4(qv[0], qv[1], qv[2], qv[3]);
      }
      warp_arrive_smem(&bars->q_ready);
      __syncwarp();  // sb_w is rewritten by the next build
      return true;
    };

    auto bias_of = [&](int u, const float* bias) -> float {
      return __ldg(bias + decode_item(u, kSplit, p.B, p.H, p.W, p.M, p.nqt).h * D + 32 * par + lane);
    };
    if (unit_at(p.sched, p.sched_stride, 0, blockIdx.x, gridDim.x, p.n_units) < p.n_units) {
      const int u0 = unit_at(p.sched, p.sched_stride, 0, blockIdx.x, gridDim.x, p.n_units);
      ok = build_q(decode_item(u0, kSplit, p.B, p.H, p.W, p.M, p.nqt), 0, bias_of(u0, p.bias_u), bias_of(u0, p.bias_v));
    }

    for (int rd = 0;; ++rd) {
      const int u = unit_at(p.sched, p.sched_stride, rd, blockIdx.x, gridDim.x, p.n_units);
      if (!ok || u >= p.n_units) break;
      const int un_next = unit_at(p.sched, p.sched_stride, rd + 1, blockIdx.x, gridDim.x, p.n_units);
      const Unit w = decode_item(u, kSplit, p.B, p.H, p.W, p.M, p.nqt);
      const uint32_t g0 = gt;
      const bool has_next = un_next < p.n_units;
      const float bu_next = has_next ? bias_of(un_next, p.bias_u) : 0.f;
      const float bv_next = has_next ? bias_of(un_next, p.bias_v) : 0.f;
      const int tl = w.nks - 1;
      const int first = (par - static_cast<int>(g0)) & 1;  // first local step of this warp
      float m_use = -INFINITY;  // running max in log2 units (lazy)
      float l_run = 0.f;
      for (int t = first; t <= tl; t += 2) {
        const uint32_t g = g0 + t, sb = g & 1;
        if (!(ok = warp_wait(&bars->s_full[sb], (g >> 1) & 1, wait_ns, abort))) break;
        tc_fence_after();
        // Distance window of this warp: ring-relative index z = 64 + a - c
        // (z < 64: tile t, < 128: tile t-1, else tile t-2).  Columns 0-31 use
        // z in [32 quad + 32, 32 quad + 96), columns 32-63 z in
        // [32 quad, 32 quad + 64); lane l of column k (within its half) sits
        // at window position l + 32 - k.
        auto zcol = [&](int z) -> uint32_t {
          return kColG + ((rb + t - (z >> 6) + 2) & (kSlots - 1)) * BN + (z & 63);
        };
        const uint32_t sc = tmem + lane_base + kColS + sb * BN;
        const int kt = w.t0 + t;                 // key step of the tile
        const int lim = p.M + w.i0 - BN * kt + a;  // column c visible iff c <= lim
        const bool diag = p.M + w.i0 - BN * kt + quad * 32 < 63;  // some lane of the warp masks
        const float m_old = m_use;
        float m_new = m_use;
        // All of this step's TMEM reads at once -- the 96-distance window and
        // both halves of S -- then one arrival hands the S buffer and the
        // ring slots back to the MMA issuers.
        float x[64];  // scores of the step's 64 columns
        {
          uint32_t bd0[16], bd1[16];
          uint32_t s0[32], s1[32];
          {
            uint32_t xa[32], xb[32], xc[32];
            tmem_ld32(tmem + lane_base + zcol(32 * quad), xa);
            tmem_ld32(tmem + lane_base + zcol(32 * quad + 32), xb);
            tmem_ld32(tmem + lane_base + zcol(32 * quad + 64), xc);
            tmem_ld32(sc, s0);
            tmem_ld32(sc + 32, s1);
            tmem_wait_ld(xa);
            tmem_wait_ld(xb);
            tmem_wait_ld(xc);
            tmem_wait_ld(s0);
            tmem_wait_ld(s1);
            warp_arrive_tc(&bars->sread[g & 3]);
            uint32_t pa[16], pb[16], pc[16];
            pack32(xa, pa);
            pack32(xb, pb);
            pack32(xc, pc);
            // columns 0-31 use window positions [32, 96), columns 32-63 [0, 64)
            window_shift_packed(pb, pc, lane, bd0);
            window_shift_packed(pa, pb, lane, bd1);
          }
          float* x0 = x;
          float* x1 = x + 32;
          add_window(s0, bd0, x0);
          add_window(s1, bd1, x1);
        }
        if (diag) {
#pragma unroll
          for (int k = 0; k < 64; ++k) x[k] = (k <= lim) ? x[k] : -INFINITY;
        }
        // Lazy running max over the step's 64 scores (log2 units).
        float t3[22];
#pragma unroll
        for (int n = 0; n < 21; ++n) t3[n] = max3f(x[3 * n], x[3 * n + 1], x[3 * n + 2]);
        t3[21] = x[63];
        float u7[8];
#pragma unroll
        for (int n = 0; n < 7; ++n) u7[n] = max3f(t3[3 * n], t3[3 * n + 1], t3[3 * n + 2]);
        u7[7] = t3[21];
        const float mx = max3f(max3f(u7[0], u7[1], u7[2]), max3f(u7[3], u7[4], u7[5]), fmaxf(u7[6], u7[7])) * sl2;
        if (mx > m_new + kLazy) m_new = mx;
        const float alpha = (m_old == -INFINITY) ? 0.f : ex2(m_old - m_new);  // m_new >= m_old
        // The PV of step g-2 (same P buffer, same accumulator) must be done
        // before P is overwritten or O rescaled.
        if (g >= 2 && !(ok = warp_wait(&bars->pv_done[sb], ((g - 2) >> 1) & 1, wait_ns, abort))) break;
        tc_fence_after();
        if (t > first && __any_sync(0xffffffffu, m_new > m_old)) {
          // O of this parity holds PV up to step t-2; rescale it in place.
          const uint32_t oc0 = tmem + lane_base + kColO + par * D;
#pragma unroll
          for (int oc = 0; oc < D / 32; ++oc) {
            uint32_t ov[32];
            tmem_ld32(oc0 + oc * 32, ov);
            tmem_wait_ld(ov);
#pragma unroll
            for (int n = 0; n < 32; ++n) ov[n] = __float_as_uint(__uint_as_float(ov[n]) * alpha);
            tmem_st32(oc0 + oc * 32, ov);
          }
          tmem_wait_st();
        }
        m_use = m_new;
        if (store_pending) {  // the last epilogue staged its output here
          if (lane == 0) bulk_wait_group_read0();
          __syncwarp();
          store_pending = false;
        }
        // A row with no visible key yet keeps m_new = -inf; its exponents are
        // then taken against 0 (all -inf, so every p is 0).
        const float m_eff = (m_new == -INFINITY) ? 0.f : m_new;
        float sum;
        {
          // Exponentials, their row sum, and the P row a into buffer sb
          // (128B-swizzled K-major, as (q+u)), eight columns per store.
          uint8_t* prow = sP + sb * kQTile + (a / 8) * 1024 + (a % 8) * 128;
          float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
          const float2 sc2 = make_float2(sl2, sl2), nm2 = make_float2(-m_eff, -m_eff);
#pragma unroll
          for (int c = 0; c < BN / 8; ++c) {
            uint32_t pk[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int n = 4 * c + i;
              const float2 y = __ffma2_rn(make_float2(x[2 * n], x[2 * n + 1]), sc2, nm2);
              const float2 e = make_float2(ex2(y.x), ex2(y.y));
              if (i & 1)
                acc1 = __fadd2_rn(acc1, e);
              else
                acc0 = __fadd2_rn(acc0, e);
              pk[i] = pack_bf16x2(e.x, e.y);
            }
            *reinterpret_cast<uint4*>(prow + ((c ^ (a % 8)) * 16)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          }
          sum = (acc0.x + acc0.y) + (acc1.x + acc1.y);
        }
        l_run = l_run * alpha + sum;
        tc_fence_before();  // orders the O rescale's tcgen05.st before the arrive
        warp_arrive_smem(&bars->p_full[sb]);
        // The next unit's (q+u), (q+v) go to the other buffer once this
        // warp's first step of this unit has seen its scores: the MMAs of the
        // unit before, which read that buffer, are complete by then.
        if (t == first && has_next &&
            !(ok = build_q(decode_item(un_next, kSplit, p.B, p.H, p.W, p.M, p.nqt), (un + 1) & 1, bu_next, bv_next)))
          break;
      }
      if (!ok) break;
      if (first > tl && has_next) {
        // No step of this unit: build after its last step's scores instead.
        const uint32_t gl = g0 + tl;
        if (!(ok = warp_wait(&bars->s_full[gl & 1], (gl >> 1) & 1, wait_ns, abort))) break;
        if (!(ok = build_q(decode_item(un_next, kSplit, p.B, p.H, p.W, p.M, p.nqt), (un + 1) & 1, bu_next, bv_next))) break;
      }
      // The warps of the unit's last step merge the two accumulators and
      // write the output; the other parity hands over its (m, l) and moves on
      // to the next unit, whose first step is its own.
      float* rm = red + (un & 1) * 2 * BM;
      const int owner = static_cast<int>((g0 + tl) & 1);
      if (par != owner) {
        // The owner of the previous unit has read that unit's (m, l).
        if (un > 0 && !(ok = warp_wait(&bars->lfree[quad], (un - 1) & 1, wait_ns, abort))) break;
        rm[a] = m_use;
        rm[BM + a] = l_run;
        mbar_arrive(&bars->lbar[quad]);
      } else {
        if (!(ok = warp_wait(&bars->lbar[quad], un & 1, wait_ns, abort))) break;
        const float m1 = rm[a], l1 = rm[BM + a];
        warp_arrive(&bars->lfree[quad]);
        if (!(ok = warp_wait(&bars->o_full, un & 1, wait_ns, abort))) break;
        tc_fence_after();
        // merge this parity's accumulator (0) with the other's (1)
        const bool has0 = first <= tl;        // this warp had steps
        const bool has1 = (first ^ 1) <= tl;  // the other parity's warp had steps
        const float m = fmaxf(has0 ? m_use : -INFINITY, has1 ? m1 : -INFINITY);
        // A row can see no key of an item only when the key steps are split.
        const bool any = m != -INFINITY;
        const float a0 = (has0 && any) ? ex2(m_use - m) : 0.f;
        const float a1 = (has1 && any) ? ex2(m1 - m) : 0.f;
        const float l = a0 * l_run + a1 * l1;
        const float inv_l = any ? 1.f / l : 0.f;
        const float c0 = a0 * inv_l, c1 = a1 * inv_l;
        // Read both accumulators into registers and hand them back to the PV
        // issuer before the stores.
        float ov[D];
#pragma unroll
        for (int oc = 0; oc < D / 32; ++oc) {
          uint32_t t0[32], t1[32];
          if (has0) {
            tmem_ld32(tmem + lane_base + kColO + par * D + oc * 32, t0);
            tmem_wait_ld(t0);
          }
          if (has1) {
            tmem_ld32(tmem + lane_base + kColO + (par ^ 1) * D + oc * 32, t1);
            tmem_wait_ld(t1);
          }
#pragma unroll
          for (int n = 0; n < 32; ++n)
            ov[oc * 32 + n] =
                (has0 ? __uint_as_float(t0[n]) * c0 : 0.f) + (has1 ? __uint_as_float(t1[n]) * c1 : 0.f);
        }
        warp_arrive_tc(&bars->o_free);
        const int i = w.i0 + a;
        if (SPLIT) {
          // This chunk's result for the warp's 32 rows goes to the scratch;
          // the warp that finishes a unit's rows last merges all chunks.
          const size_t it = static_cast<size_t>(u);
          float4* po = reinterpret_cast<float4*>(p.part_o + (it * BM + a) * D);
#pragma unroll
          for (int c = 0; c < D / 4; ++c) po[c] = make_float4(ov[4 * c], ov[4 * c + 1], ov[4 * c + 2], ov[4 * c + 3]);
          const float lse2 = any ? m + __log2f(l) : -INFINITY;
          p.part_lse[it * BM + a] = lse2;
          __threadfence();  // this chunk's rows are visible before it is counted
          __syncwarp();
          const int unit = u / kSplit;
          int done = 0;
          if (lane == 0) done = atomicAdd(&p.part_cnt[unit * 4 + quad], 1);
          done = __shfl_sync(0xffffffffu, done, 0);
          if (done == kSplit - 1) {
            __threadfence();
            // weights 2^(lse_c - max) of the chunks (lse -inf: no visible key),
            // summed in chunk order whichever chunk merges (the result does
            // not depend on which finished last).  Every chunk's rows, this
            // one's included, are read back from the scratch, so that its
            // result registers are dead here.
            const size_t it0 = static_cast<size_t>(unit) * kSplit;
            float mx = -INFINITY;
            for (int c = 0; c < kSplit; ++c) mx = fmaxf(mx, p.part_lse[(it0 + c) * BM + a]);
            float wsum = 0.f;
            float acc[D];
#pragma unroll
            for (int n = 0; n < D; ++n) acc[n] = 0.f;
            for (int c = 0; c < kSplit; ++c) {
              const float l2 = p.part_lse[(it0 + c) * BM + a];
              if (l2 == -INFINITY) continue;
              const float wt = ex2(l2 - mx);
              wsum += wt;
              const float4* src = reinterpret_cast<const float4*>(p.part_o + ((it0 + c) * BM + a) * D);
#pragma unroll
              for (int q4 = 0; q4 < D / 4; ++q4) {
                const float4 x = src[q4];
                acc[4 * q4] = fmaf(wt, x.x, acc[4 * q4]);
                acc[4 * q4 + 1] = fmaf(wt, x.y, acc[4 * q4 + 1]);
                acc[4 * q4 + 2] = fmaf(wt, x.z, acc[4 * q4 + 2]);
                acc[4 * q4 + 3] = fmaf(wt, x.w, acc[4 * q4 + 3]);
              }
            }
            if (i < p.W) {
              const float inv = 1.f / wsum;
              const size_t orow = ((static_cast<size_t>(w.b) * p.W + i) * p.H + w.h) * D;
              if (O_BF16) {
                uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.o) + orow);
#pragma unroll
                for (int c = 0; c < D / 8; ++c)
                  dst[c] = make_uint4(pack_bf16x2(acc[8 * c] * inv, acc[8 * c + 1] * inv),
                                      pack_bf16x2(acc[8 * c + 2] * inv, acc[8 * c + 3] * inv),
                                      pack_bf16x2(acc[8 * c + 4] * inv, acc[8 * c + 5] * inv),
                                      pack_bf16x2(acc[8 * c + 6] * inv, acc[8 * c + 7] * inv));
              } else {
                float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.o) + orow);
#pragma unroll
                for (int c = 0; c < D / 4; ++c)
                  dst[c] = make_float4(acc[4 * c] * inv, acc[4 * c + 1] * inv, acc[4 * c + 2] * inv,
                                       acc[4 * c + 3] * inv);
              }
              if (p.lse != nullptr)
                p.lse[(static_cast<size_t>(w.b) * p.H + w.h) * p.W + i] =
                    (mx + __log2f(wsum)) * 0.69314718055994531f;
            }
            if (lane == 0) p.part_cnt[unit * 4 + quad] = 0;  // ready for the next launch
          }
        } else if (O_BF16) {
          // bf16 rows into this warp's quadrant of its own P buffer (free
          // until its next step: the last PV that read it is complete), then
          // one TMA store of the 32-row box; rows past W are not written.
          uint8_t* orow_s = sP + par * kQTile + (a / 8) * 1024 + (a % 8) * 128;
#pragma unroll
          for (int c = 0; c < D / 8; ++c)
            *reinterpret_cast<uint4*>(orow_s + ((c ^ (a % 8)) * 16)) =
                make_uint4(pack_bf16x2(ov[8 * c], ov[8 * c + 1]), pack_bf16x2(ov[8 * c + 2], ov[8 * c + 3]),
                           pack_bf16x2(ov[8 * c + 4], ov[8 * c + 5]), pack_bf16x2(ov[8 * c + 6], ov[8 * c + 7]));
          fence_proxy_async_smem();
          __syncwarp();
          if (w.i0 + 32 * quad < p.W) {
            if (lane == 0) {
              tma_store_4d(&tm_o, sP + par * kQTile + quad * 4096, 0, w.h, w.i0 + 32 * quad, w.b);
              bulk_commit_group();
            }
            store_pending = true;
          }
        } else if (i < p.W) {
          const size_t orow = ((static_cast<size_t>(w.b) * p.W + i) * p.H + w.h) * D;
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.o) + orow);
#pragma unroll
          for (int c = 0; c < D / 4; ++c) dst[c] = make_float4(ov[4 * c], ov[4 * c + 1], ov[4 * c + 2], ov[4 * c + 3]);
        }
        if (!SPLIT && i < p.W && p.lse != nullptr)
          p.lse[(static_cast<size_t>(w.b) * p.H + w.h) * p.W + i] = (m + __log2f(l)) * 0.69314718055994531f;
      }
      gt = g0 + w.nks;
      ++un;
      rb = (rb + w.nks + 2) & (kSlots - 1);
    }
    if (!ok) report_timeout(abort, p.status);
    // Output stores in flight must finish before the CTA's shared memory goes.
    if (lane == 0) bulk_wait_group0();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
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

template <bool O_BF16, bool SPLIT, bool RING>
cudaError_t launch_typed(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                         const CUtensorMap& tm_r, const CUtensorMap& tm_o, const CUtensorMap& tm_km,
                         const CUtensorMap& tm_vm, const CUtensorMap& tm_ks, const CUtensorMap& tm_vs,
                         const Params& prm, cudaStream_t stream) {
  auto kern = relattn_tc64_kernel<O_BF16, SPLIT, RING>;
  static int configured_mask = 0;  // one bit per device ordinal < 32
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 32 || !(__atomic_load_n(&configured_mask, __ATOMIC_ACQUIRE) & (1 << dev))) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev < 32) __atomic_fetch_or(&configured_mask, 1 << dev, __ATOMIC_RELEASE);
  }
  const int grid = prm.n_units < num_sms() ? prm.n_units : num_sms();
  return launch_dependent(kern, dim3(grid), dim3(kThreads), kSmemBytes, stream, tm_q, tm_k, tm_v, tm_r, tm_o, tm_km,
                          tm_vm, tm_ks, tm_vs, prm);
}

// Units dealt to the CTAs by cost (longest-processing-time first onto the
// least-loaded CTA, then moves and swaps off the busiest CTA while they lower
// it); each CTA's units run longest first.  A unit costs its key steps plus
// kUnitCost for the unit boundary (first-score latency and epilogue, about
// 1.2 steps in traces of the kernel).  Returns the table [P][stride] (-1
// ends a row).  The unit order and step counts are those of decode_unit.
std::vector<int> plan_units(int B, int H, int W, int M, int P, int* stride_out) {
  constexpr double kUnitCost = 1.2;
  const int nqt = (W + BM - 1) / BM, n = nqt * B * H;
  std::vector<double> cost(n);
  for (int u = 0; u < n; ++u) {
    const int qt = nqt - 1 - u / (B * H);
    const int kmax = std::min(M + qt * BM + BM - 1, M + W - 1);
    cost[u] = kmax / BN + 1 + kUnitCost;
  }
  std::vector<std::vector<int>> bins(P);
  std::vector<double> load(P, 0.0);
  using Slot = std::pair<double, int>;
  std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> heap;
  for (int c = 0; c < P; ++c) heap.push({0.0, c});
  for (int u = 0; u < n; ++u) {  // units are already in decreasing cost
    const int c = heap.top().second;
    heap.pop();
    bins[c].push_back(u);
    load[c] += cost[u];
    heap.push({load[c], c});
  }
  for (int iter = 0; iter < 4 * n; ++iter) {
    const int A = static_cast<int>(std::max_element(load.begin(), load.end()) - load.begin());
    const double mx = load[A];
    double best_gain = 1e-9;
    int bx = -1, by = -1, bB = -1;  // move bins[A][bx] to B, swapping in bins[B][by] when by >= 0
    for (int B2 = 0; B2 < P; ++B2) {
      if (B2 == A) continue;
      for (int xi = 0; xi < static_cast<int>(bins[A].size()); ++xi) {
        const double cx = cost[bins[A][xi]];
        const double gm = mx - std::max(load[A] - cx, load[B2] + cx);
        if (gm > best_gain) best_gain = gm, bx = xi, by = -1, bB = B2;
        for (int yi = 0; yi < static_cast<int>(bins[B2].size()); ++yi) {
          const double cy = cost[bins[B2][yi]];
          if (cy >= cx) continue;
          const double gs = mx - std::max(load[A] - cx + cy, load[B2] - cy + cx);
          if (gs > best_gain) best_gain = gs, bx = xi, by = yi, bB = B2;
        }
      }
    }
    if (bx < 0) break;
    const int x = bins[A][bx];
    bins[A].erase(bins[A].begin() + bx);
    load[A] -= cost[x];
    if (by >= 0) {
      const int y = bins[bB][by];
      bins[bB].erase(bins[bB].begin() + by);
      load[bB] -= cost[y];
      bins[A].push_back(y);
      load[A] += cost[y];
    }
    bins[bB].push_back(x);
    load[bB] += cost[x];
  }
  size_t kmax = 0;
  for (auto& b : bins) {
    std::sort(b.begin(), b.end());  // unit index order is longest first
    kmax = std::max(kmax, b.size());
  }
  const int stride = static_cast<int>(kmax) + 1;
  std::vector<int> table(static_cast<size_t>(P) * stride, -1);
  for (int c = 0; c < P; ++c)
    for (size_t r = 0; r < bins[c].size(); ++r) table[static_cast<size_t>(c) * stride + r] = bins[c][r];
  *stride_out = stride;
  return table;
}

// Device copies of the plans, per (device, B, H, W, M, grid); made on first
// use of a shape and kept until txl_release_cached.  The table is filled in
// pinned host memory (kept with the entry, so the copy can read it at any
// time) and uploaded with an asynchronous copy on the caller's stream; an
// event recorded behind the copy orders it before launches on other streams.
// At most kMaxPlans shapes are cached: later shapes run the snake order.
struct PlanEntry {
  int* dev_table = nullptr;
  int* host_table = nullptr;
  int stride = 0;
  cudaEvent_t uploaded = nullptr;
  bool done = false;  // the upload was seen complete
};
constexpr size_t kMaxPlans = 256;
std::mutex g_plan_mutex;
std::map<std::tuple<int, int, int, int, int, int>, PlanEntry> g_plans;

void free_plan(PlanEntry& p) {
  if (p.uploaded != nullptr) cudaEventDestroy(p.uploaded);
  if (p.dev_table != nullptr) cudaFree(p.dev_table);
  if (p.host_table != nullptr) cudaFreeHost(p.host_table);
  p = PlanEntry();
}

}  // namespace

cudaError_t unit_plan(int B, int H, int W, int M, int P, cudaStream_t stream, const int** table, int* stride) {
  *table = nullptr;
  *stride = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if ((e = cudaStreamIsCapturing(stream, &cap)) != cudaSuccess) return e;
  const bool capturing = cap != cudaStreamCaptureStatusNone;
  std::lock_guard<std::mutex> lk(g_plan_mutex);
  const auto key = std::make_tuple(dev, B, H, W, M, P);
  auto it = g_plans.find(key);
  if (it == g_plans.end()) {
    // No plan yet: making one allocates and copies, which a stream being
    // captured into a graph must not see; such a call keeps the snake order,
    // and so does every shape past the cache's bound.
    if (capturing || g_plans.size() >= kMaxPlans) return cudaSuccess;
    int st = 0;
    const std::vector<int> t = plan_units(B, H, W, M, P, &st);
    const size_t bytes = t.size() * sizeof(int);
    PlanEntry pe;
    pe.stride = st;
    if ((e = cudaMallocHost(&pe.host_table, bytes)) != cudaSuccess ||
        (e = cudaMalloc(&pe.dev_table, bytes)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&pe.uploaded, cudaEventDisableTiming)) != cudaSuccess) {
      free_plan(pe);
      return e;
    }
    std::memcpy(pe.host_table, t.data(), bytes);
    if ((e = cudaMemcpyAsync(pe.dev_table, pe.host_table, bytes, cudaMemcpyHostToDevice, stream)) != cudaSuccess ||
        (e = cudaEventRecord(pe.uploaded, stream)) != cudaSuccess) {
      // nothing was queued that could still read the buffers
      cudaStreamSynchronize(stream);
      free_plan(pe);
      return e;
    }
    g_plans.emplace(key, pe);
    *table = pe.dev_table;
    *stride = pe.stride;
    return cudaSuccess;  // this stream's launch follows the copy in stream order
  }
  PlanEntry& pe = it->second;
  if (!pe.done) {
    // The upload may still be queued on the stream that made the plan.  A
    // stream being captured may not query or wait on it: snake order.
    if (capturing) return cudaSuccess;
    e = cudaEventQuery(pe.uploaded);
    if (e == cudaSuccess) {
      pe.done = true;
    } else if (e == cudaErrorNotReady) {
      if ((e = cudaStreamWaitEvent(stream, pe.uploaded, 0)) != cudaSuccess) return e;
    } else {
      return e;
    }
  }
  *table = pe.dev_table;
  *stride = pe.stride;
  return cudaSuccess;
}

cudaError_t release_plans(int dev) {
  std::lock_guard<std::mutex> lk(g_plan_mutex);
  for (auto it = g_plans.begin(); it != g_plans.end();) {
    if (std::get<0>(it->first) == dev) {
      free_plan(it->second);
      it = g_plans.erase(it);
    } else {
      ++it;
    }
  }
  return cudaGetLastError();
}

int relattn_tc64_items(int B, int H, int W, int M, int nsplit, int* items, int cap, int* n_items) {
  if (B < 0 || H < 0 || W <= 0 || M < 0 || n_items == nullptr || nsplit < 1 || nsplit > 64) return -1;
  const int nqt = (W + BM - 1) / BM;
  if (nsplit > std::min(M + BM - 1, M + W - 1) / BN + 1) return -1;  // a chunk of every unit holds a step
  const long long n = static_cast<long long>(nqt) * B * H * nsplit;
  if (n > (1 << 20)) return -1;
  *n_items = static_cast<int>(n);
  if (items == nullptr) return 0;
  if (cap < *n_items) return -2;
  for (int it = 0; it < *n_items; ++it) {
    const Unit u = decode_item(it, nsplit, B, H, W, M, nqt);
    const int row[5] = {u.b, u.h, u.i0, u.t0, u.nks};
    std::copy(row, row + 5, items + 5 * static_cast<size_t>(it));
  }
  return 0;
}

int relattn_tc64_plan_table(int B, int H, int W, int M, int P, int* table, int cap, int* stride) {
  if (B < 0 || H < 0 || W < 0 || M < 0 || P <= 0 || stride == nullptr) return -1;
  if (static_cast<long long>((W + BM - 1) / BM) * B * H > (1 << 16) || P > (1 << 16)) return -1;
  int st = 0;
  const std::vector<int> t = plan_units(B, H, W, M, P, &st);
  *stride = st;
  if (table == nullptr) return 0;
  if (cap < 0 || static_cast<size_t>(cap) < t.size()) return -2;
  std::copy(t.begin(), t.end(), table);
  return 0;
}

int relattn_tc64_split(int B, int H, int W, int M) { return relattn_tc64_split_for(B, H, W, M, num_sms()); }

int relattn_tc64_split_for(int B, int H, int W, int M, int sms) {
  // Cost in key steps of the slowest CTA: waves of work items times the
  // steps of the longest item, plus a unit boundary per item and, when
  // split, about the cost of the merge launch.
  constexpr double kBoundary = 1.5, kMerge = 4.0;
  const long long nqt = (W + BM - 1) / BM;
  const long long units = nqt * B * H;
  if (units >= sms) return 1;
  const int nks_max = (M + W - 1) / BN + 1;
  const int nks_min = (min(M + BM - 1, M + W - 1)) / BN + 1;
  int best = 1;
  double best_cost = static_cast<double>((units + sms - 1) / sms) * (nks_max + kBoundary);
  for (int s = 2; s <= nks_min && s <= 16; ++s) {
    const double waves = static_cast<double>((units * s + sms - 1) / sms);
    const double cost = waves * ((nks_max + s - 1) / s + kBoundary) + kMerge;
    if (cost < best_cost) {
      best_cost = cost;
      best = s;
    }
  }
  return best;
}

cudaError_t launch_relattn_tc64(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                const CUtensorMap& tm_r, const CUtensorMap* tm_o, const CUtensorMap* tm_km,
                                const CUtensorMap* tm_vm, int roll_src0, const RingMaps* ring,
                                const float* bias_u, const float* bias_v, void* o,
                                float* lse, int B, int W, int M, int H, bool o_bf16, float scale, int nsplit,
                                float* part_o, float* part_lse, int* part_cnt, bool allow_plan,
                                const WaitCtl& wc, cudaStream_t stream) {
  Params prm;
  prm.bias_u = bias_u;
  prm.bias_v = bias_v;
  prm.o = o;
  prm.lse = lse;
  prm.B = B;
  prm.W = W;
  prm.M = M;
  prm.H = H;
  prm.nqt = (W + BM - 1) / BM;
  prm.nsplit = nsplit;
  prm.part_o = part_o;
  prm.part_lse = part_lse;
  prm.part_cnt = part_cnt;
  prm.n_units = prm.nqt * B * H * nsplit;
  if (nsplit < 1 || (nsplit > 1 && (part_o == nullptr || part_lse == nullptr || part_cnt == nullptr)))
    return cudaErrorInvalidValue;
  prm.qsign = scale < 0.f ? -1.f : 1.f;
  prm.scale_log2e = fmaxf(fabsf(scale), 1e-30f) * 1.4426950408889634f;
  prm.status = wc.status;
  prm.wait_ns = wc.limit_ns;
  prm.inject_stall = wc.inject_stall;
  prm.roll_src0 = (tm_km != nullptr && tm_vm != nullptr) ? roll_src0 : -1;
  if (prm.roll_src0 >= 0 && prm.roll_src0 % BN != 0) return cudaErrorInvalidValue;
  prm.ring_cap = ring != nullptr ? ring->cap : 0;
  prm.ring_start = ring != nullptr ? ring->start : 0;
  prm.ring_append = ring != nullptr && ring->append ? 1 : 0;
  if (ring != nullptr && (prm.roll_src0 >= 0 || ring->cap % BN != 0 || ring->start % BN != 0 || M % BN != 0 ||
                          M > ring->cap || ring->start < 0 || ring->start >= ring->cap))
    return cudaErrorInvalidValue;
  // the appended rows must land in slots outside the memory, whole tiles only
  if (prm.ring_append && (W % BN != 0 || M + W > ring->cap)) return cudaErrorInvalidValue;
  if (o_bf16 && tm_o == nullptr) return cudaErrorInvalidValue;
  // More units than CTAs: deal them by the host's plan (made once per shape)
  prm.sched = nullptr;
  prm.sched_stride = 0;
  if (allow_plan && nsplit == 1 && prm.n_units > num_sms()) {
    const cudaError_t pe = unit_plan(B, H, W, M, num_sms(), stream, &prm.sched, &prm.sched_stride);
    if (pe != cudaSuccess) return pe;
  }
  // Unused maps (fp32 output is written with plain stores; no roll) are
  // stood in for by tm_q and never touched.
  const CUtensorMap& km = prm.roll_src0 >= 0 ? *tm_km : tm_q;
  const CUtensorMap& vm = prm.roll_src0 >= 0 ? *tm_vm : tm_q;
  const CUtensorMap& ks = ring != nullptr ? ring->tm_ks : tm_q;
  const CUtensorMap& vs = ring != nullptr ? ring->tm_vs : tm_q;
  // The ring form is its own instantiation: the loader of the ordinary one
  // stays as small as it was.
  if (ring != nullptr) {
    if (nsplit > 1)
      return o_bf16 ? launch_typed<true, true, true>(tm_q, tm_k, tm_v, tm_r, *tm_o, km, vm, ks, vs, prm, stream)
                    : launch_typed<false, true, true>(tm_q, tm_k, tm_v, tm_r, tm_q, km, vm, ks, vs, prm, stream);
    return o_bf16 ? launch_typed<true, false, true>(tm_q, tm_k, tm_v, tm_r, *tm_o, km, vm, ks, vs, prm, stream)
                  : launch_typed<false, false, true>(tm_q, tm_k, tm_v, tm_r, tm_q, km, vm, ks, vs, prm, stream);
  }
  if (nsplit > 1)
    return o_bf16 ? launch_typed<true, true, false>(tm_q, tm_k, tm_v, tm_r, *tm_o, km, vm, ks, vs, prm, stream)
                  : launch_typed<false, true, false>(tm_q, tm_k, tm_v, tm_r, tm_q, km, vm, ks, vs, prm, stream);
  return o_bf16 ? launch_typed<true, false, false>(tm_q, tm_k, tm_v, tm_r, *tm_o, km, vm, ks, vs, prm, stream)
                : launch_typed<false, false, false>(tm_q, tm_k, tm_v, tm_r, tm_q, km, vm, ks, vs, prm, stream);
}

}  // namespace txl
