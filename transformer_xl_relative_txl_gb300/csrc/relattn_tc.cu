// bf16 relative-position attention on the sm_103a tensor cores (tcgen05 + TMEM
// + TMA), fp32 accumulation.
//
//   s[i,j] = scale * ((q_i + u) . k_j + (q_i + v) . r_{M+i-j}),   j <= M+i
//   o_i = softmax(s[i,.]) V
//
// "Transformer-XL, explained", method steps 3-5: keys / values over
// [memory ; segment], queries from the segment, the four-term relative score
// (grouped here by its query-side factor), and the distance term computed once
// against every distance and shifted into place per row.  The shift is an
// index, not a pad-and-reshape: row a of a 128-query tile against key tile t
// needs distances base_t + a - c (c = key column, base_t = M + i0 - 128 t),
// which all lie in two 128-distance tiles [base_t - 128, base_t) and
// [base_t, base_t + 128).  Consecutive key tiles share one of them, so each
// step issues one new 128x128 distance MMA into a two-slot TMEM ring and the
// distance work equals the content work (step 5: "the cost stays that of
// ordinary attention").
//
// CTA = one (batch, head, 128-query tile); 6 warps:
//   warps 0-3  softmax: thread a owns query row a (TMEM lane a).  Builds the
//              bf16 (q+u) and (q+v) tiles in shared memory, then per key tile
//              reads S and its 159-distance window of the ring, shifts the
//              window per lane (5-stage select network, the lane-dependent
//              part of the index), adds, masks j > M+i, runs the online
//              softmax, rescales O when the row max grows, writes P (bf16)
//              over the S columns, and finally normalises O and stores o, lse.
//   warp 4     loader: TMA tile loads of K, V (4-D maps, zero fill past M+W)
//              and R (3-D map, zero fill outside [0, n_r)) into 128B-swizzled
//              stage rings.
//   warp 5     MMA issuer (one thread): S = (q+u) K^T, G_t = (q+v) R_t^T into
//              the ring, O += P V with P read from TMEM; tcgen05.commit
//              signals the barriers.  Also owns the TMEM allocation.
//
// TMEM (512 columns): S / P [0,128) | ring slot 0 [128,256) | slot 1
// [256,384) | O [384, 384+D).
//
// Every wait is bounded (globaltimer); a wait that runs out raises a CTA
// abort flag and the device status word, and every role unwinds: the loader
// waits for its own copies in flight, the MMA thread for its own MMAs, and
// the TMEM is freed before exit.
#include <cmath>
#include <cstdint>

#include "txl_device.cuh"
#include "txl_internal.h"

namespace txl {
namespace {

constexpr int BM = 128;         // query rows per CTA
constexpr int BN = 128;         // keys per step
constexpr int kThreads = 192;
constexpr int kLoaderWarp = 4;
constexpr int kMmaWarp = 5;
constexpr uint32_t kColS = 0;
constexpr uint32_t kColG0 = 128;
constexpr uint32_t kColG1 = 256;
constexpr uint32_t kColO = 384;
constexpr uint32_t kTmemCols = 512;
constexpr int kChunkBytes = BM * 64 * 2;  // one 128-row x 64-element bf16 block (16 KB)

template <int D>
struct Cfg {
  static constexpr int kChunks = D / 64;
  static constexpr int kTileBytes = BM * D * 2;
  static constexpr int NK = (D == 64) ? 2 : 1;
  static constexpr int NV = (D == 64) ? 2 : 1;
  static constexpr int NR = 2;
  static constexpr int kOffQu = 0;
  static constexpr int kOffQv = kOffQu + kTileBytes;
  static constexpr int kOffK = kOffQv + kTileBytes;
  static constexpr int kOffV = kOffK + NK * kTileBytes;
  static constexpr int kOffR = kOffV + NV * kTileBytes;
  static constexpr int kOffBar = kOffR + NR * kTileBytes;
  static constexpr int kBarBytes = 256;
  static constexpr int kSmemBytes = kOffBar + kBarBytes + 1024;  // + alignment slack
};

struct Params {
  const __nv_bfloat16* q;
  const float* bias_u;
  const float* bias_v;
  void* o;
  float* lse;
  int B, W, M, H;
  float scale_log2e;
  unsigned int* status;
  unsigned long long wait_ns;
  int inject_stall;
};

// Barrier block layout (8-byte slots) after the tiles.
struct Bars {
  uint64_t fullK[2], emptyK[2], fullV[2], emptyV[2], fullR[2], emptyR[2];
  uint64_t q_ready, s_full, p_full, o_done, mma_final;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Bars) <= 256, "barrier block too large");

// Five-stage select network: on return arr[m] == in[m + sh] for m in [1, 32],
// where in[] is the original arr[0..63] and 0 <= sh < 32 differs per lane.
__device__ __forceinline__ void lane_shift(float (&arr)[64], int sh) {
  const bool b16 = sh & 16, b8 = sh & 8, b4 = sh & 4, b2 = sh & 2, b1 = sh & 1;
#pragma unroll
  for (int m = 1; m <= 47; ++m) arr[m] = b16 ? arr[m + 16] : arr[m];
#pragma unroll
  for (int m = 1; m <= 39; ++m) arr[m] = b8 ? arr[m + 8] : arr[m];
#pragma unroll
  for (int m = 1; m <= 35; ++m) arr[m] = b4 ? arr[m + 4] : arr[m];
#pragma unroll
  for (int m = 1; m <= 33; ++m) arr[m] = b2 ? arr[m + 2] : arr[m];
#pragma unroll
  for (int m = 1; m <= 32; ++m) arr[m] = b1 ? arr[m + 1] : arr[m];
}

template <int D, bool O_BF16>
__global__ void __launch_bounds__(kThreads, 1)
    relattn_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_r, const Params p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  uint8_t* sQu = smem + C::kOffQu;
  uint8_t* sQv = smem + C::kOffQv;
  uint8_t* sK = smem + C::kOffK;
  uint8_t* sV = smem + C::kOffV;
  uint8_t* sR = smem + C::kOffR;
  Bars* bars = reinterpret_cast<Bars*>(smem + C::kOffBar);
  volatile int* abort = &bars->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- work unit: longest query tiles first --------------------------------
  const int nqt = (p.W + BM - 1) / BM;
  const int BH = p.B * p.H;
  const int qt = nqt - 1 - static_cast<int>(blockIdx.x / BH);
  const int bh = static_cast<int>(blockIdx.x % BH);
  const int b = bh / p.H;
  const int h = bh % p.H;
  const int i0 = qt * BM;
  const int L = p.M + p.W;
  const int kmax = min(p.M + i0 + BM - 1, L - 1);
  const int nkt = kmax / BN + 1;

  // ---- setup ---------------------------------------------------------------
  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->fullK[s], 1);
      mbar_init(&bars->emptyK[s], 1);
      mbar_init(&bars->fullV[s], 1);
      mbar_init(&bars->emptyV[s], 1);
      mbar_init(&bars->fullR[s], 1);
      mbar_init(&bars->emptyR[s], 1);
    }
    mbar_init(&bars->q_ready, 128);
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->p_full, 128);
    mbar_init(&bars->o_done, 1);
    mbar_init(&bars->mma_final, 1);
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
    // ======================= TMA loader ====================================
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_r);
      int nK = 0, nV = 0, nR = 0;
      bool ok = true;
      auto load_r = [&](int d0) -> bool {
        const int s = nR % C::NR;
        if (!mbar_wait(&bars->emptyR[s], ((nR / C::NR) & 1) ^ 1, wait_ns, abort)) return false;
        mbar_arrive_expect_tx(&bars->fullR[s], C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_3d(sR + s * C::kTileBytes + c * kChunkBytes, &tm_r, &bars->fullR[s], c * 64, h, d0);
        ++nR;
        return true;
      };
      auto load_k = [&](int t) -> bool {
        const int s = nK % C::NK;
        if (!mbar_wait(&bars->emptyK[s], ((nK / C::NK) & 1) ^ 1, wait_ns, abort)) return false;
        mbar_arrive_expect_tx(&bars->fullK[s], C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_4d(sK + s * C::kTileBytes + c * kChunkBytes, &tm_k, &bars->fullK[s], c * 64, h, t * BN, b);
        ++nK;
        return true;
      };
      auto load_v = [&](int t) -> bool {
        const int s = nV % C::NV;
        if (!mbar_wait(&bars->emptyV[s], ((nV / C::NV) & 1) ^ 1, wait_ns, abort)) return false;
        mbar_arrive_expect_tx(&bars->fullV[s], C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_4d(sV + s * C::kTileBytes + c * kChunkBytes, &tm_v, &bars->fullV[s], c * 64, h, t * BN, b);
        ++nV;
        return true;
      };
      ok = load_r(p.M + i0);  // hi tile of the first step
      for (int t = 0; ok && t < nkt; ++t) {
        if (p.inject_stall && t == 1) break;  // test hook: starve the consumers
        ok = load_k(t) && load_r(p.M + i0 - BN * (t + 1)) && load_v(t);
      }
      if (!ok) report_timeout(abort, p.status);
      // Wait for this thread's own copies in flight before the CTA may exit.
      auto drain = [&](uint64_t* full, int n, int ns) {
        for (int s = 0; s < ns && s < n; ++s) {
          const int last = s + ((n - 1 - s) / ns) * ns;
          mbar_wait_own(&full[s], (last / ns) & 1, wait_ns);
        }
      };
      drain(bars->fullK, nK, C::NK);
      drain(bars->fullV, nV, C::NV);
      drain(bars->fullR, nR, C::NR);
    }
  } else if (warp == kMmaWarp) {
    // ======================= MMA issuer ====================================
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16(128, 128, false, false);
      constexpr uint32_t idesc_o = idesc_bf16(128, D, false, true);
      const uint32_t aQu = smem_u32(sQu), aQv = smem_u32(sQv);
      const uint32_t aK = smem_u32(sK), aV = smem_u32(sV), aR = smem_u32(sR);
      bool ok = mbar_wait(&bars->q_ready, 0, wait_ns, abort);
      tc_fence_after();
      int nR = 0;
      for (int t = 0; ok && t < nkt; ++t) {
        const int sk = t % C::NK;
        ok = mbar_wait(&bars->fullK[sk], (t / C::NK) & 1, wait_ns, abort);
        if (ok && t > 0) ok = mbar_wait(&bars->o_done, (t - 1) & 1, wait_ns, abort);  // P_{t-1} consumed
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk / 4) * kChunkBytes + (kk % 4) * 32;
          mma_ss(tmem + kColS, sdesc_sw128(aQu + koff, 16, 1024),
                 sdesc_sw128(aK + sk * C::kTileBytes + koff, 16, 1024), idesc_s, kk > 0);
        }
        tc_commit(&bars->emptyK[sk]);
        const int ntiles = (t == 0) ? 2 : 1;
        for (int z = 0; z < ntiles; ++z) {
          const uint32_t slot = (t == 0 && z == 0) ? 1u : static_cast<uint32_t>(t & 1);
          const int sr = nR % C::NR;
          ok = mbar_wait(&bars->fullR[sr], (nR / C::NR) & 1, wait_ns, abort);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t koff = (kk / 4) * kChunkBytes + (kk % 4) * 32;
            mma_ss(tmem + (slot ? kColG1 : kColG0), sdesc_sw128(aQv + koff, 16, 1024),
                   sdesc_sw128(aR + sr * C::kTileBytes + koff, 16, 1024), idesc_s, kk > 0);
          }
          tc_commit(&bars->emptyR[sr]);
          ++nR;
        }
        if (!ok) break;
        tc_commit(&bars->s_full);
        const int sv = t % C::NV;
        ok = mbar_wait(&bars->p_full, t & 1, wait_ns, abort);
        if (ok) ok = mbar_wait(&bars->fullV[sv], (t / C::NV) & 1, wait_ns, abort);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          // V tile: keys are the K dimension (rows of 128 B), D the N dimension
          // (MN-major); the second 64-column block, if any, sits 16 KB further.
          mma_ts(tmem + kColO, tmem + kColS + kk * 8,
                 sdesc_sw128(aV + sv * C::kTileBytes + kk * 16 * 128, kChunkBytes, 1024), idesc_o,
                 (t > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(&bars->emptyV[sv]);
        tc_commit(&bars->o_done);
      }
      if (!ok) report_timeout(abort, p.status);
      tc_commit(&bars->mma_final);
      mbar_wait_own(&bars->mma_final, 0, wait_ns);
    }
  } else {
    // ======================= softmax warps =================================
    const int a = threadIdx.x;  // row within the tile == TMEM lane
    const int i = i0 + a;
    const bool row_valid = i < p.W;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;

    // (q + u), (q + v) rows -> bf16, 128B-swizzled K-major tiles.
    {
      const __nv_bfloat16* qrow = p.q + ((static_cast<size_t>(b) * p.W + (row_valid ? i : 0)) * p.H + h) * D;
      const float* bu = p.bias_u + h * D;
      const float* bv = p.bias_v + h * D;
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        uint4 raw = make_uint4(0, 0, 0, 0);
        if (row_valid) raw = *reinterpret_cast<const uint4*>(qrow + c * 8);
        const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
        uint32_t pu[4], pv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float x0 = bf16_lo(w4[e]), x1 = bf16_hi(w4[e]);
          const int d = c * 8 + 2 * e;
          pu[e] = pack_bf16x2(x0 + bu[d], x1 + bu[d + 1]);
          pv[e] = pack_bf16x2(x0 + bv[d], x1 + bv[d + 1]);
        }
        const int kc = c / 8, cc = c % 8;
        const int off = kc * kChunkBytes + (a / 8) * 1024 + (a % 8) * 128 + ((cc ^ (a % 8)) * 16);
        *reinterpret_cast<uint4*>(sQu + off) = make_uint4(pu[0], pu[1], pu[2], pu[3]);
        *reinterpret_cast<uint4*>(sQv + off) = make_uint4(pv[0], pv[1], pv[2], pv[3]);
      }
      fence_proxy_async_smem();
      mbar_arrive(&bars->q_ready);
    }

    float m_run = -INFINITY;  // running row max (log2 units)
    float l_run = 0.f;        // running row sum
    bool ok = true;
    const float sl2 = p.scale_log2e;
    for (int t = 0; t < nkt; ++t) {
      bool got = mbar_wait(&bars->s_full, t & 1, wait_ns, abort);
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int base = p.M + i0 - BN * t;  // distance of (row 0, key column 0)
      const uint32_t col_lo = (t & 1) ? kColG1 : kColG0;  // distances [base-128, base)
      const uint32_t col_hi = (t & 1) ? kColG0 : kColG1;  // distances [base, base+128)
      const int lim = base + a;  // key column c is visible iff c <= lim
      float s2[BN];
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t sraw[32], x0[32], x1[32];
        tmem_ld32(tmem + lane_base + kColS + ch * 32, sraw);
        // Window of the [lo | hi] distance row that this warp's lanes need:
        // columns zq .. zq+63 with zq = 96 + 32*warp - 32*ch (warp-uniform).
        const int zq = 32 * (3 + warp - ch);
        const uint32_t z0 = (zq < 128) ? col_lo + zq : col_hi + (zq - 128);
        const uint32_t z1 = (zq + 32 < 128) ? col_lo + zq + 32 : col_hi + (zq + 32 - 128);
        tmem_ld32(tmem + lane_base + z0, x0);
        tmem_ld32(tmem + lane_base + z1, x1);
        tmem_wait_ld(sraw);
        tmem_wait_ld(x0);
        tmem_wait_ld(x1);
        float arr[64];
#pragma unroll
        for (int n = 0; n < 32; ++n) {
          arr[n] = __uint_as_float(x0[n]);
          arr[n + 32] = __uint_as_float(x1[n]);
        }
        lane_shift(arr, lane);  // arr[m] = window[m + lane]
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const int c = ch * 32 + k;
          // distance base + a - c sits at window index lane + 32 - k
          const float sv = (__uint_as_float(sraw[k]) + arr[32 - k]) * sl2;
          s2[c] = (c <= lim) ? sv : -INFINITY;
        }
      }
      float mx8[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) mx8[u] = s2[u];
#pragma unroll
      for (int c = 8; c < BN; ++c) mx8[c & 7] = fmaxf(mx8[c & 7], s2[c]);
      const float mt = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                             fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
      const float m_new = fmaxf(m_run, mt);
      const float alpha = ex2(m_run - m_new);
      float sum8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      uint32_t pk0[32], pk1[32];
#pragma unroll
      for (int n = 0; n < BN / 2; ++n) {
        const float e0 = ex2(s2[2 * n] - m_new);
        const float e1 = ex2(s2[2 * n + 1] - m_new);
        sum8[n & 7] += e0 + e1;
        if (n < 32)
          pk0[n] = pack_bf16x2(e0, e1);
        else
          pk1[n - 32] = pack_bf16x2(e0, e1);
      }
      const float sum = ((sum8[0] + sum8[1]) + (sum8[2] + sum8[3])) + ((sum8[4] + sum8[5]) + (sum8[6] + sum8[7]));
      l_run = l_run * alpha + sum;
      const bool need = (t > 0) && (m_new > m_run);
      m_run = m_new;
      if (__any_sync(0xffffffffu, need)) {
        // PV_{t-1} completed before s_full(t) fired: O is stable here.
#pragma unroll
        for (int oc = 0; oc < D / 32; ++oc) {
          uint32_t ov[32];
          tmem_ld32(tmem + lane_base + kColO + oc * 32, ov);
          tmem_wait_ld(ov);
#pragma unroll
          for (int n = 0; n < 32; ++n) ov[n] = __float_as_uint(__uint_as_float(ov[n]) * alpha);
          tmem_st32(tmem + lane_base + kColO + oc * 32, ov);
        }
      }
      tmem_st32(tmem + lane_base + kColS, pk0);
      tmem_st32(tmem + lane_base + kColS + 32, pk1);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->p_full);
    }

    if (ok) {
      bool got = mbar_wait(&bars->o_done, (nkt - 1) & 1, wait_ns, abort);
      ok = __all_sync(0xffffffffu, got);
    }
    if (ok) {
      tc_fence_after();
      const float inv_l = 1.f / l_run;
      uint32_t ov[D];
#pragma unroll
      for (int oc = 0; oc < D / 32; ++oc) {
        uint32_t tmp[32];
        tmem_ld32(tmem + lane_base + kColO + oc * 32, tmp);
        tmem_wait_ld(tmp);
#pragma unroll
        for (int n = 0; n < 32; ++n) ov[oc * 32 + n] = tmp[n];
      }
      if (row_valid) {
        const size_t orow = ((static_cast<size_t>(b) * p.W + i) * p.H + h) * D;
        if (O_BF16) {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.o) + orow);
#pragma unroll
          for (int c = 0; c < D / 8; ++c) {
            uint32_t w4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w4[e] = pack_bf16x2(__uint_as_float(ov[c * 8 + 2 * e]) * inv_l,
                                  __uint_as_float(ov[c * 8 + 2 * e + 1]) * inv_l);
            dst[c] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
          }
        } else {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.o) + orow);
#pragma unroll
          for (int c = 0; c < D / 4; ++c)
            dst[c] = make_float4(__uint_as_float(ov[4 * c]) * inv_l, __uint_as_float(ov[4 * c + 1]) * inv_l,
                                 __uint_as_float(ov[4 * c + 2]) * inv_l, __uint_as_float(ov[4 * c + 3]) * inv_l);
        }
        if (p.lse != nullptr)
          p.lse[(static_cast<size_t>(b) * p.H + h) * p.W + i] = (m_run + __log2f(l_run)) * 0.69314718055994531f;
      }
    } else {
      report_timeout(abort, p.status);
    }
  }

  // ---- teardown ------------------------------------------------------------
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, bool O_BF16>
cudaError_t launch_typed(const CUtensorMap& tm_k, const CUtensorMap& tm_v, const CUtensorMap& tm_r,
                         const Params& prm, cudaStream_t stream) {
  auto kern = relattn_tc_kernel<D, O_BF16>;
  constexpr int smem = Cfg<D>::kSmemBytes;
  static int configured_mask = 0;  // one bit per device ordinal < 32
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 32 || !(__atomic_load_n(&configured_mask, __ATOMIC_ACQUIRE) & (1 << dev))) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (dev < 32) __atomic_fetch_or(&configured_mask, 1 << dev, __ATOMIC_RELEASE);
  }
  const long long nqt = (prm.W + BM - 1) / BM;
  const long long nblocks = nqt * prm.B * prm.H;
  kern<<<static_cast<unsigned>(nblocks), kThreads, smem, stream>>>(tm_k, tm_v, tm_r, prm);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_relattn_tc(const CUtensorMap& tm_k, const CUtensorMap& tm_v, const CUtensorMap& tm_r,
                              const void* q, const float* bias_u, const float* bias_v, void* o,
                              float* lse, int B, int W, int M, int H, int D, bool o_bf16, float scale,
                              const WaitCtl& wc, cudaStream_t stream) {
  Params prm;
  prm.q = static_cast<const __nv_bfloat16*>(q);
  prm.bias_u = bias_u;
  prm.bias_v = bias_v;
  prm.o = o;
  prm.lse = lse;
  prm.B = B;
  prm.W = W;
  prm.M = M;
  prm.H = H;
  prm.scale_log2e = scale * 1.4426950408889634f;
  prm.status = wc.status;
  prm.wait_ns = wc.limit_ns;
  prm.inject_stall = wc.inject_stall;
  if (D == 64)
    return o_bf16 ? launch_typed<64, true>(tm_k, tm_v, tm_r, prm, stream)
                  : launch_typed<64, false>(tm_k, tm_v, tm_r, prm, stream);
  if (D == 128)
    return o_bf16 ? launch_typed<128, true>(tm_k, tm_v, tm_r, prm, stream)
                  : launch_typed<128, false>(tm_k, tm_v, tm_r, prm, stream);
  return cudaErrorInvalidValue;
}

}  // namespace txl
