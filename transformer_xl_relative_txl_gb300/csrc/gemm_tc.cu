// The layer's dense products on the sm_103a tensor cores:
//
//   C_z [m, n] = A [m, k] . B_z [k, n]  (+ bias [n])  (then ReLU),  z < batch
//
// bf16 A, B and C, row-major; fp32 accumulation in tensor memory; the bias
// (fp32) is added to the fp32 accumulator and the ReLU applied before the one
// rounding to bf16.  "Implementing Transformer-XL", recurrent-memory chapter:
// the input projections, the output projection and the two feed-forward
// products (with b_1 and the ReLU after the first, b_2 after the second).
//
// Design (one persistent CTA per SM, 192 threads):
//   warp 0     TMA producer: per k block (128 deep for BN = 64 or 128
//              column tiles, 64 deep for BN = 256), 128 x 64 tiles of A
//              (K-major, 128-byte swizzle) and BN/64 tiles of k-rows x 64
//              columns of B (N-major: B is stored [k, n] with n contiguous)
//              into a ring of shared-memory stages;
//   warp 1     MMA issuer: tcgen05.mma kind::f16, M = 128, N = BN, K = 16,
//              into one of two TMEM accumulators, so the next tile's
//              products overlap this tile's epilogue;
//   warps 2-5  epilogue: each reads its 32-lane quadrant of the accumulator
//              (tcgen05.ld, 64 columns at a time), adds the bias, applies the
//              ReLU, rounds to bf16, stages 32 rows x 64 columns in its own
//              128-byte-swizzled buffer and writes them with one TMA store.
// Tiles (z, m block, n block) are dealt round-robin, n block fastest, so the
// CTAs working at one time share A's rows through L2.  Out-of-range rows,
// columns and k (the tails) are zero-filled by the loads and clipped by the
// stores.  Every wait is bounded: a wait that runs out raises the device
// status word, every role unwinds and the tensor memory is freed.
#include <atomic>
#include <cstdint>

#include "pdl.cuh"
#include "relattn_tc_common.cuh"
#include "txl_device.cuh"
#include "txl_internal.h"

namespace txl {
namespace {

constexpr int GBM = 128;              // rows per tile (TMEM lanes)
constexpr int kATile = GBM * 128;     // 128 rows x 64 k of A: 16 KB (one 128-byte swizzle row of bf16 per row)
constexpr int kGemmThreads = 192;
constexpr int kEpiBytes = 32 * 128;   // one epilogue warp's staging: 32 rows x 64 bf16

// Per column-tile width: k per stage and stages.  Deeper stages (fewer
// barrier round trips and loads per FLOP) measured faster with 128-column
// tiles (W_2 of the base layer: 34.6 -> 31.8 us); with 256-column tiles they
// would leave two stages, and four of 64 k stay faster.
template <int BN>
struct GemmCfg {
  static constexpr int kBK = BN <= 128 ? 128 : 64;            // k per stage
  static constexpr int kABoxes = kBK / 64;                    // 64-k tiles of A per stage
  static constexpr int kBBlock = kBK * 128;                   // kBK k-rows x 64 columns of B
  static constexpr int kStageBytes = kABoxes * kATile + (BN / 64) * kBBlock;
  static constexpr int kStages = BN == 128 ? 3 : 4;
  static constexpr int kOffEpi = kStages * kStageBytes;             // 4 x 4 KB staging
  static constexpr int kOffBias = kOffEpi + 4 * kEpiBytes;          // 4 x BN floats
  static constexpr int kOffBar = kOffBias + 4 * BN * 4;
  static constexpr int kSmem = kOffBar + 256 + 1024;                // barriers, alignment slack
  static constexpr uint32_t kTmemCols = 2 * BN;                    // two accumulators
  static_assert(kSmem <= 232448, "shared memory budget");
};

struct GemmParams {
  int m, n, k, batch;
  int mt, nt;           // row and column blocks
  int tiles1;           // batch * mt * nt: the tiles of the first product
  int m2, mt2;          // a second product (its own A, B, C; same n and k), or m2 = 0
  int tiles;            // tiles1 + mt2 * nt
  const float* bias;    // [n] or nullptr (the first product only)
  int relu;             // the first product only
  unsigned int* status;
  unsigned long long wait_ns;
};

struct GemmBars {
  uint64_t full[8], empty[8];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t done;
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}

__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}

struct TileIdx {
  int prob, z, m0, n0;
};
// Tile t: the first product's tiles, batch index slowest, then the row
// block, the column block fastest; then the second product's.
__device__ __forceinline__ TileIdx tile_of(const GemmParams& p, int t, int bn) {
  TileIdx r;
  if (t >= p.tiles1) {
    t -= p.tiles1;
    r.prob = 1;
    r.z = 0;
    r.m0 = (t / p.nt) * GBM;
    r.n0 = (t % p.nt) * bn;
    return r;
  }
  const int per_z = p.mt * p.nt;
  r.prob = 0;
  r.z = t / per_z;
  const int rem = t - r.z * per_z;
  r.m0 = (rem / p.nt) * GBM;
  r.n0 = (rem % p.nt) * bn;
  return r;
}

template <int BN>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                   const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ CUtensorMap tm_a2,
                   const __grid_constant__ CUtensorMap tm_b2, const __grid_constant__ CUtensorMap tm_c2,
                   const GemmParams p) {
  // Launched behind the previous kernel on the stream, which has completed from
  // here on.  No early trigger: the next persistent launch starts its CTAs when
  // this one completes (placed early, they timed slower back to back).
  grid_dep_wait();
  using Cfg = GemmCfg<BN>;
  constexpr int S = Cfg::kStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  GemmBars* bars = reinterpret_cast<GemmBars*>(smem + Cfg::kOffBar);
  volatile int* abort = &bars->abort;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  constexpr int GBK = Cfg::kBK;
  constexpr int kBBlock = Cfg::kBBlock;
  constexpr int kBOff = Cfg::kABoxes * kATile;  // B's blocks follow A's tiles in a stage
  const int nk = (p.k + GBK - 1) / GBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&bars->acc_full[a], 1);
      mbar_init(&bars->acc_empty[a], 4);
    }
    mbar_init(&bars->done, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, Cfg::kTmemCols);
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
      tma_prefetch_desc(&tm_a);
      tma_prefetch_desc(&tm_b);
      if (p.m2 > 0) {
        tma_prefetch_desc(&tm_a2);
        tma_prefetch_desc(&tm_b2);
      }
      uint32_t it = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < p.tiles; t += gridDim.x) {
        const TileIdx ti = tile_of(p, t, BN);
        const int n0 = ti.n0;
        const CUtensorMap* ma = ti.prob ? &tm_a2 : &tm_a;
        const CUtensorMap* mb = ti.prob ? &tm_b2 : &tm_b;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = static_cast<int>(it % S);
          if (!(ok = mbar_wait(&bars->empty[s], ((it / S) & 1) ^ 1, wait_ns, abort))) break;
          uint8_t* st = smem + s * Cfg::kStageBytes;
          mbar_arrive_expect_tx(&bars->full[s], Cfg::kStageBytes);
#pragma unroll
          for (int a = 0; a < Cfg::kABoxes; ++a)
            tma_load_2d(st + a * kATile, ma, &bars->full[s], kb * GBK + 64 * a, ti.m0);
#pragma unroll
          for (int j = 0; j < BN / 64; ++j)
            tma_load_3d(st + kBOff + j * kBBlock, mb, &bars->full[s], n0 + 64 * j, kb * GBK, ti.z);
        }
      }
      if (!ok) report_timeout(abort, p.status);
      // let the loads in flight land before the CTA can exit
      for (int s = 0; s < S && static_cast<uint32_t>(s) < it; ++s) {
        const uint32_t last = s + ((it - 1 - s) / S) * S;
        mbar_wait_own(&bars->full[s], (last / S) & 1, wait_ns);
      }
    }
  } else if (warp == 1) {
    // ============================ MMA issuer ==============================
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(GBM, BN, false, true);
      const uint32_t base = smem_u32(smem);
      uint32_t it = 0, tl = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < p.tiles; t += gridDim.x, ++tl) {
        const uint32_t acc = tl & 1;
        // the epilogue has drained this accumulator (its use two tiles back)
        if (tl >= 2 && !(ok = mbar_wait(&bars->acc_empty[acc], ((tl >> 1) - 1) & 1, wait_ns, abort))) break;
        tc_fence_after();
        const uint32_t d = tmem + acc * BN;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = static_cast<int>(it % S);
          if (!(ok = mbar_wait(&bars->full[s], (it / S) & 1, wait_ns, abort))) break;
          tc_fence_after();
          const uint32_t st = base + s * Cfg::kStageBytes;
          // A: K-major, 128-byte swizzle, 8-row groups 1024 bytes apart, one
          // 16 KB tile per 64 k.  B: N-major, 64-column blocks kBBlock apart,
          // 8-k-row groups 1024 apart.
          const uint64_t da = sdesc_sw128(st, 16, 1024);
          const uint64_t db = sdesc_sw128(st + kBOff, kBBlock, 1024);
#pragma unroll
          for (int kk = 0; kk < GBK / 16; ++kk)
            mma_ss(d, da + (kk >> 2) * (kATile >> 4) + (kk & 3) * 2, db + ((kk * 16 * 128) >> 4), idesc,
                   (kb > 0 || kk > 0) ? 1u : 0u);
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
    const int quad = warp & 3;  // TMEM lane quadrant of this warp
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    uint8_t* stg = smem + Cfg::kOffEpi + quad * kEpiBytes;
    float* sbias = reinterpret_cast<float*>(smem + Cfg::kOffBias) + quad * BN;
    const int r = lane;  // row within the warp's 32
    uint32_t tl = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < p.tiles; t += gridDim.x, ++tl) {
      const TileIdx ti = tile_of(p, t, BN);
      const int n0 = ti.n0;
      const uint32_t acc = tl & 1;
      const float* bias = ti.prob ? nullptr : p.bias;  // bias and ReLU: the first product only
      const bool relu = ti.prob == 0 && p.relu;
      // this tile's bias columns, staged once for broadcast reads
      if (bias != nullptr) {
        __syncwarp();
#pragma unroll
        for (int i = 0; i < BN / 32; ++i) {
          const int c = n0 + 32 * i + lane;
          sbias[32 * i + lane] = c < p.n ? __ldg(bias + c) : 0.f;
        }
        __syncwarp();
      }
      if (!(ok = warp_wait(&bars->acc_full[acc], (tl >> 1) & 1, wait_ns, abort))) break;
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < BN / 64; ++c) {
        uint32_t v0[32], v1[32];
        tmem_ld32(tmem + lane_base + acc * BN + c * 64, v0);
        tmem_ld32(tmem + lane_base + acc * BN + c * 64 + 32, v1);
        tmem_wait_ld(v0);
        tmem_wait_ld(v1);
        if (c == BN / 64 - 1) {
          // every column of this accumulator is in registers: hand it back
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->acc_empty[acc]);
        }
        float x[64];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          x[j] = __uint_as_float(v0[j]);
          x[32 + j] = __uint_as_float(v1[j]);
        }
        if (bias != nullptr) {
#pragma unroll
          for (int j = 0; j < 64; j += 4) {
            const float4 b = *reinterpret_cast<const float4*>(sbias + c * 64 + j);
            x[j] += b.x;
            x[j + 1] += b.y;
            x[j + 2] += b.z;
            x[j + 3] += b.w;
          }
        }
        if (relu) {
#pragma unroll
          for (int j = 0; j < 64; ++j) x[j] = fmaxf(x[j], 0.f);
        }
        // the previous store out of the staging buffer has read it
        if (lane == 0) bulk_wait_group_read0();
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 8; ++j)
          *reinterpret_cast<uint4*>(stg + r * 128 + ((j ^ (r & 7)) * 16)) =
              make_uint4(pack_bf16x2(x[8 * j], x[8 * j + 1]), pack_bf16x2(x[8 * j + 2], x[8 * j + 3]),
                         pack_bf16x2(x[8 * j + 4], x[8 * j + 5]), pack_bf16x2(x[8 * j + 6], x[8 * j + 7]));
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_3d(ti.prob ? &tm_c2 : &tm_c, stg, n0 + 64 * c, ti.m0 + 32 * quad, ti.z);
          bulk_commit_group();
        }
      }
    }
    if (!ok) report_timeout(abort, p.status);
    if (lane == 0) bulk_wait_group0();  // every store is complete before the CTA exits
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::kTmemCols);
  }
}

int gemm_num_sms() {
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

template <int BN>
cudaError_t launch_bn(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc, const CUtensorMap& ta2,
                      const CUtensorMap& tb2, const CUtensorMap& tc2, const GemmParams& p, cudaStream_t stream) {
  using Cfg = GemmCfg<BN>;
  static std::atomic<bool> attr_done[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_done[dev].load()) {
    e = cudaFuncSetAttribute(gemm_tc_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
    if (e != cudaSuccess) return e;
    attr_done[dev].store(true);
  }
  const int sms = gemm_num_sms();
  const int grid = p.tiles < sms ? p.tiles : sms;
  return launch_dependent(gemm_tc_kernel<BN>, dim3(grid), dim3(kGemmThreads), Cfg::kSmem, stream, ta, tb, tc, ta2,
                          tb2, tc2, p);
}

}  // namespace

int gemm_tc_k_block(int bn) {
  return bn == 64 ? GemmCfg<64>::kBK : bn == 128 ? GemmCfg<128>::kBK : GemmCfg<256>::kBK;
}

std::atomic<int> g_force_tile_n{0};

void gemm_tc_force_tile_n(int bn) { g_force_tile_n.store(bn == 64 || bn == 128 || bn == 256 ? bn : 0); }

int gemm_tc_tile_n(int m, int n, int batch, int m2) {
  if (const int f = g_force_tile_n.load()) return f;
  // Fewer waves of tiles against smaller tiles: the time of a wave is about
  // proportional to its tiles' columns, plus a fixed part per tile.  A
  // second product of m2 rows counts as more rows of the batch's last one.
  const long long sms = gemm_num_sms();
  const long long mt = (m + GBM - 1) / GBM, mt2 = (m2 + GBM - 1) / GBM;
  // Too few 128-column tiles to fill half the SMs: 64-column ones spread
  // the work over twice as many (the r projection of the base layer,
  // 1024 x 512 x 512: 10.2 -> 8.2 us); they are slower wherever the wider
  // tiles already fill the GPU (W_2: 36.9 against 32.8 us).
  if (2 * (batch * mt + mt2) * ((n + 127) / 128) <= sms) return 64;
  auto cost = [&](int bn) {
    const long long tiles = (batch * mt + mt2) * ((n + bn - 1) / bn);
    const long long waves = (tiles + sms - 1) / sms;
    return static_cast<double>(waves) * (bn + 32);
  };
  return cost(128) < cost(256) ? 128 : 256;
}

cudaError_t launch_gemm_tc2(const CUtensorMap& tm_a, const CUtensorMap& tm_b, const CUtensorMap& tm_c, int m, int n,
                            int k, int batch, const float* bias, bool relu, const CUtensorMap& tm_a2,
                            const CUtensorMap& tm_b2, const CUtensorMap& tm_c2, int m2, int bn, const WaitCtl& wc,
                            cudaStream_t stream) {
  if (m <= 0 || n <= 0 || k <= 0 || batch <= 0 || m2 < 0 || (bn != 64 && bn != 128 && bn != 256))
    return cudaErrorInvalidValue;
  GemmParams p;
  p.m = m;
  p.n = n;
  p.k = k;
  p.batch = batch;
  p.mt = (m + GBM - 1) / GBM;
  p.nt = (n + bn - 1) / bn;
  p.m2 = m2;
  p.mt2 = (m2 + GBM - 1) / GBM;
  const long long tiles1 = static_cast<long long>(batch) * p.mt * p.nt;
  const long long tiles = tiles1 + static_cast<long long>(p.mt2) * p.nt;
  if (tiles > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  p.tiles1 = static_cast<int>(tiles1);
  p.tiles = static_cast<int>(tiles);
  p.bias = bias;
  p.relu = relu ? 1 : 0;
  p.status = wc.status;
  p.wait_ns = wc.limit_ns;
  if (bn == 64) return launch_bn<64>(tm_a, tm_b, tm_c, tm_a2, tm_b2, tm_c2, p, stream);
  if (bn == 256) return launch_bn<256>(tm_a, tm_b, tm_c, tm_a2, tm_b2, tm_c2, p, stream);
  return launch_bn<128>(tm_a, tm_b, tm_c, tm_a2, tm_b2, tm_c2, p, stream);
}

cudaError_t launch_gemm_tc(const CUtensorMap& tm_a, const CUtensorMap& tm_b, const CUtensorMap& tm_c, int m, int n,
                           int k, int batch, int bn, const float* bias, bool relu, const WaitCtl& wc,
                           cudaStream_t stream) {
  return launch_gemm_tc2(tm_a, tm_b, tm_c, m, n, k, batch, bias, relu, tm_a, tm_b, tm_c, 0, bn, wc, stream);
}

}  // namespace txl
