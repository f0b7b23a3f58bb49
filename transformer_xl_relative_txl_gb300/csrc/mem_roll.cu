// Memory roll: mem_out = last m' rows of [mem ; h], m' = min(m, m_prev + w)
// (the simulation's mem_tau = last M rows of [stop_grad(mem_{tau-1}) ; h_tau]).
//
// Per batch the output is two contiguous byte ranges: the tail of the memory
// followed by the tail of the new segment.  HBM-bound: the algorithmic
// traffic is 2 * B * m' * row_bytes (read + write) per tensor.
//
// Two kernels:
//   - mem_roll_bulk_kernel, when every address, stride and row is a multiple
//     of 16 bytes: the ranges are cut into 16 KiB chunks dealt round-robin
//     to a persistent grid (two CTAs per SM); one thread per CTA streams its
//     chunks through a ring of shared-memory stages with bulk copies
//     (cp.async.bulk global -> shared completing on an mbarrier, then shared
//     -> global), so every SM keeps up to 192 KiB in flight with a handful of
//     instructions per chunk.  One launch rolls one or two tensors (keys and
//     values) of the same geometry.
//   - mem_roll_kernel otherwise: vector loads and stores of the widest width
//     the alignment allows, four in flight per thread, grid y = batch.
#include <atomic>
#include <cstdint>

#include "pdl.cuh"
#include "txl_device.cuh"
#include "txl_internal.h"

namespace txl {
namespace {

// ---------------------------------------------------------------------------
// Bulk-copy kernel
// ---------------------------------------------------------------------------
constexpr int kChunk = 16384;  // bytes per bulk copy
constexpr int kStages = 6;     // shared-memory stages per CTA (96 KiB: two CTAs per SM)
constexpr int kMaxParts = 4;   // two source ranges x two tensors

struct BulkPart {
  const char* src;      // first byte of batch 0's range
  char* dst;            // first output byte of batch 0's range
  long long src_bs;     // batch strides, bytes
  long long dst_bs;
  long long bytes;      // range length per batch (a multiple of 16)
  long long nchunk;     // chunks per batch
  long long first;      // index of this part's first chunk
};

struct BulkParams {
  BulkPart part[kMaxParts];
  int nparts;
  long long total;  // chunks of all parts and batches
  unsigned int* status;
  unsigned long long wait_ns;
};

__device__ __forceinline__ void bulk_load(void* dst_smem, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst_smem)),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void bulk_store(void* dst, const void* src_smem, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(reinterpret_cast<uint64_t>(dst)),
               "r"(smem_u32(src_smem)), "r"(bytes)
               : "memory");
}

// Waits until all but the most recently committed bulk store have read
// their shared-memory source.
__device__ __forceinline__ void bulk_wait_group_read1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}

// Source, destination and size of chunk c.
__device__ __forceinline__ void chunk_at(const BulkParams& p, long long c, const char** src, char** dst,
                                         uint32_t* bytes) {
  int q = 0;
#pragma unroll
  for (int x = 1; x < kMaxParts; ++x)
    if (x < p.nparts && c >= p.part[x].first) q = x;
  const BulkPart& pt = p.part[q];
  const long long local = c - pt.first;
  const long long b = local / pt.nchunk;
  const long long off = (local - b * pt.nchunk) * kChunk;
  const long long left = pt.bytes - off;
  *src = pt.src + b * pt.src_bs + off;
  *dst = pt.dst + b * pt.dst_bs + off;
  *bytes = static_cast<uint32_t>(left < kChunk ? left : kChunk);
}

__global__ void __launch_bounds__(32) mem_roll_bulk_kernel(const __grid_constant__ BulkParams p) {
  grid_dep_wait();  // launched behind the previous kernel on the stream: it has completed from here on
  grid_dep_launch_dependents();
  extern __shared__ __align__(128) unsigned char stage[];  // kStages x kChunk
  __shared__ __align__(8) uint64_t bar[kStages];
  if (threadIdx.x != 0) return;
  for (int s = 0; s < kStages; ++s) mbar_init(&bar[s], 1);
  fence_mbar_init();
  const long long G = gridDim.x;
  const long long n = p.total > blockIdx.x ? (p.total - blockIdx.x + G - 1) / G : 0;  // chunks of this CTA
  auto load = [&](long long i) {
    const char* src;
    char* dst;
    uint32_t bytes;
    chunk_at(p, blockIdx.x + i * G, &src, &dst, &bytes);
    const int s = static_cast<int>(i % kStages);
    mbar_arrive_expect_tx(&bar[s], bytes);
    bulk_load(stage + static_cast<size_t>(s) * kChunk, src, bytes, &bar[s]);
  };
  long long issued = 0;  // loads issued so far (chunks 0 .. issued-1)
  for (; issued < n && issued < kStages; ++issued) load(issued);
  long long i = 0;
  for (; i < n; ++i) {
    const int s = static_cast<int>(i % kStages);
    if (!mbar_wait_own(&bar[s], static_cast<uint32_t>((i / kStages) & 1), p.wait_ns)) {
      atomicOr(p.status, kStatusTimeoutBit);
      break;
    }
    const char* src;
    char* dst;
    uint32_t bytes;
    chunk_at(p, blockIdx.x + i * G, &src, &dst, &bytes);
    bulk_store(dst, stage + static_cast<size_t>(s) * kChunk, bytes);
    bulk_commit_group();
    // Refill the stage of chunk i-1 once its store has read it.
    if (i >= 1 && issued < n) {
      bulk_wait_group_read1();
      load(issued++);
    }
  }
  // After a timed-out wait, let the loads already issued land before exit.
  for (; i < issued; ++i)
    if (!mbar_wait_own(&bar[i % kStages], static_cast<uint32_t>((i / kStages) & 1), p.wait_ns)) break;
  bulk_wait_group0();
}

// ---------------------------------------------------------------------------
// Vector kernel (any alignment)
// ---------------------------------------------------------------------------
template <typename V>
__global__ void __launch_bounds__(256) mem_roll_kernel(const char* __restrict__ mem, const char* __restrict__ h,
                                                       char* __restrict__ out, long long n_vec,
                                                       long long split_vec, long long mem_bs, long long h_bs,
                                                       long long out_bs) {
  grid_dep_wait();  // launched behind the previous kernel on the stream: it has completed from here on
  grid_dep_launch_dependents();
  const long long b = blockIdx.y;
  const V* src_mem = reinterpret_cast<const V*>(mem + b * mem_bs);
  const V* src_h = reinterpret_cast<const V*>(h + b * h_bs);
  V* dst = reinterpret_cast<V*>(out + b * out_bs);
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x * 4;
  for (long long base = static_cast<long long>(blockIdx.x) * blockDim.x * 4 + threadIdx.x; base < n_vec;
       base += stride) {
    V tmp[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const long long i = base + static_cast<long long>(u) * blockDim.x;
      if (i < n_vec) tmp[u] = (i < split_vec) ? __ldg(src_mem + i) : __ldg(src_h + (i - split_vec));
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const long long i = base + static_cast<long long>(u) * blockDim.x;
      if (i < n_vec) dst[i] = tmp[u];
    }
  }
}

template <typename V>
cudaError_t launch_typed(const char* mem, const char* h, char* out, int B, long long total_bytes,
                         long long split_bytes, long long mem_bs, long long h_bs, long long out_bs,
                         cudaStream_t stream) {
  const long long n_vec = total_bytes / static_cast<long long>(sizeof(V));
  const long long split = split_bytes / static_cast<long long>(sizeof(V));
  const int threads = 256;
  long long blocks = (n_vec + threads * 4 - 1) / (threads * 4);
  // Enough blocks in total to keep every SM busy; each grid-strides.
  const long long target = (152LL * 8 + B - 1) / B;
  if (blocks > target) blocks = target;
  if (blocks < 1) blocks = 1;
  dim3 grid(static_cast<unsigned>(blocks), static_cast<unsigned>(B));
  return launch_dependent(mem_roll_kernel<V>, grid, dim3(threads), 0, stream, mem, h, out, n_vec, split, mem_bs, h_bs,
                          out_bs);
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess)
    return 152;
  return n > 0 ? n : 152;
}

}  // namespace

cudaError_t launch_mem_roll_multi(const RollTensor* t, int ntensors, int B, long long rows_out, long long n_from_mem,
                                  long long mem_row0, long long h_row0, long long row_bytes, long long mem_bs_bytes,
                                  long long h_bs_bytes, long long out_bs_bytes, const WaitCtl* wc,
                                  cudaStream_t stream) {
  if (ntensors < 1 || ntensors > 2) return cudaErrorInvalidValue;
  const long long total = rows_out * row_bytes;
  const long long split = n_from_mem * row_bytes;
  // Every byte range on a 16-byte boundary: the bulk-copy kernel.
  uintptr_t bits = static_cast<uintptr_t>(row_bytes) | static_cast<uintptr_t>(mem_bs_bytes) |
                   static_cast<uintptr_t>(h_bs_bytes) | static_cast<uintptr_t>(out_bs_bytes);
  for (int x = 0; x < ntensors; ++x) {
    if (split > 0) bits |= reinterpret_cast<uintptr_t>(t[x].mem);
    if (total > split) bits |= reinterpret_cast<uintptr_t>(t[x].h);
    bits |= reinterpret_cast<uintptr_t>(t[x].out);
  }
  if (wc != nullptr && bits % 16 == 0) {
    BulkParams p{};
    long long first = 0;
    for (int x = 0; x < ntensors; ++x) {
      const long long sizes[2] = {split, total - split};
      const long long sbs[2] = {mem_bs_bytes, h_bs_bytes};
      long long dst_off = 0;
      for (int y = 0; y < 2; ++y) {
        if (sizes[y] > 0) {
          BulkPart& pt = p.part[p.nparts++];
          pt.src = y == 0 ? static_cast<const char*>(t[x].mem) + mem_row0 * row_bytes
                          : static_cast<const char*>(t[x].h) + h_row0 * row_bytes;
          pt.dst = static_cast<char*>(t[x].out) + dst_off;
          pt.src_bs = sbs[y];
          pt.dst_bs = out_bs_bytes;
          pt.bytes = sizes[y];
          pt.nchunk = (sizes[y] + kChunk - 1) / kChunk;
          pt.first = first;
          first += pt.nchunk * B;
        }
        dst_off += sizes[y];
      }
    }
    p.total = first;
    p.status = wc->status;
    p.wait_ns = wc->limit_ns;
    if (p.total == 0) return cudaSuccess;
    const size_t smem = static_cast<size_t>(kStages) * kChunk;
    static std::atomic<bool> attr_set[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev].load()) {
      e = cudaFuncSetAttribute(mem_roll_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem));
      if (e != cudaSuccess) return e;
      attr_set[dev].store(true);
    }
    const long long cap = 2LL * sm_count();
    const unsigned grid = static_cast<unsigned>(p.total < cap ? p.total : cap);
    return launch_dependent(mem_roll_bulk_kernel, dim3(grid), dim3(32), smem, stream, p);
  }
  for (int x = 0; x < ntensors; ++x) {
    const char* hh = total > split ? static_cast<const char*>(t[x].h) + h_row0 * row_bytes : nullptr;
    const char* m = split > 0 ? static_cast<const char*>(t[x].mem) + mem_row0 * row_bytes : hh;
    if (hh == nullptr) hh = m;  // every row from the memory: keep the pointer valid
    char* o = static_cast<char*>(t[x].out);
    auto aligned = [&](long long a) {
      const uintptr_t v = reinterpret_cast<uintptr_t>(m) | reinterpret_cast<uintptr_t>(hh) |
                          reinterpret_cast<uintptr_t>(o) | static_cast<uintptr_t>(row_bytes) |
                          static_cast<uintptr_t>(mem_bs_bytes) | static_cast<uintptr_t>(h_bs_bytes) |
                          static_cast<uintptr_t>(out_bs_bytes);
      return (v % static_cast<uintptr_t>(a)) == 0;
    };
    cudaError_t e;
    if (aligned(16))
      e = launch_typed<uint4>(m, hh, o, B, total, split, mem_bs_bytes, h_bs_bytes, out_bs_bytes, stream);
    else if (aligned(4))
      e = launch_typed<uint32_t>(m, hh, o, B, total, split, mem_bs_bytes, h_bs_bytes, out_bs_bytes, stream);
    else if (aligned(2))
      e = launch_typed<uint16_t>(m, hh, o, B, total, split, mem_bs_bytes, h_bs_bytes, out_bs_bytes, stream);
    else
      e = launch_typed<uint8_t>(m, hh, o, B, total, split, mem_bs_bytes, h_bs_bytes, out_bs_bytes, stream);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_mem_roll(const void* mem, const void* h, void* out, int B, long long rows_out,
                            long long n_from_mem, long long mem_row0, long long h_row0, long long row_bytes,
                            long long mem_bs_bytes, long long h_bs_bytes, long long out_bs_bytes,
                            cudaStream_t stream) {
  const RollTensor t{mem, h, out};
  return launch_mem_roll_multi(&t, 1, B, rows_out, n_from_mem, mem_row0, h_row0, row_bytes, mem_bs_bytes, h_bs_bytes,
                               out_bs_bytes, nullptr, stream);
}

}  // namespace txl
