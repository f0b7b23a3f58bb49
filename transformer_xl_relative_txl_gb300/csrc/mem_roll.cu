// Memory roll: mem_out = last m' rows of [mem ; h], m' = min(m, m_prev + w)
// (the simulation's mem_tau = last M rows of [stop_grad(mem_{tau-1}) ; h_tau]).
//
// Per batch row-block the output is two contiguous byte ranges: the tail of
// the memory followed by the tail of the new segment.  The kernel copies them
// with the widest vector the alignment allows (16 bytes in practice), four
// independent vectors in flight per thread, grid y = batch.  HBM-bound: the
// algorithmic traffic is 2 * B * m' * row_bytes (read + write).
#include <cstdint>

#include "txl_internal.h"

namespace txl {
namespace {

template <typename V>
__global__ void __launch_bounds__(256) mem_roll_kernel(const char* __restrict__ mem, const char* __restrict__ h,
                                                       char* __restrict__ out, long long n_vec,
                                                       long long split_vec, long long mem_bs, long long h_bs,
                                                       long long out_bs) {
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
  mem_roll_kernel<V><<<grid, threads, 0, stream>>>(mem, h, out, n_vec, split, mem_bs, h_bs, out_bs);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_mem_roll(const void* mem, const void* h, void* out, int B, long long rows_out,
                            long long n_from_mem, long long mem_row0, long long h_row0, long long row_bytes,
                            long long mem_bs_bytes, long long h_bs_bytes, long long out_bs_bytes,
                            cudaStream_t stream) {
  const char* m = static_cast<const char*>(mem) + mem_row0 * row_bytes;
  const char* hh = static_cast<const char*>(h) + h_row0 * row_bytes;
  if (n_from_mem == 0) m = hh;  // no memory rows used: keep the pointer valid
  char* o = static_cast<char*>(out);
  const long long total = rows_out * row_bytes;
  const long long split = n_from_mem * row_bytes;
  auto aligned = [&](long long a) {
    const uintptr_t bits = reinterpret_cast<uintptr_t>(m) | reinterpret_cast<uintptr_t>(hh) |
                           reinterpret_cast<uintptr_t>(o) | static_cast<uintptr_t>(row_bytes) |
                           static_cast<uintptr_t>(mem_bs_bytes) | static_cast<uintptr_t>(h_bs_bytes) |
                           static_cast<uintptr_t>(out_bs_bytes);
    return (bits % static_cast<uintptr_t>(a)) == 0;
  };
  if (aligned(16))
    return launch_typed<uint4>(m, hh, o, B, total, split, mem_bs_bytes, h_bs_bytes, out_bs_bytes, stream);
  if (aligned(4))
    return launch_typed<uint32_t>(m, hh, o, B, total, split, mem_bs_bytes, h_bs_bytes, out_bs_bytes, stream);
  if (aligned(2))
    return launch_typed<uint16_t>(m, hh, o, B, total, split, mem_bs_bytes, h_bs_bytes, out_bs_bytes, stream);
  return launch_typed<uint8_t>(m, hh, o, B, total, split, mem_bs_bytes, h_bs_bytes, out_bs_bytes, stream);
}

}  // namespace txl
