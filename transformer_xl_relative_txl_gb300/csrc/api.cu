// C ABI of the library (see include/txl_relattn.h): argument validation,
// alias checks, TMA descriptor encoding, device status word, dispatch.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <map>
#include <vector>
#include <mutex>
#include <utility>

#include "txl_internal.h"
#include "txl_relattn.h"

namespace {

// Device status word: kernels OR error bits into it; read and cleared by
// txl_get_device_status.
__device__ unsigned int g_txl_status;

std::atomic<unsigned long long> g_wait_ns{2000000000ULL};
std::atomic<int> g_inject_stall{0};
std::atomic<int> g_force_split{0};  // test hook: > 0 forces the D = 64 kernel's split count
std::atomic<int> g_bwd_path{0};     // test hook: the bf16 D = 64 backward's path (1 fused, 2 pair terms, 0 the choice)

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
unsigned int* g_status_ptr[kMaxDevices] = {};

cudaError_t status_ptr(unsigned int** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mutex);
  if (g_status_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_txl_status);
    if (e != cudaSuccess) return e;
    g_status_ptr[dev] = static_cast<unsigned int*>(p);
  }
  *out = g_status_ptr[dev];
  return cudaSuccess;
}

// Scratch for split key ranges, per (device, stream) so that calls on
// different streams never share it: the chunks' partial results, and the
// merge counters, which live in their own buffer because the kernel relies on
// them being zero at launch (it leaves them at zero; a new counter buffer is
// zeroed).  Buffers grow on demand (the stream is synchronised before an old
// one is freed) and live until the process exits.
struct ScratchBuf {
  void* ptr = nullptr;
  size_t bytes = 0;
  int* cnt = nullptr;
  size_t cnt_n = 0;
};
std::map<std::pair<int, cudaStream_t>, ScratchBuf> g_scratch;

cudaError_t split_scratch(cudaStream_t stream, size_t bytes, size_t n_counters, void** out, int** counters) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(g_mutex);
  ScratchBuf& b = g_scratch[{dev, stream}];
  if (b.bytes < bytes || b.cnt_n < n_counters) {
    if ((b.ptr != nullptr || b.cnt != nullptr) && (e = cudaStreamSynchronize(stream)) != cudaSuccess) return e;
    if (b.bytes < bytes) {
      if (b.ptr != nullptr && (e = cudaFree(b.ptr)) != cudaSuccess) return e;
      b.ptr = nullptr;
      b.bytes = 0;
      if ((e = cudaMalloc(&b.ptr, bytes)) != cudaSuccess) return e;
      b.bytes = bytes;
    }
    if (b.cnt_n < n_counters) {
      if (b.cnt != nullptr && (e = cudaFree(b.cnt)) != cudaSuccess) return e;
      b.cnt = nullptr;
      b.cnt_n = 0;
      if ((e = cudaMalloc(&b.cnt, n_counters * sizeof(int))) != cudaSuccess) return e;
      b.cnt_n = n_counters;
      if ((e = cudaMemsetAsync(b.cnt, 0, n_counters * sizeof(int), stream)) != cudaSuccess) return e;
    }
  }
  *out = b.ptr;
  *counters = b.cnt;
  return cudaSuccess;
}

// Contiguous copies of a ring's keys and values for the ring calls the
// kernels cannot read in place, per (device, stream); grows on demand.
std::map<std::pair<int, cudaStream_t>, std::pair<void*, size_t>> g_gather;

cudaError_t gather_scratch(cudaStream_t stream, size_t bytes, void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(g_mutex);
  auto& b = g_gather[{dev, stream}];
  if (b.second < bytes) {
    if (b.first != nullptr) {
      if ((e = cudaStreamSynchronize(stream)) != cudaSuccess || (e = cudaFree(b.first)) != cudaSuccess) return e;
      b = {nullptr, 0};
    }
    if ((e = cudaMalloc(&b.first, bytes)) != cudaSuccess) return e;
    b.second = bytes;
  }
  *out = b.first;
  return cudaSuccess;
}

// Fixed scratch of txl_relattn_forward_static, which allocates nothing: the
// merge counters (kStaticCounters ints, zero at module load and left at zero
// by the kernel), then the chunks' partial results.  Shared by every call on
// the device, so such calls must not run concurrently.
constexpr size_t kStaticScratchBytes = size_t(16) << 20;
constexpr size_t kStaticCounters = 4096;  // units x 4 lane quadrants
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];
unsigned char* g_static_ptr[kMaxDevices] = {};

cudaError_t static_scratch(unsigned char** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mutex);
  if (g_static_ptr[dev] == nullptr) {
    void* p = nullptr;
    if ((e = cudaGetSymbolAddress(&p, g_static_scratch)) != cudaSuccess) return e;
    g_static_ptr[dev] = static_cast<unsigned char*>(p);
  }
  *out = g_static_ptr[dev];
  return cudaSuccess;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

size_t dsize(txl_dtype t) { return t == TXL_BF16 ? 2 : 4; }
bool dtype_ok(int t) { return t == TXL_F32 || t == TXL_BF16; }

struct Range {
  uintptr_t lo, hi;  // [lo, hi)
};
Range range_of(const void* p, size_t bytes) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  return Range{a, a + bytes};
}
bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi && a.hi > a.lo && b.hi > b.lo; }
bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// 2*pi split for the sinusoid's Cody-Waite reduction: c1 and c2 keep few
// enough significant bits that n*c1 and n*c2 are exact for every multiple n
// the table can need; c3 carries the rest.
void two_pi_split(int n_dist, float* c1, float* c2, float* c3) {
  const double two_pi = 6.283185307179586476925286766559;
  int nbits = 1;
  while (std::ldexp(1.0, nbits) < static_cast<double>(n_dist) / two_pi + 2.0) ++nbits;
  int keep = 24 - nbits;
  if (keep < 1) keep = 1;
  auto keep_bits = [](double x, int bits) {
    float f = static_cast<float>(x);
    uint32_t u;
    std::memcpy(&u, &f, 4);
    const int drop = 24 - bits;
    if (drop > 0) u &= ~((1u << drop) - 1u);
    std::memcpy(&f, &u, 4);
    return f;
  };
  *c1 = keep_bits(two_pi, keep);
  *c2 = keep_bits(two_pi - static_cast<double>(*c1), keep);
  *c3 = static_cast<float>(two_pi - static_cast<double>(*c1) - static_cast<double>(*c2));
}

int from_cuda(cudaError_t e) { return e == cudaSuccess ? TXL_OK : TXL_ERR_CUDA; }

// Wait bound and status word for a launch.
int wait_ctl(txl::WaitCtl* wc) {
  if (status_ptr(&wc->status) != cudaSuccess) return TXL_ERR_CUDA;
  wc->limit_ns = g_wait_ns.load();
  wc->inject_stall = 0;
  return TXL_OK;
}

// The memory roll of n (1 or 2) tensors of one geometry in one launch:
// validation, alias checks (every output against every input and against
// the other output), then the roll kernel.
int roll_impl(const txl::RollTensor* t, int n, int m_prev, int w, int m, int B, int C, long long mem_bs,
              long long h_bs, long long out_bs, int* m_out, txl_dtype dtype, cudaStream_t stream) {
  if (B < 0 || m_prev < 0 || w < 0 || m < 0 || C <= 0 || !dtype_ok(dtype)) return TXL_ERR_INVALID_ARG;
  const long long keep = std::min<long long>(m, static_cast<long long>(m_prev) + w);
  if (m_out != nullptr) *m_out = static_cast<int>(keep);
  if (B == 0 || keep == 0) return TXL_OK;
  if (B > 65535) return TXL_ERR_UNSUPPORTED;
  const long long from_h = std::min<long long>(keep, w);
  const long long from_mem = keep - from_h;
  for (int x = 0; x < n; ++x) {
    if (t[x].out == nullptr) return TXL_ERR_INVALID_ARG;
    if (from_mem > 0 && t[x].mem == nullptr) return TXL_ERR_INVALID_ARG;
    if (from_h > 0 && t[x].h == nullptr) return TXL_ERR_INVALID_ARG;
  }
  const long long es = static_cast<long long>(dsize(dtype));
  if (B > 1 && (mem_bs < static_cast<long long>(m_prev) * C || h_bs < static_cast<long long>(w) * C ||
                out_bs < keep * C))
    return TXL_ERR_INVALID_ARG;
  if (mem_bs < 0 || h_bs < 0 || out_bs < 0) return TXL_ERR_INVALID_ARG;
  const long long row_bytes = static_cast<long long>(C) * es;
  // Extents actually read / written (all batches).
  std::vector<Range> outs, ins;
  for (int x = 0; x < n; ++x) {
    outs.push_back(range_of(t[x].out, static_cast<size_t>((B - 1) * out_bs * es + keep * row_bytes)));
    if (from_mem > 0) {
      const char* src = static_cast<const char*>(t[x].mem) + (m_prev - from_mem) * row_bytes;
      ins.push_back(range_of(src, static_cast<size_t>((B - 1) * mem_bs * es + from_mem * row_bytes)));
    }
    if (from_h > 0) {
      const char* src = static_cast<const char*>(t[x].h) + (w - from_h) * row_bytes;
      ins.push_back(range_of(src, static_cast<size_t>((B - 1) * h_bs * es + from_h * row_bytes)));
    }
  }
  for (size_t x = 0; x < outs.size(); ++x) {
    for (const Range& y : ins)
      if (overlap(outs[x], y)) return TXL_ERR_ALIAS;
    for (size_t z = x + 1; z < outs.size(); ++z)
      if (overlap(outs[x], outs[z])) return TXL_ERR_ALIAS;
  }
  txl::WaitCtl wc;
  if (wait_ctl(&wc) != TXL_OK) return TXL_ERR_CUDA;
  return from_cuda(txl::launch_mem_roll_multi(t, n, B, keep, from_mem, m_prev - from_mem, w - from_h, row_bytes,
                                              mem_bs * es, h_bs * es, out_bs * es, &wc, stream));
}

// The dense product of the layer on this library's tensor-core GEMM:
// C_z = A B_z (+ bias) (ReLU), bf16 row-major, A [m, k] shared, B_z
// [k, n] at B + z b_stride, C_z [m, n] at C + z c_stride (elements); with
// m2 > 0 also C2 [m2, n] = A2 [m2, k] B2 [k, n] in the same launch.
// Arguments already validated (alignment, strides).
int dense_impl(const void* A, const void* B, void* C, int m, int n, int k, int batch, long long b_stride,
               long long c_stride, const float* bias, bool relu, cudaStream_t stream, const void* A2 = nullptr,
               const void* B2 = nullptr, void* C2 = nullptr, int m2 = 0) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (encode == nullptr) return TXL_ERR_CUDA;
  const cuuint32_t estr[3] = {1, 1, 1};
  auto enc = [&](CUtensorMap* map, const void* base, cuuint32_t rank, const cuuint64_t* dims,
                 const cuuint64_t* strides, const cuuint32_t* box) {
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  };
  const int bn = txl::gemm_tc_tile_n(m, n, batch, m2);
  CUtensorMap ta, tb, tc, ta2, tb2, tc2;
  {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(k), static_cast<cuuint64_t>(m)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(k) * 2};
    const cuuint32_t box[2] = {64, 128};
    if (!enc(&ta, A, 2, dims, strides, box)) return TXL_ERR_CUDA;
  }
  {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(n), static_cast<cuuint64_t>(k),
                                static_cast<cuuint64_t>(batch)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(n) * 2, static_cast<cuuint64_t>(b_stride) * 2};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(txl::gemm_tc_k_block(bn)), 1};
    if (!enc(&tb, B, 3, dims, strides, box)) return TXL_ERR_CUDA;
  }
  {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(n), static_cast<cuuint64_t>(m),
                                static_cast<cuuint64_t>(batch)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(n) * 2, static_cast<cuuint64_t>(c_stride) * 2};
    const cuuint32_t box[3] = {64, 32, 1};
    if (!enc(&tc, C, 3, dims, strides, box)) return TXL_ERR_CUDA;
  }
  if (m2 > 0) {
    const cuuint64_t da[2] = {static_cast<cuuint64_t>(k), static_cast<cuuint64_t>(m2)};
    const cuuint64_t sa[1] = {static_cast<cuuint64_t>(k) * 2};
    const cuuint32_t ba[2] = {64, 128};
    const cuuint64_t db[3] = {static_cast<cuuint64_t>(n), static_cast<cuuint64_t>(k), 1};
    const cuuint64_t sb[2] = {static_cast<cuuint64_t>(n) * 2, static_cast<cuuint64_t>(n) * k * 2};
    const cuuint32_t bb[3] = {64, static_cast<cuuint32_t>(txl::gemm_tc_k_block(bn)), 1};
    const cuuint64_t dc[3] = {static_cast<cuuint64_t>(n), static_cast<cuuint64_t>(m2), 1};
    const cuuint64_t sc[2] = {static_cast<cuuint64_t>(n) * 2, static_cast<cuuint64_t>(n) * m2 * 2};
    const cuuint32_t bc[3] = {64, 32, 1};
    if (!enc(&ta2, A2, 2, da, sa, ba) || !enc(&tb2, B2, 3, db, sb, bb) || !enc(&tc2, C2, 3, dc, sc, bc))
      return TXL_ERR_CUDA;
  } else {
    ta2 = ta;
    tb2 = tb;
    tc2 = tc;
  }
  txl::WaitCtl wc;
  if (wait_ctl(&wc) != TXL_OK) return TXL_ERR_CUDA;
  return from_cuda(
      txl::launch_gemm_tc2(ta, tb, tc, m, n, k, batch, bias, relu, ta2, tb2, tc2, m2, bn, wc, stream));
}

// txl_mem_ring_append for n (1 or 2) rings of one geometry, each run of
// rows in one launch for all of them.
int ring_append_impl(void* const* mem, const void* const* h, int n, int cap, int start, int m, int w, int B, int C,
                     long long h_bs, int* start_out, int* m_out, txl_dtype dtype, cudaStream_t stream) {
  if (B < 0 || cap <= 0 || m < 0 || m > cap || w < 0 || C <= 0 || !dtype_ok(dtype)) return TXL_ERR_INVALID_ARG;
  if (m > 0 && (start < 0 || start >= cap)) return TXL_ERR_INVALID_ARG;
  if (m == 0) start = 0;
  const long long total = static_cast<long long>(m) + w;
  const long long drop = total > cap ? total - cap : 0;  // oldest rows pushed out
  const int new_start = static_cast<int>((start + drop) % cap);
  const int new_m = static_cast<int>(std::min<long long>(total, cap));
  if (B == 0 || w == 0) {
    if (start_out != nullptr) *start_out = new_start;
    if (m_out != nullptr) *m_out = new_m;
    return TXL_OK;
  }
  if ((B > 1 && h_bs < static_cast<long long>(w) * C) || h_bs < 0) return TXL_ERR_INVALID_ARG;
  if (B > 65535) return TXL_ERR_UNSUPPORTED;
  const long long es = static_cast<long long>(dsize(dtype)), row_bytes = static_cast<long long>(C) * es;
  for (int x = 0; x < n; ++x) {
    if (mem[x] == nullptr || h[x] == nullptr) return TXL_ERR_INVALID_ARG;
    const Range rm = range_of(mem[x], static_cast<size_t>(B) * cap * row_bytes);
    for (int y = 0; y < n; ++y) {
      if (overlap(rm, range_of(h[y], static_cast<size_t>((B - 1) * h_bs * es + w * row_bytes)))) return TXL_ERR_ALIAS;
      if (y > x && overlap(rm, range_of(mem[y], static_cast<size_t>(B) * cap * row_bytes))) return TXL_ERR_ALIAS;
    }
  }
  txl::WaitCtl wc;
  if (wait_ctl(&wc) != TXL_OK) return TXL_ERR_CUDA;
  // rows x0 .. w-1 of h go to ring rows (start + m + x) % cap: one or two runs
  const long long x0 = w > cap ? w - cap : 0;
  long long x = x0;
  while (x < w) {
    const long long dst = (start + m + x) % cap;
    const long long len = std::min<long long>(w - x, cap - dst);
    txl::RollTensor t[2];
    for (int y = 0; y < n; ++y)
      t[y] = txl::RollTensor{nullptr, static_cast<const char*>(h[y]) + x * row_bytes,
                             static_cast<char*>(mem[y]) + dst * row_bytes};
    if (txl::launch_mem_roll_multi(t, n, B, len, 0, 0, 0, row_bytes, 0, h_bs * es, cap * row_bytes, &wc, stream) !=
        cudaSuccess)
      return TXL_ERR_CUDA;
    x += len;
  }
  if (start_out != nullptr) *start_out = new_start;
  if (m_out != nullptr) *m_out = new_m;
  return TXL_OK;
}

}  // namespace

extern "C" {

int txl_version(void) { return TXL_VERSION; }

const char* txl_status_string(int status) {
  switch (status) {
    case TXL_OK: return "TXL_OK";
    case TXL_ERR_INVALID_ARG: return "TXL_ERR_INVALID_ARG";
    case TXL_ERR_UNSUPPORTED: return "TXL_ERR_UNSUPPORTED";
    case TXL_ERR_ALIAS: return "TXL_ERR_ALIAS";
    case TXL_ERR_CUDA: return "TXL_ERR_CUDA";
    case TXL_ERR_DEVICE_TIMEOUT: return "TXL_ERR_DEVICE_TIMEOUT";
    default: return "TXL_ERR_UNKNOWN";
  }
}

int txl_debug_set_wait_limit_ns(unsigned long long ns) {
  if (ns < 1000ULL) return TXL_ERR_INVALID_ARG;
  g_wait_ns.store(ns);
  return TXL_OK;
}

int txl_debug_inject_stall(int on) {
  g_inject_stall.store(on ? 1 : 0);
  return TXL_OK;
}

int txl_debug_set_bwd_chunk_bytes(unsigned long long bytes) {
  txl::relattn_bwd_pairs_set_chunk_bytes(static_cast<size_t>(bytes));
  return TXL_OK;
}

int txl_debug_pair_split_tiles(int n_query_tiles, int seq_heads, int W, int M, int sms) {
  if (n_query_tiles < 0 || seq_heads < 0 || W < 0 || M < 0 || sms <= 0) return -1;
  return txl::relattn_bwd_pairs_split_tiles(n_query_tiles, seq_heads, W, M, sms);
}

int txl_debug_attention_split(int B, int H, int W, int M, int sms) {
  if (B <= 0 || H <= 0 || W <= 0 || M < 0 || sms <= 0) return -1;
  return txl::relattn_tc64_split_for(B, H, W, M, sms);
}

int txl_debug_attention_items(int B, int H, int W, int M, int nsplit, int* items, int cap, int* n_items) {
  return txl::relattn_tc64_items(B, H, W, M, nsplit, items, cap, n_items);
}

int txl_debug_unit_plan(int B, int H, int W, int M, int ctas, int* table, int cap, int* stride) {
  return txl::relattn_tc64_plan_table(B, H, W, M, ctas, table, cap, stride);
}

int txl_debug_bwd_pairs_work(int B, int W, int M, int H, int split_qt, int* n_ctas, int* n_tiles, int* ctas,
                             int cap_ctas, int* tiles, int cap_tiles) {
  return txl::relattn_bwd_pairs_work(B, W, M, H, split_qt, n_ctas, n_tiles, ctas, cap_ctas, tiles, cap_tiles);
}

int txl_debug_force_bwd_path(int path) {
  if (path < 0 || path > 2) return TXL_ERR_INVALID_ARG;
  g_bwd_path.store(path);
  return TXL_OK;
}

int txl_debug_force_dense_tile_n(int bn) {
  if (bn != 0 && bn != 64 && bn != 128 && bn != 256) return TXL_ERR_INVALID_ARG;
  txl::gemm_tc_force_tile_n(bn);
  return TXL_OK;
}

int txl_debug_force_split(int nsplit) {
  if (nsplit < 0 || nsplit > 64) return TXL_ERR_INVALID_ARG;
  g_force_split.store(nsplit);
  return TXL_OK;
}

int txl_get_device_status(cudaStream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return TXL_ERR_CUDA;
  unsigned int* p = nullptr;
  if (status_ptr(&p) != cudaSuccess) return TXL_ERR_CUDA;
  unsigned int v = 0;
  if (cudaMemcpy(&v, p, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return TXL_ERR_CUDA;
  if (v != 0) {
    const unsigned int zero = 0;
    if (cudaMemcpy(p, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return TXL_ERR_CUDA;
  }
  if (v & txl::kStatusTimeoutBit) {
    // A kernel that gave up a wait may have left split-merge counters
    // counted: zero this device's scratch buffers (after the device is idle).
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) return TXL_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mutex);
    for (auto& kv : g_scratch)
      if (kv.first.first == dev && kv.second.cnt != nullptr &&
          cudaMemset(kv.second.cnt, 0, kv.second.cnt_n * sizeof(int)) != cudaSuccess)
        return TXL_ERR_CUDA;
    if (dev < kMaxDevices && g_static_ptr[dev] != nullptr &&
        cudaMemset(g_static_ptr[dev], 0, kStaticCounters * sizeof(int)) != cudaSuccess)
      return TXL_ERR_CUDA;
    return TXL_ERR_DEVICE_TIMEOUT;
  }
  return TXL_OK;
}

int txl_release_cached(void) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) return TXL_ERR_CUDA;
  int rc = TXL_OK;
  {
    std::lock_guard<std::mutex> lk(g_mutex);
    for (auto it = g_scratch.begin(); it != g_scratch.end();) {
      if (it->first.first != dev) {
        ++it;
        continue;
      }
      if ((it->second.ptr != nullptr && cudaFree(it->second.ptr) != cudaSuccess) ||
          (it->second.cnt != nullptr && cudaFree(it->second.cnt) != cudaSuccess))
        rc = TXL_ERR_CUDA;
      it = g_scratch.erase(it);
    }
    for (auto it = g_gather.begin(); it != g_gather.end();) {
      if (it->first.first != dev) {
        ++it;
        continue;
      }
      if (it->second.first != nullptr && cudaFree(it->second.first) != cudaSuccess) rc = TXL_ERR_CUDA;
      it = g_gather.erase(it);
    }
  }
  if (txl::release_plans(dev) != cudaSuccess) rc = TXL_ERR_CUDA;
  return rc;
}

int txl_sinusoid_rel(void* R, int n_dist, int dim, txl_dtype dtype, cudaStream_t stream) {
  if (n_dist < 0 || dim < 2 || (dim % 2) != 0 || !dtype_ok(dtype)) return TXL_ERR_INVALID_ARG;
  if (n_dist == 0) return TXL_OK;
  if (R == nullptr || !aligned(R, 2 * dsize(dtype))) return TXL_ERR_INVALID_ARG;
  if (n_dist > (1 << 24)) return TXL_ERR_UNSUPPORTED;  // distances must stay exact in fp32
  float c1, c2, c3;
  two_pi_split(n_dist, &c1, &c2, &c3);
  const double rho = std::pow(10000.0, -2.0 / static_cast<double>(dim));
  const float rho_hi = static_cast<float>(rho);
  const float rho_lo = static_cast<float>(rho - static_cast<double>(rho_hi));
  return from_cuda(
      txl::launch_sinusoid(R, n_dist, dim, dtype == TXL_BF16, rho_hi, rho_lo, c1, c2, c3, stream));
}

int txl_mem_update(const void* mem, int m_prev, const void* h, int w, void* mem_out, int m, int B, int C,
                   long long mem_bs, long long h_bs, long long out_bs, int* m_out, txl_dtype dtype,
                   cudaStream_t stream) {
  const txl::RollTensor t{mem, h, mem_out};
  return roll_impl(&t, 1, m_prev, w, m, B, C, mem_bs, h_bs, out_bs, m_out, dtype, stream);
}

int txl_mem_update_kv(const void* k_mem, const void* v_mem, int m_prev, const void* k_h, const void* v_h, int w,
                      void* k_out, void* v_out, int m, int B, int C, long long mem_bs, long long h_bs,
                      long long out_bs, int* m_out, txl_dtype dtype, cudaStream_t stream) {
  const txl::RollTensor t[2] = {{k_mem, k_h, k_out}, {v_mem, v_h, v_out}};
  return roll_impl(t, 2, m_prev, w, m, B, C, mem_bs, h_bs, out_bs, m_out, dtype, stream);
}

}  // extern "C"

namespace {

// Memory roll done by the attention kernel itself: the kept rows
// [src0, M+W) of k and v go to k_out / v_out (batch stride out_bs elements).
struct FusedRoll {
  void* k_out;
  void* v_out;
  long long keep, src0, out_bs;
};

// Keys and values of a ring-buffer call: k and v passed to forward_impl are
// then the rings [B, cap, H, D]; the segment rows come from k_seg, v_seg.
struct RingArgs {
  const void* k_seg;
  const void* v_seg;
  int cap, start;
  bool append;  // the kernel also writes the segment's rows into the ring
};

// The attention (validated arguments); `roll` non-null asks the bf16
// tensor-core kernel to write the memory roll too (the caller has checked
// it can).
int forward_impl(const void* q, const void* k, const void* v, const void* r, const float* bias_u,
                 const float* bias_v, void* o, float* lse, int B, int W, int M, int H, int D, int n_r, float scale,
                 txl_dtype dtype, txl_dtype o_dtype, const FusedRoll* roll, bool static_scratch_only,
                 cudaStream_t stream, const RingArgs* ring = nullptr);

// Shapes and dtypes the forward kernels take (TXL_OK or TXL_ERR_UNSUPPORTED).
int shape_support(int B, int W, int M, int H, int D, txl_dtype dtype, txl_dtype o_dtype) {
  const long long L = static_cast<long long>(M) + W;
  if (dtype == TXL_F32) {
    if (o_dtype != TXL_F32 || D > 256 || B > 65535 || H > 65535) return TXL_ERR_UNSUPPORTED;
    if (sizeof(float) * (2 * static_cast<size_t>(D) + L) > 220 * 1024) return TXL_ERR_UNSUPPORTED;
  } else {
    if (D != 64 && D != 128) return TXL_ERR_UNSUPPORTED;
    const long long nqt = (W + 127) / 128;
    if (nqt * B * H > 0x7FFFFFFFLL || L > 0x7FFFFFFFLL) return TXL_ERR_UNSUPPORTED;
  }
  return TXL_OK;
}

int check_forward(const void* q, const void* k, const void* v, const void* r, const float* bias_u,
                  const float* bias_v, void* o, float* lse, int B, int W, int M, int H, int D, int n_r, float scale,
                  txl_dtype dtype, txl_dtype o_dtype) {
  if (B < 0 || W < 0 || M < 0 || H <= 0 || D <= 0 || !dtype_ok(dtype) || !dtype_ok(o_dtype))
    return TXL_ERR_INVALID_ARG;
  if (B == 0 || W == 0) return TXL_OK;
  if (q == nullptr || k == nullptr || v == nullptr || r == nullptr || bias_u == nullptr || bias_v == nullptr ||
      o == nullptr)
    return TXL_ERR_INVALID_ARG;
  if (static_cast<long long>(n_r) < static_cast<long long>(M) + W) return TXL_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return TXL_ERR_INVALID_ARG;
  const size_t in_align = (dtype == TXL_BF16) ? 16 : 4;
  if (!aligned(q, in_align) || !aligned(k, in_align) || !aligned(v, in_align) || !aligned(r, in_align) ||
      !aligned(o, 16) || !aligned(bias_u, 4) || !aligned(bias_v, 4) || (lse != nullptr && !aligned(lse, 4)))
    return TXL_ERR_INVALID_ARG;

  const long long L = static_cast<long long>(M) + W;
  const size_t es = dsize(dtype);
  const size_t hd = static_cast<size_t>(H) * D;
  const Range rq = range_of(q, B * static_cast<size_t>(W) * hd * es);
  const Range rk = range_of(k, B * static_cast<size_t>(L) * hd * es);
  const Range rv = range_of(v, B * static_cast<size_t>(L) * hd * es);
  const Range rr = range_of(r, static_cast<size_t>(n_r) * hd * es);
  const Range ru = range_of(bias_u, hd * 4);
  const Range rb = range_of(bias_v, hd * 4);
  const Range ro = range_of(o, B * static_cast<size_t>(W) * hd * dsize(o_dtype));
  for (Range x : {rq, rk, rv, rr, ru, rb})
    if (overlap(ro, x)) return TXL_ERR_ALIAS;
  if (lse != nullptr) {
    const Range rl = range_of(lse, B * static_cast<size_t>(H) * W * 4);
    for (Range x : {rq, rk, rv, rr, ru, rb, ro})
      if (overlap(rl, x)) return TXL_ERR_ALIAS;
  }
  return shape_support(B, W, M, H, D, dtype, o_dtype);
}

int forward_impl(const void* q, const void* k, const void* v, const void* r, const float* bias_u,
                 const float* bias_v, void* o, float* lse, int B, int W, int M, int H, int D, int n_r, float scale,
                 txl_dtype dtype, txl_dtype o_dtype, const FusedRoll* roll, bool static_scratch_only,
                 cudaStream_t stream, const RingArgs* ring) {
  const long long L = static_cast<long long>(M) + W;
  const size_t hd = static_cast<size_t>(H) * D;
  if (ring != nullptr && (dtype != TXL_BF16 || D != 64)) return TXL_ERR_UNSUPPORTED;
  if (dtype == TXL_F32) {
    return from_cuda(txl::launch_relattn_f32(
        static_cast<const float*>(q), static_cast<const float*>(k), static_cast<const float*>(v),
        static_cast<const float*>(r), bias_u, bias_v, static_cast<float*>(o), lse, B, W, M, H, D, scale,
        stream));
  }

  // bf16 tensor-core path
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (encode == nullptr) return TXL_ERR_CUDA;
  CUtensorMap tm_q, tm_k, tm_v, tm_r;
  auto encode_bf16 = [&](CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
                         const cuuint64_t* strides, const cuuint32_t* box) {
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  };
  {
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                                static_cast<cuuint64_t>(W), static_cast<cuuint64_t>(B)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2, hd * 2, static_cast<cuuint64_t>(W) * hd * 2};
    const cuuint32_t box[4] = {64, 1, 128, 1};
    if (!encode_bf16(&tm_q, q, 4, dims, strides, box)) return TXL_ERR_CUDA;
  }
  {
    // k, v rows: L per sequence, or the ring's cap
    const long long rows = ring != nullptr ? ring->cap : L;
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                                static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(B)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2, hd * 2,
                                   static_cast<cuuint64_t>(rows) * hd * 2};
    const cuuint32_t box[4] = {64, 1, 64, 1};
    if (!encode_bf16(&tm_k, k, 4, dims, strides, box) || !encode_bf16(&tm_v, v, 4, dims, strides, box))
      return TXL_ERR_CUDA;
  }
  txl::RingMaps ring_maps;
  if (ring != nullptr) {
    if (D != 64 || roll != nullptr) return TXL_ERR_UNSUPPORTED;
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                                static_cast<cuuint64_t>(W), static_cast<cuuint64_t>(B)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2, hd * 2, static_cast<cuuint64_t>(W) * hd * 2};
    const cuuint32_t box[4] = {64, 1, 64, 1};
    if (!encode_bf16(&ring_maps.tm_ks, ring->k_seg, 4, dims, strides, box) ||
        !encode_bf16(&ring_maps.tm_vs, ring->v_seg, 4, dims, strides, box))
      return TXL_ERR_CUDA;
    ring_maps.cap = ring->cap;
    ring_maps.start = ring->start;
    ring_maps.append = ring->append;
  }
  {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                                static_cast<cuuint64_t>(n_r)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, hd * 2};
    const cuuint32_t box[3] = {64, 1, 64};
    if (!encode_bf16(&tm_r, r, 3, dims, strides, box)) return TXL_ERR_CUDA;
  }
  // bf16 output of the D = 64 kernel leaves through TMA stores of 32-row boxes.
  CUtensorMap tm_o;
  const bool o_tma = D == 64 && o_dtype == TXL_BF16;
  if (o_tma) {
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                                static_cast<cuuint64_t>(W), static_cast<cuuint64_t>(B)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2, hd * 2, static_cast<cuuint64_t>(W) * hd * 2};
    const cuuint32_t box[4] = {64, 1, 32, 1};
    if (!encode_bf16(&tm_o, o, 4, dims, strides, box)) return TXL_ERR_CUDA;
  }
  // Memory-roll outputs: [B, keep, H, D] with batch stride out_bs, stored
  // from the kernel's 64-row key and value tiles.
  CUtensorMap tm_km, tm_vm;
  if (roll != nullptr) {
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                                static_cast<cuuint64_t>(roll->keep), static_cast<cuuint64_t>(B)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2, hd * 2,
                                   static_cast<cuuint64_t>(roll->out_bs) * 2};
    const cuuint32_t box[4] = {64, 1, 64, 1};
    if (!encode_bf16(&tm_km, roll->k_out, 4, dims, strides, box) ||
        !encode_bf16(&tm_vm, roll->v_out, 4, dims, strides, box))
      return TXL_ERR_CUDA;
  }
  txl::WaitCtl wc;
  if (status_ptr(&wc.status) != cudaSuccess) return TXL_ERR_CUDA;
  wc.limit_ns = g_wait_ns.load();
  wc.inject_stall = g_inject_stall.exchange(0);
  if (D == 64) {
    // Too few units to fill the SMs: split each unit's key steps into
    // chunks; the last chunk of each unit merges their partial results.
    int nsplit = txl::relattn_tc64_split(B, H, W, M);
    if (const int f = g_force_split.load(); f > 0) {
      // never more chunks than the shortest unit has key steps
      const int nks_min = (std::min(M + 127, M + W - 1)) / 64 + 1;
      nsplit = std::min(f, nks_min);
    }
    float* part_o = nullptr;
    float* part_lse = nullptr;
    int* part_cnt = nullptr;
    if (nsplit > 1) {
      const size_t units = static_cast<size_t>((W + 127) / 128) * B * H;
      const size_t rows = units * nsplit * 128;
      const size_t part_bytes = rows * (D + 1) * sizeof(float);
      if (static_scratch_only) {
        if (units * 4 > kStaticCounters || kStaticCounters * sizeof(int) + part_bytes > kStaticScratchBytes)
          return TXL_ERR_UNSUPPORTED;
        unsigned char* base = nullptr;
        if (static_scratch(&base) != cudaSuccess) return TXL_ERR_CUDA;
        part_cnt = reinterpret_cast<int*>(base);
        part_o = reinterpret_cast<float*>(base + kStaticCounters * sizeof(int));
      } else {
        void* buf = nullptr;
        if (split_scratch(stream, part_bytes, units * 4, &buf, &part_cnt) != cudaSuccess) return TXL_ERR_CUDA;
        part_o = static_cast<float*>(buf);
      }
      part_lse = part_o + rows * D;
    }
    return from_cuda(txl::launch_relattn_tc64(tm_q, tm_k, tm_v, tm_r, o_tma ? &tm_o : nullptr,
                                              roll ? &tm_km : nullptr, roll ? &tm_vm : nullptr,
                                              roll ? static_cast<int>(roll->src0) : -1,
                                              ring != nullptr ? &ring_maps : nullptr, bias_u, bias_v, o, lse, B,
                                              W, M, H, o_dtype == TXL_BF16, scale, nsplit, part_o, part_lse,
                                              part_cnt, !static_scratch_only, wc, stream));
  }
  return from_cuda(txl::launch_relattn_tc(tm_q, tm_k, tm_v, tm_r, roll ? &tm_km : nullptr, roll ? &tm_vm : nullptr,
                                          roll ? static_cast<int>(roll->src0) : -1, bias_u, bias_v, o, lse, B, W,
                                          M, H, D, o_dtype == TXL_BF16, scale, !static_scratch_only, wc, stream));
}

}  // namespace

extern "C" {

int txl_relattn_backward(const void* q, const void* k, const void* v, const void* r, const float* bias_u,
                         const float* bias_v, const void* o, const float* lse, const void* dout, float* dq,
                         float* dk, float* dv, float* dr, float* dbias_u, float* dbias_v, int B, int W, int M,
                         int H, int D, int n_r, float scale, txl_dtype dtype, txl_dtype go_dtype,
                         cudaStream_t stream) {
  if (B < 0 || W < 0 || M < 0 || H <= 0 || D <= 0 || !dtype_ok(dtype) || !dtype_ok(go_dtype))
    return TXL_ERR_INVALID_ARG;
  if (B == 0 || W == 0) return TXL_OK;
  const void* ins[] = {q, k, v, r, bias_u, bias_v, o, lse, dout};
  const void* outs[] = {dq, dk, dv, dr, dbias_u, dbias_v};
  for (const void* p : ins)
    if (p == nullptr || !aligned(p, 16)) return TXL_ERR_INVALID_ARG;
  for (const void* p : outs)
    if (p == nullptr || !aligned(p, 16)) return TXL_ERR_INVALID_ARG;
  if (static_cast<long long>(n_r) < static_cast<long long>(M) + W || !std::isfinite(scale))
    return TXL_ERR_INVALID_ARG;
  if (D > 256 || B > 65535 || H > 65535) return TXL_ERR_UNSUPPORTED;
  const long long L = static_cast<long long>(M) + W;
  if (L > 0x7FFFFFFFLL) return TXL_ERR_UNSUPPORTED;
  const size_t es = dsize(dtype), gs = dsize(go_dtype);
  const size_t hd = static_cast<size_t>(H) * D, bw = static_cast<size_t>(B) * W;
  const Range in_r[] = {range_of(q, bw * hd * es),
                        range_of(k, B * static_cast<size_t>(L) * hd * es),
                        range_of(v, B * static_cast<size_t>(L) * hd * es),
                        range_of(r, static_cast<size_t>(n_r) * hd * es),
                        range_of(bias_u, hd * 4),
                        range_of(bias_v, hd * 4),
                        range_of(o, bw * hd * gs),
                        range_of(lse, bw * H * 4),
                        range_of(dout, bw * hd * gs)};
  const Range out_r[] = {range_of(dq, bw * hd * 4), range_of(dk, bw * hd * 4), range_of(dv, bw * hd * 4),
                         range_of(dr, static_cast<size_t>(n_r) * hd * 4), range_of(dbias_u, hd * 4),
                         range_of(dbias_v, hd * 4)};
  for (size_t x = 0; x < 6; ++x) {
    for (const Range& y : in_r)
      if (overlap(out_r[x], y)) return TXL_ERR_ALIAS;
    for (size_t z = x + 1; z < 6; ++z)
      if (overlap(out_r[x], out_r[z])) return TXL_ERR_ALIAS;
  }
  void* scratch = nullptr;
  int* unused = nullptr;
  // bf16 on the tensor cores: the materialised pair terms (D = 64 or 128);
  // the test hook can send D = 64 to the fused kernels
  const bool tc = dtype == TXL_BF16 && go_dtype == TXL_BF16;
  const bool pairs = tc && txl::relattn_bwd_pairs_supported(W, M, D) && !(D == 64 && g_bwd_path.load() == 1);
  if (tc && D == 64 && !pairs) {
    // tensor-core path, fused
    if (split_scratch(stream, txl::relattn_bwd_tc64_scratch_bytes(B, W, H), 0, &scratch, &unused) != cudaSuccess)
      return TXL_ERR_CUDA;
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (encode == nullptr) return TXL_ERR_CUDA;
    auto encode_bf16 = [&](CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
                           const cuuint64_t* strides, const cuuint32_t* box) {
      const cuuint32_t estr[4] = {1, 1, 1, 1};
      return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    };
    CUtensorMap tm_q, tm_do, tm_k, tm_v, tm_rw;
    {
      const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                                  static_cast<cuuint64_t>(W), static_cast<cuuint64_t>(B)};
      const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2, hd * 2, static_cast<cuuint64_t>(W) * hd * 2};
      const cuuint32_t box[4] = {64, 1, 128, 1};
      if (!encode_bf16(&tm_q, q, 4, dims, strides, box) || !encode_bf16(&tm_do, dout, 4, dims, strides, box))
        return TXL_ERR_CUDA;
    }
    {
      const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                                  static_cast<cuuint64_t>(L), static_cast<cuuint64_t>(B)};
      const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2, hd * 2, static_cast<cuuint64_t>(L) * hd * 2};
      const cuuint32_t box[4] = {64, 1, 64, 1};
      if (!encode_bf16(&tm_k, k, 4, dims, strides, box) || !encode_bf16(&tm_v, v, 4, dims, strides, box))
        return TXL_ERR_CUDA;
    }
    {
      const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                                  static_cast<cuuint64_t>(n_r)};
      const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, hd * 2};
      const cuuint32_t box[3] = {64, 1, 192};
      if (!encode_bf16(&tm_rw, r, 3, dims, strides, box)) return TXL_ERR_CUDA;
    }
    CUtensorMap tm_dr;  // fp32 [n_r, H, D]: boxes of 64 distances x 32 dims of one head, for the TMA reductions
    {
      const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                                  static_cast<cuuint64_t>(n_r)};
      const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 4, hd * 4};
      const cuuint32_t box[3] = {32, 1, 64};
      const cuuint32_t estr[3] = {1, 1, 1};
      if (encode(&tm_dr, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, dr, dims, strides, box, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return TXL_ERR_CUDA;
    }
    txl::WaitCtl wc;
    if (status_ptr(&wc.status) != cudaSuccess) return TXL_ERR_CUDA;
    wc.limit_ns = g_wait_ns.load();
    wc.inject_stall = g_inject_stall.exchange(0);
    const long long nqt = (W + 127) / 128;
    if (nqt * B * H > 0x7FFFFFFFLL) return TXL_ERR_UNSUPPORTED;
    return from_cuda(txl::launch_relattn_bwd_tc64(tm_q, tm_k, tm_v, tm_rw, tm_do, tm_dr, bias_u, bias_v, lse, o,
                                                  dout, dq,
                                                  dk, dv, dr, dbias_u, dbias_v, B, W, M, H, n_r, scale, scratch, wc,
                                                  stream));
  }
  if (pairs) {
    // tensor-core path, pair terms materialised
    if (split_scratch(stream, txl::relattn_bwd_pairs_scratch_bytes(B, W, M, H, D), 0, &scratch, &unused) !=
        cudaSuccess)
      return TXL_ERR_CUDA;
    txl::WaitCtl wc;
    if (status_ptr(&wc.status) != cudaSuccess) return TXL_ERR_CUDA;
    wc.limit_ns = g_wait_ns.load();
    wc.inject_stall = g_inject_stall.exchange(0);
    if ((W + 127) / 128 * static_cast<long long>(B) * H > 0x7FFFFFFFLL) return TXL_ERR_UNSUPPORTED;
    return from_cuda(txl::launch_relattn_bwd_pairs(tensor_map_encoder(), q, k, v, r, bias_u, bias_v, lse, o, dout,
                                                   dq, dk, dv, dr, dbias_u, dbias_v, B, W, M, H, D, n_r, scale,
                                                   scratch, wc, stream));
  }
  if (split_scratch(stream, txl::relattn_bwd_simt_scratch_bytes(B, W, H, D), 0, &scratch, &unused) != cudaSuccess)
    return TXL_ERR_CUDA;
  const bool vec16 = (D * es) % 16 == 0;  // with 16-byte aligned bases, every row is then aligned
  return from_cuda(txl::launch_relattn_bwd_simt(q, k, v, r, bias_u, bias_v, o, lse, dout, dq, dk, dv, dr, dbias_u,
                                                dbias_v, B, W, M, H, D, n_r, scale, dtype == TXL_BF16,
                                                go_dtype == TXL_BF16, vec16, scratch, stream));
}

int txl_relattn_forward(const void* q, const void* k, const void* v, const void* r, const float* bias_u,
                        const float* bias_v, void* o, float* lse, int B, int W, int M, int H, int D, int n_r,
                        float scale, txl_dtype dtype, txl_dtype o_dtype, cudaStream_t stream) {
  const int st = check_forward(q, k, v, r, bias_u, bias_v, o, lse, B, W, M, H, D, n_r, scale, dtype, o_dtype);
  if (st != TXL_OK || B == 0 || W == 0) return st;
  return forward_impl(q, k, v, r, bias_u, bias_v, o, lse, B, W, M, H, D, n_r, scale, dtype, o_dtype, nullptr,
                      false, stream);
}

int txl_relattn_forward_static(const void* q, const void* k, const void* v, const void* r, const float* bias_u,
                               const float* bias_v, void* o, float* lse, int B, int W, int M, int H, int D, int n_r,
                               float scale, txl_dtype dtype, txl_dtype o_dtype, cudaStream_t stream) {
  const int st = check_forward(q, k, v, r, bias_u, bias_v, o, lse, B, W, M, H, D, n_r, scale, dtype, o_dtype);
  if (st != TXL_OK || B == 0 || W == 0) return st;
  return forward_impl(q, k, v, r, bias_u, bias_v, o, lse, B, W, M, H, D, n_r, scale, dtype, o_dtype, nullptr,
                      true, stream);
}

int txl_relattn_forward_roll(const void* q, const void* k, const void* v, const void* r, const float* bias_u,
                             const float* bias_v, void* o, float* lse, int B, int W, int M, int H, int D, int n_r,
                             float scale, txl_dtype dtype, txl_dtype o_dtype, void* k_mem_out, void* v_mem_out,
                             int m, long long mem_out_bs, int* m_out, cudaStream_t stream) {
  const int st = check_forward(q, k, v, r, bias_u, bias_v, o, lse, B, W, M, H, D, n_r, scale, dtype, o_dtype);
  if (st != TXL_OK) return st;
  if (m < 0) return TXL_ERR_INVALID_ARG;
  const long long L = static_cast<long long>(M) + W;
  const long long keep = std::min<long long>(m, L);
  const long long C = static_cast<long long>(H) * D;
  if (B == 0 || W == 0) {
    if (m_out != nullptr) *m_out = static_cast<int>(keep);
    return TXL_OK;
  }
  if (keep > 0) {
    if (k_mem_out == nullptr || v_mem_out == nullptr || mem_out_bs < 0) return TXL_ERR_INVALID_ARG;
    if (B > 1 && mem_out_bs < keep * C) return TXL_ERR_INVALID_ARG;
    // Roll outputs against each other and against everything the attention touches.
    const size_t es = dsize(dtype);
    const size_t out_bytes = static_cast<size_t>(((B - 1) * mem_out_bs + keep * C) * static_cast<long long>(es));
    const Range rkm = range_of(k_mem_out, out_bytes), rvm = range_of(v_mem_out, out_bytes);
    if (overlap(rkm, rvm)) return TXL_ERR_ALIAS;
    const size_t hd = static_cast<size_t>(C);
    const Range others[] = {range_of(q, B * static_cast<size_t>(W) * hd * es),
                            range_of(k, B * static_cast<size_t>(L) * hd * es),
                            range_of(v, B * static_cast<size_t>(L) * hd * es),
                            range_of(r, static_cast<size_t>(n_r) * hd * es),
                            range_of(bias_u, hd * 4),
                            range_of(bias_v, hd * 4),
                            range_of(o, B * static_cast<size_t>(W) * hd * dsize(o_dtype)),
                            range_of(lse, lse ? B * static_cast<size_t>(H) * W * 4 : 0)};
    for (const Range& x : others)
      if (overlap(rkm, x) || overlap(rvm, x)) return TXL_ERR_ALIAS;
  }
  if (m_out != nullptr) *m_out = static_cast<int>(keep);
  // Fused when the kept rows start on a 64-row key tile of the bf16 tensor-core kernels.
  const bool fused = keep > 0 && dtype == TXL_BF16 && (D == 64 || D == 128) && (L - keep) % 64 == 0 &&
                     aligned(k_mem_out, 16) && aligned(v_mem_out, 16) && (mem_out_bs * 2) % 16 == 0 &&
                     keep <= 0x7FFFFFFFLL;
  if (fused) {
    const FusedRoll fr{k_mem_out, v_mem_out, keep, L - keep, mem_out_bs};
    return forward_impl(q, k, v, r, bias_u, bias_v, o, lse, B, W, M, H, D, n_r, scale, dtype, o_dtype, &fr,
                        false, stream);
  }
  int rc = forward_impl(q, k, v, r, bias_u, bias_v, o, lse, B, W, M, H, D, n_r, scale, dtype, o_dtype, nullptr,
                        false, stream);
  if (rc != TXL_OK || keep == 0) return rc;
  const long long bs = L * C;
  const size_t es = dsize(dtype);
  const char* kb = static_cast<const char*>(k);
  const char* vb = static_cast<const char*>(v);
  return txl_mem_update_kv(kb, vb, M, kb + static_cast<size_t>(M) * C * es, vb + static_cast<size_t>(M) * C * es, W,
                           k_mem_out, v_mem_out, m, B, static_cast<int>(C), bs, bs, mem_out_bs, nullptr, dtype,
                           stream);
}

int txl_mem_ring_append(void* mem, int cap, int start, int m, const void* h, int w, int B, int C, long long h_bs,
                        int* start_out, int* m_out, txl_dtype dtype, cudaStream_t stream) {
  void* const mems[1] = {mem};
  const void* const hs[1] = {h};
  return ring_append_impl(mems, hs, 1, cap, start, m, w, B, C, h_bs, start_out, m_out, dtype, stream);
}

}  // extern "C"

namespace {
// [memory in ring order ; segment] into contiguous scratch, then the
// ordinary call.
int linear_ring_forward(const void* q, const void* k_mem, const void* v_mem, int cap, int start, int M,
                        const void* k_seg, const void* v_seg, const void* r, const float* bias_u, const float* bias_v,
                        void* o, float* lse, int B, int W, int H, int D, int n_r, float scale, txl_dtype dtype,
                        txl_dtype o_dtype, cudaStream_t stream) {
  if (B > 65535) return TXL_ERR_UNSUPPORTED;
  const size_t es = dsize(dtype), hd = static_cast<size_t>(H) * D;
  const long long L = static_cast<long long>(M) + W;
  const long long row_bytes = static_cast<long long>(hd * es);
  void* buf = nullptr;
  if (gather_scratch(stream, 2 * static_cast<size_t>(B) * L * row_bytes, &buf) != cudaSuccess) return TXL_ERR_CUDA;
  char* lin[2] = {static_cast<char*>(buf), static_cast<char*>(buf) + static_cast<size_t>(B) * L * row_bytes};
  const void* mem[2] = {k_mem, v_mem};
  const void* seg[2] = {k_seg, v_seg};
  const long long n1 = M > 0 ? std::min<long long>(M, cap - start) : 0;  // rows before the ring wraps
  for (int x = 0; x < 2; ++x) {
    if (n1 > 0 &&
        txl::launch_mem_roll(mem[x], nullptr, lin[x], B, n1, n1, start, 0, row_bytes, cap * row_bytes, 0,
                             L * row_bytes, stream) != cudaSuccess)
      return TXL_ERR_CUDA;
    if (txl::launch_mem_roll(mem[x], seg[x], lin[x] + n1 * row_bytes, B, L - n1, M - n1, 0, 0, row_bytes,
                             cap * row_bytes, W * row_bytes, L * row_bytes, stream) != cudaSuccess)
      return TXL_ERR_CUDA;
  }
  return forward_impl(q, lin[0], lin[1], r, bias_u, bias_v, o, lse, B, W, M, H, D, n_r, scale, dtype, o_dtype,
                      nullptr, false, stream);
}


int ring_impl(const void* q, const void* k_mem, const void* v_mem, int cap, int start, int M, const void* k_seg,
              const void* v_seg, const void* r, const float* bias_u, const float* bias_v, void* o, float* lse, int B,
              int W, int H, int D, int n_r, float scale, txl_dtype dtype, txl_dtype o_dtype, bool append,
              int* start_out, int* m_out, cudaStream_t stream) {
  if (B < 0 || W < 0 || M < 0 || H <= 0 || D <= 0 || cap < M || !dtype_ok(dtype) || !dtype_ok(o_dtype))
    return TXL_ERR_INVALID_ARG;
  if (M > 0 && (start < 0 || start >= cap)) return TXL_ERR_INVALID_ARG;
  if (append && (cap <= 0 || k_mem == nullptr || v_mem == nullptr)) return TXL_ERR_INVALID_ARG;
  if (M == 0) start = 0;
  if (append) {  // the ring after the call: the last min(cap, M + W) rows of [memory ; segment]
    const long long total = static_cast<long long>(M) + W;
    if (start_out != nullptr) *start_out = static_cast<int>((start + (total > cap ? total - cap : 0)) % cap);
    if (m_out != nullptr) *m_out = static_cast<int>(std::min<long long>(total, cap));
  }
  if (B == 0 || W == 0) return TXL_OK;
  if (q == nullptr || k_seg == nullptr || v_seg == nullptr || r == nullptr || bias_u == nullptr ||
      bias_v == nullptr || o == nullptr || (M > 0 && (k_mem == nullptr || v_mem == nullptr)))
    return TXL_ERR_INVALID_ARG;
  if (static_cast<long long>(n_r) < static_cast<long long>(M) + W || !std::isfinite(scale))
    return TXL_ERR_INVALID_ARG;
  const size_t in_align = (dtype == TXL_BF16) ? 16 : 4;
  for (const void* x : {q, k_seg, v_seg, r})
    if (!aligned(x, in_align)) return TXL_ERR_INVALID_ARG;
  if (M > 0 && (!aligned(k_mem, in_align) || !aligned(v_mem, in_align))) return TXL_ERR_INVALID_ARG;
  if (!aligned(o, 16) || !aligned(bias_u, 4) || !aligned(bias_v, 4) || (lse != nullptr && !aligned(lse, 4)))
    return TXL_ERR_INVALID_ARG;
  const size_t es = dsize(dtype), hd = static_cast<size_t>(H) * D, bw = static_cast<size_t>(B) * W;
  std::vector<Range> ins = {range_of(q, bw * hd * es), range_of(k_seg, bw * hd * es), range_of(v_seg, bw * hd * es),
                            range_of(r, static_cast<size_t>(n_r) * hd * es), range_of(bias_u, hd * 4),
                            range_of(bias_v, hd * 4)};
  if (M > 0 || append) {
    ins.push_back(range_of(k_mem, static_cast<size_t>(B) * cap * hd * es));
    ins.push_back(range_of(v_mem, static_cast<size_t>(B) * cap * hd * es));
  }
  if (append) {  // the rings are written: they must not overlap the segment rows or each other
    const Range rk = range_of(k_mem, static_cast<size_t>(B) * cap * hd * es);
    const Range rv = range_of(v_mem, static_cast<size_t>(B) * cap * hd * es);
    if (overlap(rk, rv)) return TXL_ERR_ALIAS;
    for (size_t x = 0; x < 6; ++x)
      if (overlap(rk, ins[x]) || overlap(rv, ins[x])) return TXL_ERR_ALIAS;
  }
  const Range ro = range_of(o, bw * hd * dsize(o_dtype));
  for (const Range& x : ins)
    if (overlap(ro, x)) return TXL_ERR_ALIAS;
  if (lse != nullptr) {
    const Range rl = range_of(lse, bw * H * 4);
    if (overlap(rl, ro)) return TXL_ERR_ALIAS;
    for (const Range& x : ins)
      if (overlap(rl, x)) return TXL_ERR_ALIAS;
  }
  const int sup = shape_support(B, W, M, H, D, dtype, o_dtype);
  if (sup != TXL_OK) return sup;
  const bool in_place = dtype == TXL_BF16 && D == 64 && M % 64 == 0 && cap % 64 == 0 && start % 64 == 0;
  if (append && in_place && W % 64 == 0 && static_cast<long long>(M) + W <= cap) {
    // one launch: the kernel reads the ring in place and stores the
    // segment's rows into ring slots the memory does not use
    const RingArgs ra{k_seg, v_seg, cap, start, true};
    return forward_impl(q, k_mem, v_mem, r, bias_u, bias_v, o, lse, B, W, M, H, D, n_r, scale, dtype, o_dtype,
                        nullptr, false, stream, &ra);
  }
  int st = TXL_OK;
  if (M == 0) {  // no memory: the segment alone
    st = forward_impl(q, k_seg, v_seg, r, bias_u, bias_v, o, lse, B, W, 0, H, D, n_r, scale, dtype, o_dtype, nullptr,
                      false, stream);
  } else if (in_place) {  // the kernel reads the ring in place
    const RingArgs ra{k_seg, v_seg, cap, start, false};
    st = forward_impl(q, k_mem, v_mem, r, bias_u, bias_v, o, lse, B, W, M, H, D, n_r, scale, dtype, o_dtype,
                      nullptr, false, stream, &ra);
  } else {
    st = linear_ring_forward(q, k_mem, v_mem, cap, start, M, k_seg, v_seg, r, bias_u, bias_v, o, lse, B, W, H, D,
                             n_r, scale, dtype, o_dtype, stream);
  }
  if (st != TXL_OK || !append) return st;
  // then the segment's rows into the rings (after the attention, in stream order), keys and values in one launch
  const int C = H * D;
  void* const mems[2] = {const_cast<void*>(k_mem), const_cast<void*>(v_mem)};
  const void* const segs[2] = {k_seg, v_seg};
  return ring_append_impl(mems, segs, 2, cap, start, M, W, B, C, static_cast<long long>(W) * C, nullptr, nullptr,
                          dtype, stream);
}


}  // namespace

extern "C" {

int txl_relattn_forward_ring(const void* q, const void* k_mem, const void* v_mem, int cap, int start, int M,
                             const void* k_seg, const void* v_seg, const void* r, const float* bias_u,
                             const float* bias_v, void* o, float* lse, int B, int W, int H, int D, int n_r,
                             float scale, txl_dtype dtype, txl_dtype o_dtype, cudaStream_t stream) {
  return ring_impl(q, k_mem, v_mem, cap, start, M, k_seg, v_seg, r, bias_u, bias_v, o, lse, B, W, H, D, n_r, scale,
                   dtype, o_dtype, false, nullptr, nullptr, stream);
}

int txl_relattn_forward_ring_append(void* k_mem, void* v_mem, int cap, int start, int M, const void* q,
                                    const void* k_seg, const void* v_seg, const void* r, const float* bias_u,
                                    const float* bias_v, void* o, float* lse, int B, int W, int H, int D, int n_r,
                                    float scale, txl_dtype dtype, txl_dtype o_dtype, int* start_out, int* m_out,
                                    cudaStream_t stream) {
  return ring_impl(q, k_mem, v_mem, cap, start, M, k_seg, v_seg, r, bias_u, bias_v, o, lse, B, W, H, D, n_r, scale,
                   dtype, o_dtype, true, start_out, m_out, stream);
}

namespace {
size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
}  // namespace

int txl_dense(const void* x, const void* W, void* y, int m, int n, int k, int batch, long long w_batch_stride,
              long long y_batch_stride, const float* bias, int relu, cudaStream_t stream) {
  if (m < 0 || n <= 0 || k <= 0 || batch <= 0) return TXL_ERR_INVALID_ARG;
  if (m == 0) return TXL_OK;
  if (x == nullptr || W == nullptr || y == nullptr) return TXL_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(W, 16) || !aligned(y, 16) || (bias != nullptr && !aligned(bias, 4)))
    return TXL_ERR_INVALID_ARG;
  if (n % 8 != 0 || k % 8 != 0) return TXL_ERR_UNSUPPORTED;
  const long long wsz = static_cast<long long>(k) * n, ysz = static_cast<long long>(m) * n;
  if (batch > 1 && (w_batch_stride < wsz || y_batch_stride < ysz || w_batch_stride % 8 != 0 ||
                    y_batch_stride % 8 != 0))
    return TXL_ERR_INVALID_ARG;
  if (batch == 1) w_batch_stride = wsz, y_batch_stride = ysz;
  const Range ry = range_of(y, static_cast<size_t>(((batch - 1) * y_batch_stride + ysz) * 2));
  if (overlap(ry, range_of(x, static_cast<size_t>(m) * k * 2)) ||
      overlap(ry, range_of(W, static_cast<size_t>(((batch - 1) * w_batch_stride + wsz) * 2))) ||
      (bias != nullptr && overlap(ry, range_of(bias, static_cast<size_t>(n) * 4))))
    return TXL_ERR_ALIAS;
  return dense_impl(x, W, y, m, n, k, batch, w_batch_stride, y_batch_stride, bias, relu != 0, stream);
}

size_t txl_layer_workspace_bytes(int B, int W, int d_model, int H, int D, int d_ff, int n_r) {
  if (B <= 0 || W <= 0 || d_model <= 0 || H <= 0 || D <= 0 || d_ff <= 0 || n_r <= 0) return 0;
  const size_t bw = static_cast<size_t>(B) * W, hd = static_cast<size_t>(H) * D;
  return 4 * align256(bw * hd * 2) + align256(static_cast<size_t>(n_r) * hd * 2) + 3 * align256(bw * d_model * 2) +
         align256(bw * d_ff * 2);
}

namespace {
// One layer (validated arguments; d_model, d_ff, H*D multiples of 8).
int layer_impl(const void* h, void* out, void* k_mem, void* v_mem, int cap, int start, int M,
               const txl_layer_weights* w, const void* R, int n_r, int B, int W, int d_model, int H, int D, int d_ff,
               float scale, void* workspace, int* start_out, int* m_out, cudaStream_t stream) {
  const size_t bw = static_cast<size_t>(B) * W, hd = static_cast<size_t>(H) * D;
  // workspace carve-up
  char* p = static_cast<char*>(workspace);
  auto take = [&](size_t bytes) {
    char* r = p;
    p += align256(bytes);
    return r;
  };
  void* q = take(bw * hd * 2);
  void* ks = take(bw * hd * 2);
  void* vs = take(bw * hd * 2);
  void* a = take(bw * hd * 2);
  void* r = take(static_cast<size_t>(n_r) * hd * 2);
  void* y = take(bw * d_model * 2);
  void* x = take(bw * d_model * 2);
  void* z = take(bw * d_model * 2);
  void* f = take(bw * d_ff * 2);
  const int rows = static_cast<int>(bw);
  const int HD = static_cast<int>(hd);
  // W_q, W_k, W_v packed back to back: the three projections as one batched GEMM
  const size_t wbytes = static_cast<size_t>(d_model) * hd * 2;
  const bool packed = static_cast<const char*>(w->W_k) == static_cast<const char*>(w->W_q) + wbytes &&
                      static_cast<const char*>(w->W_v) == static_cast<const char*>(w->W_k) + wbytes;
  const long long qkv_stride = static_cast<long long>((static_cast<char*>(ks) - static_cast<char*>(q)) / 2);
  const long long wsz = static_cast<long long>(d_model) * HD;
  int st = TXL_OK;
  if (packed) {
    // q, k, v and r = R W_r in one launch (r's tiles after the projections')
    st = dense_impl(h, w->W_q, q, rows, HD, d_model, 3, wsz, qkv_stride, nullptr, false, stream, R, w->W_r, r, n_r);
  } else {
    const void* wm[3] = {w->W_q, w->W_k, w->W_v};
    void* om[3] = {q, ks, vs};
    for (int i = 0; i < 3 && st == TXL_OK; ++i)
      st = dense_impl(h, wm[i], om[i], rows, HD, d_model, 1, wsz, 0, nullptr, false, stream);
    if (st == TXL_OK) st = dense_impl(R, w->W_r, r, n_r, HD, d_model, 1, wsz, 0, nullptr, false, stream);
  }
  if (st != TXL_OK) return st;
  if ((st = txl_relattn_forward_ring_append(k_mem, v_mem, cap, start, M, q, ks, vs, r, w->bias_u, w->bias_v, a,
                                            nullptr, B, W, H, D, n_r, scale, TXL_BF16, TXL_BF16, start_out, m_out,
                                            stream)) != TXL_OK)
    return st;
  if ((st = dense_impl(a, w->W_o, y, rows, d_model, HD, 1, wsz, 0, nullptr, false, stream)) != TXL_OK) return st;
  if (txl::launch_add_ln(h, y, nullptr, w->ln1_gamma, w->ln1_beta, x, rows, d_model, stream) != cudaSuccess)
    return TXL_ERR_CUDA;
  // b_1 + ReLU and b_2 in the GEMMs' epilogues, on the fp32 accumulators
  const long long w1sz = static_cast<long long>(d_model) * d_ff;
  if ((st = dense_impl(x, w->W_1, f, rows, d_ff, d_model, 1, w1sz, 0, w->b_1, true, stream)) != TXL_OK) return st;
  if ((st = dense_impl(f, w->W_2, z, rows, d_model, d_ff, 1, w1sz, 0, w->b_2, false, stream)) != TXL_OK) return st;
  if (txl::launch_add_ln(x, z, nullptr, w->ln2_gamma, w->ln2_beta, out, rows, d_model, stream) != cudaSuccess)
    return TXL_ERR_CUDA;
  return TXL_OK;
}

int check_layer(const void* h, void* out, const void* k_mem, const void* v_mem, int cap, int M,
                const txl_layer_weights* w, const void* R, int B, int W, int d_model, int H, int D, int d_ff) {
  if (w == nullptr || h == nullptr || out == nullptr || R == nullptr || B <= 0 || W <= 0 || d_model <= 0 || H <= 0 ||
      D <= 0 || d_ff <= 0 || M < 0 || cap < M || cap <= 0)
    return TXL_ERR_INVALID_ARG;
  const void* ptrs[] = {w->W_q, w->W_k, w->W_v, w->W_r, w->bias_u, w->bias_v, w->W_o, w->ln1_gamma, w->ln1_beta,
                        w->W_1, w->b_1, w->W_2, w->b_2, w->ln2_gamma, w->ln2_beta, k_mem, v_mem};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned(p, 16)) return TXL_ERR_INVALID_ARG;
  if (!aligned(h, 16) || !aligned(out, 16) || !aligned(R, 16)) return TXL_ERR_INVALID_ARG;
  if (d_model % 8 != 0 || d_model > 1024 || d_ff % 8 != 0) return TXL_ERR_UNSUPPORTED;
  const size_t bw = static_cast<size_t>(B) * W;
  if (overlap(range_of(out, bw * d_model * 2), range_of(h, bw * d_model * 2))) return TXL_ERR_ALIAS;
  return TXL_OK;
}
}  // namespace

int txl_layer_forward(const void* h, void* out, void* k_mem, void* v_mem, int cap, int start, int M,
                      const txl_layer_weights* w, const void* R, int n_r, int B, int W, int d_model, int H, int D,
                      int d_ff, float scale, void* workspace, size_t workspace_bytes, int* start_out, int* m_out,
                      cudaStream_t stream) {
  int st = check_layer(h, out, k_mem, v_mem, cap, M, w, R, B, W, d_model, H, D, d_ff);
  if (st != TXL_OK) return st;
  if (workspace == nullptr || !aligned(workspace, 256)) return TXL_ERR_INVALID_ARG;
  if (workspace_bytes < txl_layer_workspace_bytes(B, W, d_model, H, D, d_ff, n_r)) return TXL_ERR_INVALID_ARG;
  return layer_impl(h, out, k_mem, v_mem, cap, start, M, w, R, n_r, B, W, d_model, H, D, d_ff, scale, workspace,
                    start_out, m_out, stream);
}

size_t txl_stack_workspace_bytes(int B, int W, int d_model, int H, int D, int d_ff, int n_r) {
  const size_t lw = txl_layer_workspace_bytes(B, W, d_model, H, D, d_ff, n_r);
  if (lw == 0) return 0;
  return lw + 2 * align256(static_cast<size_t>(B) * W * d_model * 2);
}

int txl_stack_forward(const void* h, void* out, int n_layers, void* const* k_mem, void* const* v_mem, int cap,
                      int start, int M, const txl_layer_weights* w, const void* R, int n_r, int B, int W, int d_model,
                      int H, int D, int d_ff, float scale, void* workspace, size_t workspace_bytes, int* start_out,
                      int* m_out, cudaStream_t stream) {
  if (n_layers <= 0 || k_mem == nullptr || v_mem == nullptr || w == nullptr) return TXL_ERR_INVALID_ARG;
  for (int l = 0; l < n_layers; ++l) {
    const int st = check_layer(h, out, k_mem[l], v_mem[l], cap, M, &w[l], R, B, W, d_model, H, D, d_ff);
    if (st != TXL_OK) return st;
  }
  if (workspace == nullptr || !aligned(workspace, 256)) return TXL_ERR_INVALID_ARG;
  if (workspace_bytes < txl_stack_workspace_bytes(B, W, d_model, H, D, d_ff, n_r)) return TXL_ERR_INVALID_ARG;
  // every layer's rings are distinct from every other layer's
  const size_t ring_bytes = static_cast<size_t>(B) * cap * H * D * 2;
  for (int l = 0; l < n_layers; ++l)
    for (int j = l + 1; j < n_layers; ++j)
      if (overlap(range_of(k_mem[l], ring_bytes), range_of(k_mem[j], ring_bytes)) ||
          overlap(range_of(k_mem[l], ring_bytes), range_of(v_mem[j], ring_bytes)) ||
          overlap(range_of(v_mem[l], ring_bytes), range_of(k_mem[j], ring_bytes)) ||
          overlap(range_of(v_mem[l], ring_bytes), range_of(v_mem[j], ring_bytes)))
        return TXL_ERR_ALIAS;
  // layer outputs ping-pong between two buffers after the layer workspace; the last goes to out
  const size_t lw = txl_layer_workspace_bytes(B, W, d_model, H, D, d_ff, n_r);
  char* buf[2] = {static_cast<char*>(workspace) + lw,
                  static_cast<char*>(workspace) + lw + align256(static_cast<size_t>(B) * W * d_model * 2)};
  const void* x = h;
  for (int l = 0; l < n_layers; ++l) {
    void* y = l == n_layers - 1 ? out : buf[l & 1];
    const int st = layer_impl(x, y, k_mem[l], v_mem[l], cap, start, M, &w[l], R, n_r, B, W, d_model, H, D, d_ff,
                              scale, workspace, start_out, m_out, stream);
    if (st != TXL_OK) return st;
    x = y;
  }
  return TXL_OK;
}

}  // extern "C"
