/*
 * txl_relattn.h -- C ABI of the GB300 (sm_103a) Transformer-XL relative-position
 * attention library.
 *
 * The library computes the per-segment hot path of Transformer-XL:
 *
 *   - txl_relattn_forward: relative multi-head attention of one W-token segment
 *     over [memory of M cached rows ; segment] with the four-term relative score
 *     and an in-kernel distance index (no pad-and-reshape), causal mask,
 *     online softmax and P.V;
 *   - txl_mem_update: the memory roll, keeping the last M rows of
 *     [memory ; segment];
 *   - txl_relattn_forward_roll: both of the above in one call (the roll
 *     done by the attention kernel from the tiles it loads, where it can);
 *   - txl_sinusoid_rel: the parameter-free sinusoidal distance table R.
 *
 * Conventions shared by every entry point
 *   - Pointers marked "device" are device memory owned by the caller; the
 *     library never allocates, frees or retains them.  Host pointers are only
 *     read or written during the call.
 *   - Library-owned memory.  Some calls keep device memory of their own, each
 *     named in the call's comment under "Allocates": per-(device, stream)
 *     scratch, made with cudaMalloc on the first call that needs it and
 *     regrown (stream synchronised, old buffer freed) when a later call needs
 *     more; and per-shape unit plans of the bf16 attention kernels (below).
 *     Both are kept until txl_release_cached or process exit.
 *     txl_relattn_forward_static, txl_mem_update and txl_dense allocate
 *     nothing.
 *   - Every call is asynchronous on `stream` (0 = legacy default stream) and
 *     keeps stream order.  The library's bf16 and roll kernels are launched
 *     with programmatic stream serialisation: their CTAs may become resident
 *     while the kernel before them on the stream drains, but each waits at its
 *     first instruction until that kernel has completed and its writes are
 *     visible, so no memory is touched earlier.  Each call returns a
 *     txl_status code.  Argument errors are detected on the host before
 *     any launch, and then nothing is launched.  A failed launch returns
 *     TXL_ERR_CUDA.  Errors detected inside a kernel (a bounded wait that ran out)
 *     are recorded in a device status word read by txl_get_device_status.
 *   - Layouts are dense row-major ("BSHD"): the innermost index is the head
 *     dimension D, then the head H, then the row (query, key or distance), then
 *     the batch B.
 *   - B == 0 or W == 0 is a valid empty call: TXL_OK, nothing is launched.
 *   - The entry points are thread-safe; shape-keyed descriptor caches are
 *     guarded by a mutex.
 */
#ifndef TXL_RELATTN_H
#define TXL_RELATTN_H

#include <cuda_runtime.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TXL_VERSION 160 /* 1.6.0 */

/* Symbols of the shared library (built with hidden default visibility). */
#if defined(__GNUC__)
#define TXL_API __attribute__((visibility("default")))
#else
#define TXL_API
#endif

typedef enum {
  TXL_F32 = 0, /* IEEE binary32 */
  TXL_BF16 = 1 /* bfloat16 (storage); arithmetic accumulates in fp32 */
} txl_dtype;

typedef enum {
  TXL_OK = 0,
  TXL_ERR_INVALID_ARG = 1,    /* null pointer, negative size, r too short, ... */
  TXL_ERR_UNSUPPORTED = 2,    /* valid request outside what this build supports */
  TXL_ERR_ALIAS = 3,          /* an output range overlaps an input range */
  TXL_ERR_CUDA = 4,           /* a CUDA runtime / driver call failed */
  TXL_ERR_DEVICE_TIMEOUT = 5  /* a kernel's bounded wait expired (see below) */
} txl_status;

/*
 * txl_relattn_forward -- relative multi-head attention of one segment.
 *
 * Defines the score of "Transformer-XL, explained", method step 4 (content
 * against content, content against a sinusoidal encoding of the distance i - j,
 * and the two global biases u and v that replace the query in a content-only
 * and a distance-only term, with separate key projections), grouped by the
 * query-side factor:
 *
 *   s[i,j] = scale * ( (q_i + u_h) . k_j  +  (q_i + v_h) . r_{M+i-j} )   j <= M+i
 *   s[i,j] = -inf                                                          j >  M+i
 *   o_i    = sum_j softmax_j(s[i,.]) v_j          lse_i = log sum_j exp(s[i,j])
 *
 * Keys and values extend over [memory ; segment] with the memory first and
 * queries from the segment only (method step 3 and the concatenation in the
 * symbol legend); the distance term is evaluated once per distance and each
 * row is shifted into place (method step 5) by indexing row d = M+i-j of r
 * inside the kernel; the mask lets query i see all M memory rows and segment
 * rows up to i ("Implementing Transformer-XL", relative_attention's causal
 * mask); the scale multiplies the sum of all terms (the same function's
 * division by sqrt(d_head); the simulation's softmax(QK^T/sqrt(d))).
 *
 *   q      device, [B, W, H, D]   `dtype`   queries of the current segment
 *   k      device, [B, M+W, H, D] `dtype`   keys, memory rows 0..M-1 first
 *   v      device, [B, M+W, H, D] `dtype`   values, same row order as k
 *   r      device, [n_r, H, D]    `dtype`   projected distance keys, row d is
 *                                           distance d; n_r >= M+W
 *   bias_u device, [H, D] fp32              global content bias u
 *   bias_v device, [H, D] fp32              global distance bias v
 *   o      device, [B, W, H, D]   `o_dtype` output (must not overlap inputs)
 *   lse    device, [B, H, W] fp32 or NULL   natural-log softmax normaliser
 *   M      memory rows in this call (0 for the first segment)
 *   scale  score scale, 1/sqrt(D) by convention
 *   dtype  TXL_BF16: tensor-core path (tcgen05), D in {64, 128}, fp32
 *          accumulation, o_dtype TXL_BF16 or TXL_F32;
 *          TXL_F32: exact fp32 path (CUDA cores), 1 <= D <= 256, o_dtype TXL_F32.
 *
 * Requirements: q, k, v, r and o 16-byte aligned (TXL_ERR_INVALID_ARG
 * otherwise); o must not overlap q, k, v, r, bias_u, bias_v or lse
 * (TXL_ERR_ALIAS).  Memory rows are only read (stop-gradient).
 *
 * Allocates (bf16 path only; the fp32 path allocates nothing):
 *   - unit plan: with more (batch, head, 128-query tile) units than SMs, the
 *     first call of a shape on a device builds a cost-balanced assignment of
 *     units to the persistent CTAs: a small pinned host buffer and device
 *     table (about 4 * (units + SMs) bytes) plus an event, uploaded by an
 *     asynchronous copy on `stream` (the host does not wait for it).  No plan
 *     is made while `stream` is being captured, nor for a new shape once 256
 *     shapes hold one: those calls deal the units in a fixed order instead,
 *     with the same result;
 *   - split scratch: with fewer units than SMs (D = 64), each unit's key
 *     range is split across CTAs and the partial results take
 *     units * chunks * 128 * 65 * 4 bytes, plus units * 16 bytes of merge
 *     counters, per (device, stream) (see the conventions above).
 */
TXL_API int txl_relattn_forward(const void* q, const void* k, const void* v, const void* r,
                        const float* bias_u, const float* bias_v, void* o, float* lse,
                        int B, int W, int M, int H, int D, int n_r, float scale,
                        txl_dtype dtype, txl_dtype o_dtype, cudaStream_t stream);

/*
 * txl_relattn_forward_static -- txl_relattn_forward that allocates nothing.
 *
 * For callers that cannot call cudaMalloc: a host that has handed all device
 * memory to its own pool up front, code running inside another library's
 * allocator or memory callbacks, or a loop that must never stall on the
 * allocator (cudaMalloc and cudaFree can synchronise the device).  Same
 * arguments, result and errors as txl_relattn_forward, bit for bit (the same
 * kernels run); the units are dealt in a fixed order, never by a plan.
 *
 * When a launch has too few units to fill the GPU, its key ranges are split
 * across CTAs and the partial results need scratch.  This entry point keeps
 * that scratch in one fixed 16 MiB array inside the library (a __device__
 * array that every GPU loading the library holds until exit): at most 4096
 * merge counters (1024 units), then at most 16 MiB - 16 KiB of partial
 * results; a split that needs more returns TXL_ERR_UNSUPPORTED before any
 * launch.  Launches that do not split use no scratch.
 *
 * Set-up: the first call on each device (made current) looks the array's
 * device address up with cudaGetSymbolAddress, which may load the library's
 * device code; make that first call before any stream capture.  Every call
 * on a device shares the one array, which keeps what the last call left: the
 * merge counters must start at zero, and each launch returns them to zero
 * (after a reported TXL_ERR_DEVICE_TIMEOUT, txl_get_device_status zeroes
 * them).  Calls whose kernels overlap on the GPU (different streams without
 * ordering between them) race on the array and give undefined results.  The
 * pages have no counterpart; this is a property of the implementation only.
 */
TXL_API int txl_relattn_forward_static(const void* q, const void* k, const void* v, const void* r,
                               const float* bias_u, const float* bias_v, void* o, float* lse,
                               int B, int W, int M, int H, int D, int n_r, float scale,
                               txl_dtype dtype, txl_dtype o_dtype, cudaStream_t stream);

/*
 * txl_mem_update -- the memory roll.
 *
 * Defines mem_tau = last M rows of [stop_grad(mem_{tau-1}) ; h_tau] from the
 * "Long-context transformers" simulation's segment-recurrence equations (the
 * "Transformer-XL" glossary page's recurrence example is the case M equal to
 * the segment length: the detached segment becomes the memory).  Rows are
 * copied bit for bit.  Allocates nothing.
 *
 *   mem      device, [B, m_prev, C] rows, batch stride mem_bs elements  (may be
 *            NULL when m_prev == 0)
 *   h        device, [B, w, C] rows, batch stride h_bs elements
 *   mem_out  device, [B, m', C] rows, batch stride out_bs elements, with
 *            m' = min(m, m_prev + w); must not overlap mem or h (TXL_ERR_ALIAS)
 *   m_out    host, receives m' (may be NULL)
 *   dtype    element type (TXL_F32 or TXL_BF16); C >= 1
 *
 * A typical caller ping-pongs two [B, M+W, C] buffers: the roll writes the
 * head of the next buffer from the current one (mem = buf, h = buf + M*C,
 * out_bs = mem_bs = h_bs = (M+W)*C).
 */
TXL_API int txl_mem_update(const void* mem, int m_prev, const void* h, int w, void* mem_out, int m,
                   int B, int C, long long mem_bs, long long h_bs, long long out_bs,
                   int* m_out, txl_dtype dtype, cudaStream_t stream);

/*
 * txl_mem_update_kv -- txl_mem_update of the keys and of the values in one
 * launch.  The result is exactly that of txl_mem_update(k_mem, m_prev, k_h,
 * w, k_out, m, ...) and txl_mem_update(v_mem, m_prev, v_h, w, v_out, m, ...)
 * with the shared batch strides; no output may overlap another output or any
 * input (TXL_ERR_ALIAS).  The pages roll keys and values by the same rule;
 * the single launch is a scheduling of the two.  Allocates nothing.
 */
TXL_API int txl_mem_update_kv(const void* k_mem, const void* v_mem, int m_prev, const void* k_h, const void* v_h,
                              int w, void* k_out, void* v_out, int m, int B, int C, long long mem_bs, long long h_bs,
                              long long out_bs, int* m_out, txl_dtype dtype, cudaStream_t stream);

/*
 * txl_relattn_forward_roll -- txl_relattn_forward and the memory roll of its
 * keys and values in one call.
 *
 * The result is exactly that of txl_relattn_forward(q, k, v, ...) followed
 * by txl_mem_update on k and on v, each with mem = the call's memory rows
 * (m_prev = M), h = its segment rows (w = W) and the batch stride of k and v
 * ((M+W)*H*D elements): k_mem_out and v_mem_out receive the last
 * m' = min(m, M+W) rows of [memory ; segment] of every sequence, bit for bit
 * ("Long-context transformers", segment recurrence: the cache for the next
 * segment is the tail of this one's keys and values).
 *
 *   k_mem_out, v_mem_out  device, [B, m', H, D] rows with batch stride
 *                         mem_out_bs elements (>= m'*H*D), `dtype`; must not
 *                         overlap each other or any input or output of the
 *                         attention (TXL_ERR_ALIAS)
 *   m                     memory length to keep (>= 0)
 *   m_out                 host, receives m' (may be NULL)
 *
 * On the bf16 paths (D = 64 and 128), when the kept rows start on a 64-row tile
 * boundary of k and v (M+W-m' a multiple of 64) and k_mem_out, v_mem_out and
 * the stride are 16-byte aligned, the attention kernel writes the kept rows
 * itself, from the key and value tiles it has already loaded, with tensor
 * stores; otherwise the call runs the attention and then the roll kernel.
 * Other arguments and errors as txl_relattn_forward and txl_mem_update.  This
 * fused form has no counterpart on the pages: it is a scheduling of their
 * two steps.  Allocates what txl_relattn_forward allocates for the shape.
 */
TXL_API int txl_relattn_forward_roll(const void* q, const void* k, const void* v, const void* r,
                             const float* bias_u, const float* bias_v, void* o, float* lse,
                             int B, int W, int M, int H, int D, int n_r, float scale,
                             txl_dtype dtype, txl_dtype o_dtype,
                             void* k_mem_out, void* v_mem_out, int m, long long mem_out_bs, int* m_out,
                             cudaStream_t stream);

/*
 * txl_relattn_forward_ring -- txl_relattn_forward with the memory held in a
 * ring buffer instead of in front of the segment's rows.
 *
 * The result is exactly that of txl_relattn_forward with
 *   k = [memory rows in ring order ; k_seg],  v likewise,
 * where memory row m (m = 0 .. M-1, oldest first) is row (start + m) % cap
 * of k_mem / v_mem.  "Transformer-XL, explained", method step 7: with
 * relative positions the memory can be much longer at evaluation time; a
 * ring keeps it in place, so moving to the next segment writes only the
 * segment's own rows (txl_mem_ring_append) instead of copying M rows.  The
 * ring layout has no counterpart on the pages; it stores the same memory.
 *
 *   k_mem, v_mem  device, [B, cap, H, D] `dtype` (may be NULL when M = 0)
 *   cap           ring rows per sequence (>= M)
 *   start         ring row of memory row 0 (0 <= start < cap when M > 0)
 *   M             memory rows in this call
 *   k_seg, v_seg  device, [B, W, H, D] `dtype`  the segment's keys and values
 * Other arguments and errors as txl_relattn_forward.
 *
 * On the bf16 D = 64 path with cap, start and M multiples of 64 the kernel
 * reads the ring in place (a key tile never wraps); otherwise the call first
 * copies [memory ; segment] into library scratch per (device, stream)
 * (2 * B * (M+W) * H * D elements; see the conventions above).  Allocates
 * that scratch and what txl_relattn_forward allocates for the shape.
 */
TXL_API int txl_relattn_forward_ring(const void* q, const void* k_mem, const void* v_mem, int cap, int start,
                             int M, const void* k_seg, const void* v_seg, const void* r,
                             const float* bias_u, const float* bias_v, void* o, float* lse,
                             int B, int W, int H, int D, int n_r, float scale,
                             txl_dtype dtype, txl_dtype o_dtype, cudaStream_t stream);

/*
 * txl_relattn_forward_ring_append -- txl_relattn_forward_ring, then
 * txl_mem_ring_append of k_seg into k_mem and of v_seg into v_mem: the
 * result, the rings afterwards and *start_out / *m_out are exactly those of
 * the three calls in order.  With bf16, D = 64, cap, start, M and W
 * multiples of 64 and M + W <= cap, it is one launch: the new rows go to ring
 * slots the memory does not occupy, so the attention kernel stores them from
 * the tiles it loads while it runs.  Otherwise the three calls run in order.
 * Arguments as in the two calls; k_seg and v_seg must not overlap the rings.
 * Allocates what txl_relattn_forward_ring allocates.
 */
TXL_API int txl_relattn_forward_ring_append(void* k_mem, void* v_mem, int cap, int start, int M,
                                    const void* q, const void* k_seg, const void* v_seg, const void* r,
                                    const float* bias_u, const float* bias_v, void* o, float* lse,
                                    int B, int W, int H, int D, int n_r, float scale,
                                    txl_dtype dtype, txl_dtype o_dtype, int* start_out, int* m_out,
                                    cudaStream_t stream);

/*
 * txl_mem_ring_append -- the memory roll of a ring buffer.
 *
 * The ring holds m rows (memory row x at ring row (start + x) % cap).  After
 * the call it holds the last min(cap, m + w) rows of [memory ; h], oldest
 * first from ring row *start_out -- the rows txl_mem_update(mem, m, h, w,
 * out, cap) would give, without moving the ones that stay ("Long-context
 * transformers", segment recurrence: the next memory is the last M rows of
 * [memory ; segment]).  Only the new rows are written: ring rows
 * (start + m + x) % cap for x >= max(0, w - cap).
 *
 *   mem      device, [B, cap, C] `dtype`, batch stride cap*C elements
 *   h        device, [B, w, C] rows with batch stride h_bs elements (>= w*C)
 *   start_out, m_out  host, receive the new start and row count (may be NULL)
 *
 * Run it after the attention that reads the ring (stream order): it
 * overwrites the oldest rows.  h must not overlap the ring (TXL_ERR_ALIAS).
 * Allocates nothing.
 */
TXL_API int txl_mem_ring_append(void* mem, int cap, int start, int m, const void* h, int w, int B, int C,
                        long long h_bs, int* start_out, int* m_out, txl_dtype dtype, cudaStream_t stream);

/*
 * txl_dense -- the layer's dense products: y_z = x W_z (+ bias) (then ReLU),
 * z = 0 .. batch-1, on this library's tensor-core GEMM.
 *
 * "Implementing Transformer-XL", recurrent-memory chapter: the input
 * projections (q = h W_q, k = h W_{k,E}, v = h W_v, r = R W_{k,R}), the output
 * projection and feed_forward's two products, the first with b_1 and the
 * ReLU, the second with b_2.
 *
 *   x       device, [m, k] bf16 row-major (shared by the batch)
 *   W       device, [k, n] bf16 row-major, matrix z at W + z w_batch_stride
 *   y       device, [m, n] bf16 row-major, matrix z at y + z y_batch_stride
 *   bias    device, [n] fp32 or NULL (the same for every z)
 *   relu    nonzero: ReLU after the bias
 *   batch   >= 1; the strides (elements) are ignored when batch == 1, else
 *           w_batch_stride >= k n, y_batch_stride >= m n, both multiples of 8
 *
 * bf16 operands, fp32 accumulation; the bias is added to the fp32 sum and the
 * ReLU applied before the one rounding to bf16.  n and k multiples of 8
 * (TXL_ERR_UNSUPPORTED otherwise); x, W, y 16-byte aligned; y must not
 * overlap x, W or bias (TXL_ERR_ALIAS).  m == 0 is an empty call.  Allocates
 * nothing.
 */
TXL_API int txl_dense(const void* x, const void* W, void* y, int m, int n, int k, int batch, long long w_batch_stride,
                      long long y_batch_stride, const float* bias, int relu, cudaStream_t stream);

/*
 * txl_layer_forward -- one Transformer-XL layer on a segment, the attention
 * memory kept as a ring of projected keys and values.
 *
 * "Implementing Transformer-XL", recurrent-memory chapter (forward,
 * layer_norm, feed_forward), with the attention of txl_relattn_forward:
 *
 *   q = h W_q,  k_seg = h W_k,  v_seg = h W_v,  r = R W_r
 *   a = relative attention of q over [memory ; segment] (the ring's M rows)
 *   x = LN1(h + a W_o)
 *   out = LN2(x + ReLU(x W_1 + b_1) W_2 + b_2)
 *   LN(z) = gamma (z - mean(z)) / (std(z) + 1e-6) + beta  (population std)
 *
 * then k_seg and v_seg are appended to the rings (txl_mem_ring_append
 * semantics; *start_out, *m_out receive the rings' new state).  The
 * memory's keys and values are cached already projected: the projections act
 * row by row, so this equals caching the layer's input rows and projecting
 * [memory ; segment] again ("Transformer-XL, explained", method step 2).
 *
 *   h, out     device, [B, W, d_model] bf16 (out must not overlap h)
 *   k_mem, v_mem  device, [B, cap, H, D] bf16 rings (memory row m at
 *              ring row (start + m) % cap)
 *   w          host struct of device weight pointers (below); bf16 matrices
 *              row-major [in, out], fp32 vectors
 *   R          device, [n_r, d_model] bf16 raw distance table (txl_sinusoid_rel),
 *              n_r >= M + W
 *   workspace  device, txl_layer_workspace_bytes(...) bytes, 256-byte aligned
 *   D          64 or 128; d_model and d_ff multiples of 8, d_model <= 1024
 *
 * Every product runs on txl_dense's GEMM (bf16 in, fp32 accumulation, bf16
 * out), b_1 with the ReLU and b_2 in its epilogue; when W_k starts right after
 * W_q and W_v right after W_k (one [3, d_model, H*D] allocation), the three
 * projections and r = R W_r run as one launch.  Every intermediate lives in
 * `workspace`; the attention inside may make a unit plan as
 * txl_relattn_forward does, and when the ring cannot be read in place (cap,
 * start or M not multiples of 64) it takes the ring scratch of
 * txl_relattn_forward_ring.
 */
typedef struct {
  const void* W_q;        /* [d_model, H*D] */
  const void* W_k;        /* [d_model, H*D]  content keys (W_{k,E}) */
  const void* W_v;        /* [d_model, H*D] */
  const void* W_r;        /* [d_model, H*D]  distance keys (W_{k,R}) */
  const float* bias_u;    /* [H, D] */
  const float* bias_v;    /* [H, D] */
  const void* W_o;        /* [H*D, d_model] */
  const float* ln1_gamma; /* [d_model] */
  const float* ln1_beta;  /* [d_model] */
  const void* W_1;        /* [d_model, d_ff] */
  const float* b_1;       /* [d_ff] */
  const void* W_2;        /* [d_ff, d_model] */
  const float* b_2;       /* [d_model] */
  const float* ln2_gamma; /* [d_model] */
  const float* ln2_beta;  /* [d_model] */
} txl_layer_weights;

TXL_API size_t txl_layer_workspace_bytes(int B, int W, int d_model, int H, int D, int d_ff, int n_r);

TXL_API int txl_layer_forward(const void* h, void* out, void* k_mem, void* v_mem, int cap, int start, int M,
                      const txl_layer_weights* w, const void* R, int n_r,
                      int B, int W, int d_model, int H, int D, int d_ff, float scale,
                      void* workspace, size_t workspace_bytes, int* start_out, int* m_out,
                      cudaStream_t stream);

/*
 * txl_stack_forward -- n_layers layers of txl_layer_forward on a segment, the
 * output of layer l the input of layer l+1, each layer with its own rings.
 *
 * "Transformer-XL, explained", method step 6: each layer caches its own
 * states, so layer l of this segment reads what layer l-1 saw of the last
 * one and the reach grows with depth ("Implementing Transformer-XL", the
 * stacked layers).  Every layer's rings hold the same M rows from ring row
 * `start` (they advance together); *start_out, *m_out receive their common
 * new state, as from txl_layer_forward.
 *
 *   h, out        device, [B, W, d_model] bf16 (out must not overlap h)
 *   k_mem, v_mem  host arrays of n_layers device ring pointers, [B, cap, H, D]
 *                 bf16 each, all distinct (TXL_ERR_ALIAS otherwise)
 *   w             host array of n_layers weight structs
 *   workspace     device, txl_stack_workspace_bytes(...) bytes, 256-byte
 *                 aligned (the layer workspace and two [B, W, d_model]
 *                 buffers for the layers' outputs)
 * Other arguments, requirements and allocations as txl_layer_forward.
 */
TXL_API size_t txl_stack_workspace_bytes(int B, int W, int d_model, int H, int D, int d_ff, int n_r);

TXL_API int txl_stack_forward(const void* h, void* out, int n_layers, void* const* k_mem, void* const* v_mem,
                              int cap, int start, int M, const txl_layer_weights* w, const void* R, int n_r, int B,
                              int W, int d_model, int H, int D, int d_ff, float scale, void* workspace,
                              size_t workspace_bytes, int* start_out, int* m_out, cudaStream_t stream);

/*
 * txl_relattn_backward -- gradients of txl_relattn_forward.
 *
 * Given dout = dL/do for the forward's o, writes the gradients of L through
 * the score of txl_relattn_forward:
 *
 *   p[i,j] = exp(s[i,j] - lse_i),  Delta_i = dout_i . o_i
 *   g[i,j] = scale * p[i,j] * (dout_i . v_j - Delta_i)
 *   dq_i   = sum_j g[i,j] (k_j + r_{M+i-j})
 *   dk_j, dv_j (segment rows j = M..M+W-1 only):
 *          dk_j = sum_i g[i,j] (q_i + u),   dv_j = sum_i p[i,j] dout_i
 *   dr_d   = sum over pairs with M+i-j = d of g[i,j] (q_i + v)
 *   dbias_u = sum_{b,i} sum_j g[i,j] k_j,   dbias_v = sum_{b,i} sum_j g[i,j] r_{M+i-j}
 *
 * "Transformer-XL, explained", method step 2 and the symbol SG(.): the memory
 * is read as a fixed input and backpropagation stays inside the current
 * segment, so the memory rows of k and v receive no gradient; r, u and v are
 * shared by every pair and receive all of theirs.
 *
 *   q, k, v, r, bias_u, bias_v, B, W, M, H, D, n_r, scale, dtype
 *                as in the forward call that produced o and lse
 *   o      device, [B, W, H, D] `go_dtype`  the forward's output
 *   lse    device, [B, H, W] fp32            the forward's lse (required)
 *   dout   device, [B, W, H, D] `go_dtype`  gradient of the output
 *   dq     device, [B, W, H, D] fp32
 *   dk, dv device, [B, W, H, D] fp32   gradients of k, v rows M..M+W-1
 *   dr     device, [n_r, H, D] fp32    rows no pair uses (d >= M+W) are zero
 *   dbias_u, dbias_v  device, [H, D] fp32
 *
 * Every output is overwritten (not accumulated into).  Outputs must not
 * overlap each other or any input (TXL_ERR_ALIAS); every pointer 16-byte
 * aligned (TXL_ERR_INVALID_ARG).  D <= 256 (TXL_ERR_UNSUPPORTED otherwise).
 * Paths: bf16 q, k, v, r with bf16 o and dout and D = 64 or 128 run on the
 * tensor cores (tcgen05) with the pair terms materialised: a kernel rebuilds
 * p and g per 64-key step and writes them in bf16 to scratch (g in key and in
 * distance order, p in key order), one launch of tcgen05 products then forms
 * dq (key and distance parts in one tile, with the bias gradients'
 * partials), dk, dv and dr, and an ordered sum the bias gradients;
 * deterministic.  Every other case runs on CUDA cores in fp32 arithmetic,
 * fully deterministic.  (A test hook sends D = 64 to fused tensor-core
 * kernels instead: a dq kernel over query tiles, which also sums dr and the
 * bias gradients, and a dk/dv kernel over 64-key blocks; there dr arrives by
 * fp32 atomic adds, so its last bits may differ between calls.)
 * Allocates: per-(device, stream) scratch (see the conventions above): for
 * the pair-term path, per chunk of Bc sequences, 3 * Bc*H*W*LP * 2 bytes of
 * pair terms (LP = M + W rounded up to 64) plus (q+u), (q+v) in bf16
 * (2 * Bc*W*H*D * 2 bytes), and the bias partials, Bc the most sequences that
 * fit 1 GiB (at least one; the chunks run in turn): all 8 sequences, 0.47 GB,
 * at B=8 H=8 D=128 W=M=768, all 22, 0.58 GB, at B=22 H=8 D=64 W=M=512; for
 * the fused D = 64 kernels the per-row Delta and the per-tile partial sums.
 */
TXL_API int txl_relattn_backward(const void* q, const void* k, const void* v, const void* r,
                         const float* bias_u, const float* bias_v, const void* o, const float* lse,
                         const void* dout, float* dq, float* dk, float* dv, float* dr,
                         float* dbias_u, float* dbias_v,
                         int B, int W, int M, int H, int D, int n_r, float scale,
                         txl_dtype dtype, txl_dtype go_dtype, cudaStream_t stream);

/*
 * txl_sinusoid_rel -- the raw sinusoidal distance table R[n_dist, dim].
 *
 * "Transformer-XL, explained", symbol legend: R_{i-j} is a sinusoidal encoding
 * of the distance with no trained parameters; fixed sinusoids give encodings
 * to distances longer than any seen in training, so no distance is clipped.
 *
 *   R[d, 2k]   = sin(d * w_k),   R[d, 2k+1] = cos(d * w_k),
 *   w_k = 10000^(-2k/dim),  d = 0 .. n_dist-1
 *
 * The angle is formed and reduced modulo 2*pi in extended precision before the
 * fp32 sine and cosine, so |R - exact| stays near 1e-7 for every distance.
 *
 *   R      device, [n_dist, dim] `dtype`
 *   dim    even, >= 2;  n_dist >= 0 (0 is an empty call)
 * Allocates nothing.
 */
TXL_API int txl_sinusoid_rel(void* R, int n_dist, int dim, txl_dtype dtype, cudaStream_t stream);

/*
 * txl_get_device_status -- synchronises `stream`, then reads and clears the
 * device status word of the current device.  Returns TXL_OK, or
 * TXL_ERR_DEVICE_TIMEOUT when a kernel gave up a bounded wait (it then exits
 * cleanly, leaving its outputs undefined, and the context stays usable), or
 * TXL_ERR_CUDA if the synchronisation itself failed.
 */
TXL_API int txl_get_device_status(cudaStream_t stream);

/*
 * txl_release_cached -- synchronises the current device, then frees the
 * library-owned memory kept for it: every stream's split, ring and backward
 * scratch and every unit plan.  Later calls make them again as needed.  No
 * call of this library may be in flight on the device from another thread.
 * Returns TXL_OK or TXL_ERR_CUDA.
 */
TXL_API int txl_release_cached(void);

/* Human-readable name of a txl_status value (static string). */
TXL_API const char* txl_status_string(int status);

/* TXL_VERSION of the built library. */
TXL_API int txl_version(void);

/*
 * Test hooks (not part of the numerical API).
 *
 * txl_debug_set_wait_limit_ns: upper bound, in nanoseconds, of every bounded
 * wait inside the kernels (default 2e9).  Values < 1000 are rejected.
 *
 * txl_debug_inject_stall: when nonzero, the next txl_relattn_forward or
 * txl_relattn_backward on a tensor-core path has its loads stop early (the
 * forward's loader after the first key tile, the backward's after the first
 * two key steps), so the consumers' bounded waits expire and the call reports
 * TXL_ERR_DEVICE_TIMEOUT through txl_get_device_status.  The flag clears
 * itself after that one call.
 */
TXL_API int txl_debug_set_wait_limit_ns(unsigned long long ns);
TXL_API int txl_debug_inject_stall(int on);
/* Test hook: nsplit > 0 makes the bf16 D = 64 forward split every unit's
 * key steps into min(nsplit, steps of the shortest unit) chunks instead of
 * the count its cost model picks; 0 restores the model. */
TXL_API int txl_debug_force_split(int nsplit);
/* Test hook: the cap, in bytes, on the scratch of one chunk of sequences of
 * the D = 128 tensor-core backward (default 1 GiB; 0 restores it).  A smaller
 * cap splits the batch into more chunks, run one after the other. */
TXL_API int txl_debug_set_bwd_chunk_bytes(unsigned long long bytes);
/* Test hook: bn = 64, 128 or 256 fixes the column tile of txl_dense's GEMM
 * (and the layer's products) instead of the width its cost model picks per
 * shape; 0 restores the model.  TXL_ERR_INVALID_ARG for any other value. */
TXL_API int txl_debug_force_dense_tile_n(int bn);
/* Test hook: the path of the bf16 backward at D = 64: 1 the fused kernels, 2
 * the pair terms materialised in scratch (the path it takes by default, as
 * at D = 128), 0 restores the choice.  TXL_ERR_INVALID_ARG for any other
 * value. */
TXL_API int txl_debug_force_bwd_path(int path);
/* Test hook, host only: how many of the longest query tiles the backward's
 * pair-term kernel runs as two CTAs per (sequence, head) unit, each over half
 * of the unit's key steps (0, 1 or 2), for n_query_tiles tiles of 128 queries
 * of seq_heads (sequence, head) pairs on `sms` SMs.  The host models the
 * launch as CTAs starting in order on the first free SM, a CTA costing its
 * key steps plus 3, and takes the count with the shortest modelled launch
 * (0 without modelling when (n_query_tiles + 2) * seq_heads exceeds 200000).
 * Returns -1 for negative sizes or sms <= 0. */
TXL_API int txl_debug_pair_split_tiles(int n_query_tiles, int seq_heads, int W, int M, int sms);
/* Test hooks, host only: the key-range split of the bf16 D = 64 attention
 * (txl_relattn_forward, "Allocates").  txl_debug_attention_split returns the
 * number of chunks (1: no split) the library takes for a device of `sms`
 * SMs, -1 for bad arguments.  txl_debug_attention_items writes *n_items and,
 * where items is non-null and cap (items) suffices, items [n_items][5]: work
 * item it covers sequence b, head h, queries i0 .. i0+127 and 64-key steps
 * t0 .. t0+nks-1 (item it is chunk it % nsplit of unit it / nsplit; units
 * are numbered longest query tile first).  nsplit runs from 1 to 64 and may
 * not exceed the key steps of the shortest unit (the forced split is clamped
 * to that).  Returns 0, -1 for bad arguments, -2 if cap is short. */
TXL_API int txl_debug_attention_split(int B, int H, int W, int M, int sms);
TXL_API int txl_debug_attention_items(int B, int H, int W, int M, int nsplit, int* items, int cap, int* n_items);
/* Test hook, host only: the unit plan the bf16 attention (D = 64 and 128)
 * builds for a shape with more units than CTAs (txl_relattn_forward,
 * "Allocates"):
 * units (batch, head, 128-query tile), numbered longest query tile first,
 * dealt to `ctas` persistent CTAs by cost (key steps plus a unit boundary).
 * Writes *stride and, where table is non-null and cap (entries) suffices,
 * table [ctas][stride]: CTA c runs units table[c][0], table[c][1], ... up
 * to the first -1.  Returns 0, -1 for bad arguments or a shape past 65536
 * units or CTAs, -2 if cap is short. */
TXL_API int txl_debug_unit_plan(int B, int H, int W, int M, int ctas, int* table, int cap, int* stride);
/* Test hook, host only: how the backward's two tensor-core launches divide
 * the work for B sequences (one chunk) of W queries, M memory rows and H
 * heads, with the split_qt longest query tiles split (0 to min(2, query
 * tiles)).  Writes *n_ctas and *n_tiles; then, where the array is non-null
 * and its capacity (entries) suffices:
 *   ctas  [n_ctas][5]: the pair kernel's CTA u works on sequence b, head h,
 *         queries i0 .. i0+127 and 64-key steps t0 .. t0+nks-1;
 *   tiles [n_tiles][6]: the products' tile u: mode (0 dq, 1 dk, 2 dv, 3 dr),
 *         z (sequence * H + head, or the head for dr), m0 (first output row:
 *         query, key or distance), kb0 (first 64-deep k block), nkb (k blocks),
 *         nkb_c (dq: k blocks of its key part; the distance part has as many).
 * Returns 0, -1 for bad arguments, -2 if a capacity is short. */
TXL_API int txl_debug_bwd_pairs_work(int B, int W, int M, int H, int split_qt, int* n_ctas, int* n_tiles,
                                     int* ctas, int cap_ctas, int* tiles, int cap_tiles);

#ifdef __cplusplus
}
#endif

#endif /* TXL_RELATTN_H */
