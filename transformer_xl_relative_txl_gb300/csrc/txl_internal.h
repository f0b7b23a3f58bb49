// Internal launch interface between the C-ABI layer (api.cu) and the kernel
// translation units.  Arguments are validated by the caller.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

namespace txl {

// Bits of the device status word.
constexpr unsigned int kStatusTimeoutBit = 1u;  // a bounded wait expired

struct WaitCtl {
  unsigned int* status;           // device status word
  unsigned long long limit_ns;    // bound of every wait
  int inject_stall;               // loader stops after the first key tile
};

// Sinusoidal distance table.  rho_hi + rho_lo: 10000^(-2/dim) as a
// double-float; c1..c3: 2*pi split into three floats whose products with the
// needed multiples are exact (Cody-Waite reduction constants).
cudaError_t launch_sinusoid(void* R, int n_dist, int dim, bool bf16, float rho_hi, float rho_lo, float c1,
                            float c2, float c3, cudaStream_t stream);

// Memory roll over raw bytes: out[b] = rows [mem_row0, mem_row0 + n_from_mem)
// of mem[b], then rows from h_row0 of h[b], rows_out rows in all.
cudaError_t launch_mem_roll(const void* mem, const void* h, void* out, int B, long long rows_out,
                            long long n_from_mem, long long mem_row0, long long h_row0, long long row_bytes,
                            long long mem_bs_bytes, long long h_bs_bytes, long long out_bs_bytes,
                            cudaStream_t stream);
// The same for one or two tensors of one geometry (keys and values) in one
// launch.  With wc given and every address, stride and row a multiple of 16
// bytes it runs the bulk-copy kernel (bounded waits reported through wc),
// else the vector kernel, one launch per tensor.
struct RollTensor {
  const void* mem;
  const void* h;
  void* out;
};
cudaError_t launch_mem_roll_multi(const RollTensor* t, int ntensors, int B, long long rows_out, long long n_from_mem,
                                  long long mem_row0, long long h_row0, long long row_bytes, long long mem_bs_bytes,
                                  long long h_bs_bytes, long long out_bs_bytes, const WaitCtl* wc,
                                  cudaStream_t stream);

// Exact fp32 relative attention (CUDA cores).
cudaError_t launch_relattn_f32(const float* q, const float* k, const float* v, const float* r,
                               const float* bias_u, const float* bias_v, float* o, float* lse, int B,
                               int W, int M, int H, int D, float scale, cudaStream_t stream);

// bf16 tensor-core relative attention (tcgen05 + TMEM + TMA).
// Tensor maps: q over {D, H, W, B} with a {64, 1, 128, 1} box; k and v over
// {D, H, M+W, B} with {64, 1, 64, 1}; r over {D, H, n_r} with {64, 1, 64};
// all bf16, 128-byte swizzle, zero fill out of bounds.
cudaError_t launch_relattn_tc(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                              const CUtensorMap& tm_r, const CUtensorMap* tm_km, const CUtensorMap* tm_vm,
                              int roll_src0, const float* bias_u, const float* bias_v, void* o, float* lse, int B,
                              int W, int M, int H, int D, bool o_bf16, float scale, bool allow_plan,
                              const WaitCtl& wc, cudaStream_t stream);

// Keys and values split between a ring of memory rows and the segment: the
// maps of launch_relattn_tc64's tm_k / tm_v then describe the rings
// {D, H, cap, B} (memory row m at ring row (start + m) % cap), and tm_ks /
// tm_vs the segment rows {D, H, W, B}, all with a {64, 1, 64, 1} box.  cap,
// start and M are multiples of 64 and M <= cap.  append: the kernel also
// stores the segment's rows into ring rows (start + M + x) % cap (needs
// W % 64 == 0 and M + W <= cap, so they miss the memory being read).
struct RingMaps {
  CUtensorMap tm_ks, tm_vs;
  int cap, start;
  bool append;
};

// Specialisation for D = 64 (same tensor maps).
// tm_o: the bf16 output's map (box 64 x 1 x 32 x 1); required when o_bf16.
// roll_src0 >= 0: also store rows [roll_src0, M+W) of k and v (a multiple of
// 64) to the memory outputs described by tm_km / tm_vm (box 64 x 1 x 64 x 1,
// rows counted from roll_src0); -1: no roll.
// nsplit > 1: every unit's key steps are split into nsplit chunks run as
// separate work items; their results go to part_o
// [units*nsplit][128][64] fp32 and part_lse [units*nsplit][128] fp32; the
// last chunk to finish a unit's rows merges them into o and lse, counting in
// part_cnt [units][4], which must be zero before the launch (and is again
// after it).
// allow_plan: with more units than SMs, deal them to the CTAs by a
// host-made, cost-balanced plan (built and uploaded once per shape, which
// allocates, except during stream capture); otherwise, or without
// allow_plan, the snake order.
// A cost-balanced assignment of the (batch, head, query tile) units, longest
// first, to P persistent CTAs: device table [P][*stride] of unit indices
// (-1 ends a row), made on first use of a shape (a pinned host buffer, a
// device buffer, an event and an asynchronous upload on `stream`) and kept
// until release_plans (relattn_tc64.cu).  *table is set to nullptr (the
// caller keeps the snake order, nothing is allocated) while `stream` is being
// captured and the shape has no completed upload, and for new shapes once
// 256 are cached.
cudaError_t unit_plan(int B, int H, int W, int M, int P, cudaStream_t stream, const int** table, int* stride);
// Frees every plan of device `dev` (no launch that reads one may be in flight).
cudaError_t release_plans(int dev);

cudaError_t launch_relattn_tc64(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                const CUtensorMap& tm_r, const CUtensorMap* tm_o, const CUtensorMap* tm_km,
                                const CUtensorMap* tm_vm, int roll_src0, const RingMaps* ring,
                                const float* bias_u, const float* bias_v, void* o, float* lse, int B, int W, int M,
                                int H, bool o_bf16, float scale, int nsplit, float* part_o, float* part_lse,
                                int* part_cnt, bool allow_plan, const WaitCtl& wc, cudaStream_t stream);

// Backward on CUDA cores (fp32 arithmetic; q, k, v, r fp32 or bf16, o and
// dout fp32 or bf16; D <= 256).  dk, dv cover the segment's key rows.
// scratch: relattn_bwd_simt_scratch_bytes(B, W, H, D) bytes.  vec16: every
// row of q, k, v, r starts on a 16-byte boundary and D is a multiple of the
// 16-byte vector width.
size_t relattn_bwd_simt_scratch_bytes(int B, int W, int H, int D);
cudaError_t launch_relattn_bwd_simt(const void* q, const void* k, const void* v, const void* r,
                                    const float* bias_u, const float* bias_v, const void* o, const float* lse,
                                    const void* dout, float* dq, float* dk, float* dv, float* dr, float* du,
                                    float* dvb, int B, int W, int M, int H, int D, int n_r, float scale, bool bf16,
                                    bool go_bf16, bool vec16, void* scratch, cudaStream_t stream);

// du, dv_bias of each head from per-tile partial sums part [n_part][H][2][D]
// (d(q+u) columns, then d(q+v)), summed in order.
cudaError_t launch_bwd_bias(const float* part, int n_part, int H, int D, float* du, float* dvb,
                            cudaStream_t stream);

// Backward on the tensor cores, bf16 inputs, o and dout, D = 64.  Tensor
// maps as the forward's (q and dout over {D, H, W, B} with a {64, 1, 128, 1}
// box, k and v {64, 1, 64, 1}); tm_rw: r over {D, H, n_r} with a
// {64, 1, 192} box.  dr is zeroed here, then receives atomic sums.
// scratch: relattn_bwd_tc64_scratch_bytes(B, W, H) bytes.
size_t relattn_bwd_tc64_scratch_bytes(int B, int W, int H);
cudaError_t launch_relattn_bwd_tc64(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                    const CUtensorMap& tm_rw, const CUtensorMap& tm_do, const CUtensorMap& tm_dr,
                                    const float* bias_u,
                                    const float* bias_v, const float* lse, const void* o, const void* dout,
                                    float* dq, float* dk, float* dv, float* dr, float* du, float* dvb, int B,
                                    int W, int M, int H, int n_r, float scale, void* scratch, const WaitCtl& wc,
                                    cudaStream_t stream);

// Backward on the tensor cores, bf16 inputs, o and dout, D = 64 or 128
// (relattn_bwd_pairs.cu): the pair terms are materialised in bf16 scratch and
// the gradient products run as tensor-core GEMMs (any M: the dk / dv tiles
// start on a multiple of 8 key columns at or before column M).  Encodes its
// own tensor maps with `encode`.  Every output is
// written in full (dr rows >= M + W are zeroed).
// scratch: relattn_bwd_pairs_scratch_bytes(B, W, M, H, D) bytes.
// The scratch holds one chunk of sequences (as many as keep it within 1 GiB,
// at least one); the chunks run one after the other and dr accumulates over
// them.  relattn_bwd_pairs_set_chunk_bytes changes the cap (0: the default).
size_t relattn_bwd_pairs_scratch_bytes(int B, int W, int M, int H, int D);
void relattn_bwd_pairs_set_chunk_bytes(size_t bytes);
bool relattn_bwd_pairs_supported(int W, int M, int D);
// How many of the longest query tiles the pair kernel runs as two CTAs per
// unit (0-2), for nqt query tiles of bh (sequence, head) pairs on sms SMs.
int relattn_bwd_pairs_split_tiles(int nqt, int bh, int W, int M, int sms);
// The pair kernel's CTAs (b, h, i0, t0, nks per CTA) and the products'
// tiles (mode, z, m0, kb0, nkb, nkb_c per tile) for B sequences, as the two
// launches map them; host only.  0, -1 for bad arguments, -2 if a cap is short.
int relattn_bwd_pairs_work(int B, int W, int M, int H, int split_qt, int* n_ctas, int* n_tiles, int* ctas,
                           int cap_ctas, int* tiles, int cap_tiles);
cudaError_t launch_relattn_bwd_pairs(PFN_cuTensorMapEncodeTiled_v12000 encode, const void* q, const void* k,
                                     const void* v, const void* r, const float* bias_u, const float* bias_v,
                                     const float* lse, const void* o, const void* dout, float* dq, float* dk,
                                     float* dv, float* dr, float* du, float* dvb, int B, int W, int M, int H, int D,
                                     int n_r, float scale, void* scratch, const WaitCtl& wc, cudaStream_t stream);

// The layer's dense products on the tensor cores (gemm_tc.cu): row-major
// bf16 C_z [m, n] = A [m, k] B_z [k, n] (+ bias [n], fp32) (then ReLU),
// z < batch, fp32 accumulation, one rounding.  Tensor maps (bf16, 128-byte
// swizzle, zero fill): tm_a over {k, m} with a {64, 128} box; tm_b over
// {n, k, batch} with a {64, gemm_tc_k_block(bn), 1} box; tm_c over
// {n, m, batch} with a {64, 32, 1} box.  bn: columns per tile, 64, 128 or
// 256 (gemm_tc_tile_n picks one for the shape).
// launch_gemm_tc2 runs a second product C2 [m2, n] = A2 [m2, k] B2 [k, n]
// (no bias, no ReLU; maps as above with batch 1) in the same launch, its
// tiles after the first product's; m2 = 0: none.
int gemm_tc_tile_n(int m, int n, int batch, int m2 = 0);
void gemm_tc_force_tile_n(int bn);  // test hook: 64, 128 or 256 fixes the column tile, 0 restores the choice
int gemm_tc_k_block(int bn);
cudaError_t launch_gemm_tc(const CUtensorMap& tm_a, const CUtensorMap& tm_b, const CUtensorMap& tm_c, int m, int n,
                           int k, int batch, int bn, const float* bias, bool relu, const WaitCtl& wc,
                           cudaStream_t stream);
cudaError_t launch_gemm_tc2(const CUtensorMap& tm_a, const CUtensorMap& tm_b, const CUtensorMap& tm_c, int m, int n,
                            int k, int batch, const float* bias, bool relu, const CUtensorMap& tm_a2,
                            const CUtensorMap& tm_b2, const CUtensorMap& tm_c2, int m2, int bn, const WaitCtl& wc,
                            cudaStream_t stream);
// out = LN(a + b (+ bias)) row by row over d columns (bf16 rows, fp32 gamma,
// beta, bias; d a multiple of 8, <= 1024) (layer.cu).
cudaError_t launch_add_ln(const void* a, const void* b, const float* bias, const float* gamma, const float* beta,
                          void* out, long long rows, int d, cudaStream_t stream);

// The bf16 attention kernels' unit plan for P CTAs as the library builds it: [P][stride]
// unit indices, -1 ending each row; host only.  0, -1 for bad arguments or a
// shape past 65536 units or CTAs, -2 if cap is short (*stride set).
int relattn_tc64_plan_table(int B, int H, int W, int M, int P, int* table, int cap, int* stride);
// Number of chunks the D = 64 kernel should split each unit's key steps
// into (1: no split), from the shape and the device's SM count.
int relattn_tc64_split(int B, int H, int W, int M);
// The same choice for a device of `sms` SMs; host only.
int relattn_tc64_split_for(int B, int H, int W, int M, int sms);
// The attention's work items for nsplit chunks per unit (1 to 64, at most a
// unit's key steps), as (b, h, i0, t0, nks) rows in launch order; host only.
// 0, -1 for bad arguments, -2 if cap (items) is short (*n_items set).
int relattn_tc64_items(int B, int H, int W, int M, int nsplit, int* items, int cap, int* n_items);

}  // namespace txl
