// Internal launchers behind the C ABI (one per kernel family).
#pragma once

#include "pe_common.cuh"

namespace pe {

// CUDA-core forward (fp32 any head_dim; bf16 head_dims without a tensor-core kernel).
int simt_rows_per_item();
pe_status fwd_simt(pe_dtype dtype, int D, const void* q, const void* k, const void* v,
                   const int32_t* cu, int32_t B, int32_t H, float scale, Window win, void* out,
                   float* lse, int64_t N, TilePlan plan, cudaStream_t stream);

// First-token query (one query row per sequence).
bool first_token_supported(int D);
// With a window the query at position 0 sees keys 0 .. win.right.
// Returns at once on the device when `status` holds an error (a layout that
// failed its check).
pe_status fwd_first_token(pe_dtype dtype, int D, const void* q, const void* k, const void* v,
                          const int32_t* cu, int32_t B, int32_t H, int32_t S, float scale,
                          Window win, void* out, float* lse, float* part,
                          const DeviceStatus* status, cudaStream_t stream);

// First-token query, streaming form: chunks of whole token rows per CTA (all
// heads); sequences that cross chunk edges leave partial states that a second
// kernel merges. Needs first_token_stream_partial_bytes() of scratch in
// `part`; a pipeline wait that gives up records PE_ERR_DEVICE_TIMEOUT in
// `status`, and both kernels return at entry when `status` already holds an
// error (a layout that failed its check). Returns PE_ERR_UNSUPPORTED for
// shapes it does not take.
bool first_token_stream_supported(pe_dtype dtype, int32_t H, int32_t D);
int32_t first_token_stream_chunk(int64_t N);
size_t first_token_stream_partial_bytes(int64_t N, int32_t H, int32_t D);
pe_status fwd_first_token_stream(pe_dtype dtype, int32_t D, const void* q, const void* k,
                                 const void* v, const int32_t* cu, int32_t B, int32_t H,
                                 int64_t N, int32_t S, float scale, Window win, void* out,
                                 float* lse, float* part, DeviceStatus* status,
                                 cudaStream_t stream);

// First-token query, streaming backward: the same chunks of whole token rows;
// dk and dv rows are written as they stream, and dq sums of sequences that
// cross chunk edges are added in chunk order by a second kernel. Delta = dO.O
// is formed in the kernel. Needs first_token_bwd_stream_partial_bytes() of
// scratch in `part`; waits and status as in the forward above.
bool first_token_bwd_stream_supported(pe_dtype dtype, int32_t H, int32_t D);
size_t first_token_bwd_stream_partial_bytes(int64_t N, int32_t H, int32_t D);
pe_status bwd_first_token_stream(pe_dtype dtype, int32_t D, const void* q, const void* k,
                                 const void* v, const void* out, const void* dout,
                                 const float* lse, const int32_t* cu, int32_t B, int32_t H,
                                 int64_t N, int32_t S, float scale, Window win, void* dq,
                                 void* dk, void* dv, float* part, DeviceStatus* status,
                                 cudaStream_t stream);

// CUDA-core backward; delta is [H, Nq] fp32 scratch.
pe_status bwd_simt(pe_dtype dtype, int D, const void* q, const void* k, const void* v,
                   const int32_t* cu, int32_t B, int32_t H, int64_t Nq, float scale,
                   int first_token, Window win, const void* out, const float* lse, const void* dout,
                   void* dq, void* dk, void* dv, float* delta, TilePlan plan, LayoutCheck check,
                   cudaStream_t stream);

// Tensor-core forward, bf16, head_dim 64 (sm_103a). Work items are pairs of
// 128-row query tiles, so the tile plan is built with sm103_fwd_rows_per_item().
int sm103_fwd_rows_per_item();
// Sequences of at most this many tokens run two heads per work item (tile 0
// and tile 1 take one head each); 0 with a window.
int sm103_fwd_pair_heads_rows(Window win);
// ... and at most this many four heads (two per tile, 64 rows each).
int sm103_fwd_quad_heads_rows(Window win);
// 1 when a longer sequence with an odd number of 128-row blocks runs the last
// query tiles of two heads in one item (the plan's pair_odd_tails); 0 with a
// window.
int sm103_fwd_pair_odd_tails(Window win);
pe_status fwd_sm103(const void* q, const void* k, const void* v, const int32_t* cu, int32_t B,
                    int32_t H, int64_t N, float scale, Window win, void* out, float* lse,
                    TilePlan plan, DeviceStatus* status, cudaStream_t stream);

// Tensor-core forward, fp32, head_dim 64, full attention (sm_103a): every
// operand split into bf16 hi and lo parts, three products per GEMM. Same work
// items as the bf16 kernel.
int sm103_f32_fwd_rows_per_item();
int sm103_f32_fwd_pair_heads_rows();
int sm103_f32_fwd_quad_heads_rows();
pe_status fwd_sm103_f32(const void* q, const void* k, const void* v, const int32_t* cu,
                        int32_t B, int32_t H, int64_t N, float scale, void* out, float* lse,
                        TilePlan plan, DeviceStatus* status, cudaStream_t stream);

// Tensor-core forward, bf16, head_dim 128, full attention (sm_103a): P written
// over the first half of its tile's score columns. Same work items as the
// head_dim-64 kernel.
int sm103_d128_fwd_rows_per_item();
int sm103_d128_fwd_pair_heads_rows();
int sm103_d128_fwd_quad_heads_rows();
int sm103_d128_fwd_pair_odd_tails();   // as sm103_fwd_pair_odd_tails, full attention only
pe_status fwd_sm103_d128(const void* q, const void* k, const void* v, const int32_t* cu,
                         int32_t B, int32_t H, int64_t N, float scale, void* out, float* lse,
                         TilePlan plan, DeviceStatus* status, cudaStream_t stream);

// Delta[h, r] = dO_r . O_r (bf16, head_dim 64 or 128) into [H, Nq] fp32.
pe_status bwd_preprocess(pe_dtype dtype, int D, const void* out, const void* dout, int64_t Nq,
                         int32_t H, float* delta, cudaStream_t stream);

// Tensor-core backward, bf16, head_dim 64, full mode (sm_103a): a key pass
// (dK, dV) and a query pass (dQ), each with its own tile plan over 128-row blocks.
pe_status bwd_sm103(const void* q, const void* k, const void* v, const int32_t* cu, int32_t B,
                    int32_t H, int64_t N, float scale, Window win, const float* lse,
                    const void* dout,
                    const float* delta, void* dq, void* dk, void* dv, TilePlan plan,
                    LayoutCheck check, cudaStream_t stream);
// The same two passes for head_dim 128 (full or local); each key-pass item
// accumulates one 64-column half of dK and dV.
pe_status bwd_sm103_d128(const void* q, const void* k, const void* v, const int32_t* cu,
                         int32_t B, int32_t H, int64_t N, float scale, Window win,
                         const float* lse, const void* dout, const float* delta, void* dq,
                         void* dk, void* dv, TilePlan plan, LayoutCheck check,
                         cudaStream_t stream);

}  // namespace pe
