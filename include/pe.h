/*
 * pe.h - C ABI of the padding-free packed attention library (libpe).
 *
 * Variable-length sequences live in one flat token-major buffer
 * [num_tokens, num_heads, head_dim] with no padding; int32 cu_seqlens marks
 * where each sequence starts, and every sequence attends only to itself
 * (page "Source code for gigl.nn.packed_attention", module docstring,
 * "Data flow of a packed forward").
 *
 * Conventions shared by every call:
 *   - Every buffer argument is DEVICE memory owned by the caller, except the
 *     host out-parameters and the host grids of pe_upload_packed and
 *     pe_download_padded. The library allocates nothing; between calls it
 *     keeps only per-device attribute caches, the process-wide wait limit
 *     (pe_set_wait_limit_ns) and the allocation-free forward's static array.
 *   - Every call is asynchronous on `stream` (NULL = the legacy default
 *     stream), except pe_pack_sequences, pe_pack_document_ids and
 *     pe_flatten_packed_metadata, which perform one host read each, and the
 *     status readers.
 *   - Arguments are checked on the host before anything is launched; a
 *     failed check returns a status and launches nothing. The return value of
 *     an asynchronous call can only carry what the host checks: what the
 *     attention kernels find later (a cu_seqlens that fails the device-side
 *     layout check, a pipeline wait that gave up) is recorded in the status
 *     word at the head of the call's workspace, which pe_read_device_status
 *     reads back (pe_read_noalloc_status for the allocation-free forward).
 *   - Rows are row-major and tightly packed. bf16 is IEEE bfloat16; fp32 is
 *     IEEE binary32. Accumulation is always fp32.
 *   - Kernels run on the current CUDA device, which must be compute
 *     capability 10.3 (sm_103a); any other device gives PE_ERR_UNSUPPORTED.
 */
#ifndef PE_H_
#define PE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; NULL selects the legacy default stream. */
typedef struct CUstream_st* pe_stream_t;

typedef enum pe_status {
  PE_OK = 0,
  PE_ERR_INVALID_ARG = 1,    /* null pointer, negative size, bad scale, ...        */
  PE_ERR_BAD_LENGTH = 2,     /* a sequence length < 1 or > max_seq_len             */
  PE_ERR_OVERFLOW = 3,       /* token count (or tile count) does not fit in int32  */
  PE_ERR_UNSUPPORTED = 4,    /* head_dim, dtype, alignment or device not supported */
  PE_ERR_WORKSPACE = 5,      /* workspace null or smaller than *_workspace_size     */
  PE_ERR_CUDA = 6,           /* a CUDA runtime call failed                         */
  PE_ERR_DEVICE_TIMEOUT = 7  /* a kernel gave up waiting on its own pipeline
                                (device status word only, never a return value) */
} pe_status;

typedef enum pe_dtype { PE_BF16 = 0, PE_FP32 = 1 } pe_dtype;

/* Text for a status code; never NULL. */
const char* pe_status_string(int status);

/* Version of this ABI (incremented when an entry point is added or changed;
 * 2 added pe_packed_attention_fwd_local, pe_packed_attention_bwd_local,
 * pe_rows_workspace_size, pe_pack_document_ids, pe_flatten_packed_metadata,
 * pe_packed_positions, pe_rope_packed, pe_layernorm, pe_geglu, pe_upload_packed;
 * later additions within 2: pe_download_padded; 3 added the device-side
 * layout check of the attention calls, pe_set_wait_limit_ns and
 * pe_read_noalloc_status; later additions within 3:
 * pe_attention_kernel_local). */
int pe_abi_version(void);

/* ------------------------------------------------------------------------
 * pack_sequences  (module docstring, "Data flow of a packed forward",
 * "Constraints" and "Example": lengths [3,1,2], max_seq_len 3 give
 * flat_index [0,1,2,3,6,7]; packing reads the token count back to the host
 * once, and nothing else syncs).
 *
 *   cu_seqlens[0] = 0, cu_seqlens[i+1] = cu_seqlens[i] + lengths[i]
 *   flat_index[cu_seqlens[i] + j] = i * max_seq_len + j   for 0 <= j < lengths[i]
 *
 * lengths:      int32 [num_sequences], device.
 * flat_index:   int64, device, capacity >= num_sequences * max_seq_len entries
 *               (a bound the host knows, so no allocation waits on the count);
 *               the first *num_tokens entries are written.
 * cu_seqlens:   int32 [num_sequences + 1], device.
 * num_tokens:   HOST out: the token count N. This is the single device-to-host
 *               read; the call synchronizes `stream` to perform it.
 * workspace:    device, >= pe_pack_workspace_size() bytes.
 * Errors: PE_ERR_BAD_LENGTH if some length is < 1 or > max_seq_len (detected
 * on the device, reported through the same host read; flat_index is then not
 * written), PE_ERR_OVERFLOW if N >= 2^31. num_sequences == 0 gives N = 0 and
 * cu_seqlens = [0].
 * ------------------------------------------------------------------------ */
size_t pe_pack_workspace_size(int32_t num_sequences);
pe_status pe_pack_sequences(const int32_t* lengths, int32_t num_sequences, int32_t max_seq_len,
                            int64_t* flat_index, int32_t* cu_seqlens, int64_t* num_tokens,
                            void* workspace, size_t workspace_bytes, pe_stream_t stream);

/* ------------------------------------------------------------------------
 * Padded -> packed gather: packed[t, :] = padded[flat_index[t], :]
 * (module docstring, "Data flow of a packed forward": grid.flatten()[flat_index]).
 *
 * padded:     device memory, or pinned host memory mapped into the device
 *             address space (cudaHostAlloc / cudaHostRegister memory, mapped
 *             by default under unified addressing): the kernel then reads only
 *             the real rows across the host link, with no separate copy of
 *             the padded grid. Rows of row_bytes bytes (any number of rows;
 *             every flat_index value must name one of them).
 * flat_index: int64 [num_tokens], device (from pe_pack_sequences).
 * packed:     device, [num_tokens] rows of row_bytes bytes.
 * 16-byte vector copies when row_bytes and both pointers are 16-byte aligned,
 * 4-byte copies when 4-byte aligned, byte copies otherwise (all on the GPU).
 * ------------------------------------------------------------------------ */
pe_status pe_gather_packed(const void* padded, const int64_t* flat_index, int64_t num_tokens,
                           int64_t row_bytes, void* packed, pe_stream_t stream);

/* ------------------------------------------------------------------------
 * Host padded grid -> packed device buffer with the copy engines: the same
 * result as pe_gather_packed on a grid in host memory, for callers that hold
 * the lengths on the host. Sequence i's rows are one contiguous run in both
 * layouts (padded rows i*max_seq_len .. +L_i-1, packed rows cu_i .. +L_i-1),
 * so the call enqueues one asynchronous host-to-device copy per sequence on
 * `stream` and returns: only real rows cross the host link, and no kernel
 * runs, so the copies overlap kernels running on other streams.
 *
 * padded_host:  host memory (pinned for asynchronous copies), [num_sequences *
 *               max_seq_len] rows of row_bytes bytes.
 * lengths_host: int32 [num_sequences], host; 1 <= L_i <= max_seq_len, else
 *               PE_ERR_BAD_LENGTH before any copy; PE_ERR_OVERFLOW if
 *               sum L_i >= 2^31.
 * packed:       device, [sum L_i] rows of row_bytes bytes.
 * The host buffers must stay valid until the copies complete.
 * ------------------------------------------------------------------------ */
pe_status pe_upload_packed(const void* padded_host, const int32_t* lengths_host,
                           int32_t num_sequences, int32_t max_seq_len, int64_t row_bytes,
                           void* packed, pe_stream_t stream);

/* ------------------------------------------------------------------------
 * Packed device buffer -> host padded grid with the copy engines: the real
 * rows of pe_scatter_padded's result (function _padded_packed_attention,
 * to_dense_batch) written into a grid in host memory, for callers that hold
 * the lengths on the host. One asynchronous device-to-host copy per sequence
 * (packed rows cu_i .. +L_i-1 to padded rows i*max_seq_len .. +L_i-1) on
 * `stream`; no kernel runs, and only real rows cross the host link.
 *
 * Pad rows (j >= L_i) of padded_host are NOT written: to_dense_batch's zero
 * fill is the caller's, once per layout (e.g. a host grid allocated zeroed and
 * reused for batches of the same lengths).
 *
 * packed:       device, [sum L_i] rows of row_bytes bytes.
 * lengths_host: int32 [num_sequences], host; 1 <= L_i <= max_seq_len, else
 *               PE_ERR_BAD_LENGTH before any copy; PE_ERR_OVERFLOW if
 *               sum L_i >= 2^31.
 * padded_host:  host memory (pinned for asynchronous copies), [num_sequences *
 *               max_seq_len] rows of row_bytes bytes.
 * The rows are on the host once `stream` has passed the copies.
 * ------------------------------------------------------------------------ */
pe_status pe_download_padded(const void* packed, const int32_t* lengths_host,
                             int32_t num_sequences, int32_t max_seq_len, int64_t row_bytes,
                             void* padded_host, pe_stream_t stream);

/* ------------------------------------------------------------------------
 * Packed -> padded scatter with zero fill (function _padded_packed_attention,
 * which unpacks with to_dense_batch, fill value 0):
 *   padded[i*max_seq_len + j, :] = j < L_i ? packed[cu_seqlens[i] + j, :] : 0
 *
 * packed:     device, [cu_seqlens[num_sequences]] rows of row_bytes bytes.
 * cu_seqlens: int32 [num_sequences + 1], device (trusted output of pack).
 * padded:     device memory, or pinned host memory mapped into the device
 *             address space (then the kernel writes the rows across the host
 *             link, with no separate copy back): [num_sequences * max_seq_len]
 *             rows; every row is written.
 * ------------------------------------------------------------------------ */
pe_status pe_scatter_padded(const void* packed, const int32_t* cu_seqlens, int32_t num_sequences,
                            int32_t max_seq_len, int64_t row_bytes, void* padded,
                            pe_stream_t stream);

/* ------------------------------------------------------------------------
 * Packed rows: padded [B, S] layouts that hold several documents per row
 * (page "nemo_automodel.components.models.common.packing"), turned into the
 * flat_index / cu_seqlens layout that the gather, scatter and attention calls
 * consume. Documents follow each other row by row; flat_index holds indices
 * into the padded [B, S] layout (row * S + position).
 *
 * pe_pack_document_ids: an indexed packing mask document_ids [B, S] int32
 *   (function is_indexed_packed_mask: document i of a row, 1-based, marked i;
 *   padding 0), e.g. the row [1,1,1,2,2,3,3,0,0] gives flat_index 0..6 and
 *   cu_seqlens [0,3,5,7].
 * pe_flatten_packed_metadata: function flatten_packed_sequence_metadata's
 *   inputs, row-local token indices token_indices [B, S] int64 and row-local
 *   cumulative lengths row_cu_seqlens [B, M1] int32, both -1 padded.
 * Readings where the page is silent: padding is trailing in every row;
 * documents are non-empty and numbered 1, 2, ... in order within a row;
 * row-local boundaries start at 0, increase strictly and end at the row's
 * token count; token indices lie in [0, S). Any other layout returns
 * PE_ERR_INVALID_ARG (nothing is written to the outputs then); a token count of
 * 2^31 or more returns PE_ERR_OVERFLOW.
 * Outputs (device, caller-owned): flat_index with room for B*S entries,
 * cu_seqlens with room for B*S + 1 (document ids) or B*(M1-1) + 1 (row
 * boundaries) entries; *num_tokens and *num_documents are written on the
 * host: each call reads 16 bytes back once and synchronizes the stream.
 * Workspace: pe_rows_workspace_size(B) bytes, 16-byte aligned, device.
 * ------------------------------------------------------------------------ */
size_t pe_rows_workspace_size(int32_t num_rows);
pe_status pe_pack_document_ids(const int32_t* document_ids, int32_t num_rows,
                               int32_t sequence_length, int64_t* flat_index,
                               int32_t* cu_seqlens, int64_t* num_tokens,
                               int32_t* num_documents, void* workspace, size_t workspace_bytes,
                               pe_stream_t stream);
pe_status pe_flatten_packed_metadata(const int64_t* token_indices, const int32_t* row_cu_seqlens,
                                     int32_t num_rows, int32_t sequence_length,
                                     int32_t row_cu_columns, int64_t* flat_index,
                                     int32_t* cu_seqlens, int64_t* num_tokens,
                                     int32_t* num_documents, void* workspace,
                                     size_t workspace_bytes, pe_stream_t stream);

/* ------------------------------------------------------------------------
 * Packed attention forward (function packed_attention and the custom op
 * gigl::varlen_attention, which returns the output and the log-sum-exp).
 *
 * For every sequence i, head h and query row r:
 *   O[r,h,:]  = sum_j softmax_j(scale * q[r,h,:] . k[j,h,:]) v[j,h,:]
 *   lse[h,r]  = log sum_j exp(scale * q[r,h,:] . k[j,h,:])      (natural log)
 * with j over the keys of sequence i only (cu_seqlens[i] <= j < cu_seqlens[i+1]).
 *
 * query_is_first_token = 0: q and out are [num_tokens, H, D]; row r of
 *   sequence i is token cu_seqlens[i] + r.
 * query_is_first_token = 1: q and out are [num_sequences, H, D]; q[i] is the
 *   query of sequence i (its first token, as the caller sliced it), and out[i]
 *   equals row cu_seqlens[i] of the full-mode output.
 * k, v: [num_tokens, H, D]. dtype applies to q, k, v and out.
 * lse: fp32 [H, Nq] (Nq = num_tokens or num_sequences), or NULL to skip it.
 * cu_seqlens: int32 [num_sequences + 1], device, normally the output of
 *   pe_pack_sequences. Before any kernel reads q, k or v through it, the call
 *   checks it on the device: cu_seqlens[0] = 0, cu_seqlens[num_sequences] =
 *   num_tokens and 1 <= cu_seqlens[i+1] - cu_seqlens[i] <= max_seq_len (every
 *   sequence non-empty, so no packed layout can make one sequence attend
 *   across another's tokens or past the buffers; page
 *   "nemo_automodel.components.models.common.packing" fails such layouts
 *   loudly too). A layout that fails records PE_ERR_BAD_LENGTH (a length out
 *   of range) or PE_ERR_INVALID_ARG (a wrong first or last entry) in the
 *   workspace status word, and the call then computes nothing: out and lse
 *   are left as they were. Only the num_sequences + 1 entries are read.
 * scale: finite and > 0 (1/sqrt(D) is the pages' default).
 * head_dim: a multiple of 8 (the module docstring's "Constraints" require
 *   it for the aligned kernels), at most 128. Full attention runs on the
 *   tcgen05 tensor cores for bf16 with head_dim 64 or 128 (forward and
 *   backward) and for fp32 with head_dim 64 (forward; fp32 operands split
 *   into bf16 hi and lo parts, three products each, fp32 accumulation);
 *   other shapes run on the CUDA cores.
 * All tensor pointers 16-byte aligned.
 * workspace: device, >= pe_attention_workspace_size(...) bytes. Its first 4
 *   bytes receive a device-side status (PE_OK, PE_ERR_BAD_LENGTH or
 *   PE_ERR_INVALID_ARG from the layout check, or PE_ERR_DEVICE_TIMEOUT),
 *   readable with pe_read_device_status after the call. In first-token mode
 *   the reported size includes room for partial softmax states, so that long
 *   sequences can be spread over several CTAs: when a token row
 *   (num_heads*head_dim elements) is 512, 1024, ..., 4096 bytes and head_dim
 *   is 32, 64 or 128, the token range is cut into equal chunks of whole rows
 *   (one CTA each) and each chunk keeps up to two partial states per head;
 *   otherwise, with max_seq_len > 1024, each (sequence, head) is split into
 *   1024-key chunks. A workspace without that room (but large enough
 *   otherwise) is accepted and runs one CTA per sequence and head.
 *   For a first-token backward (backward = 1) the reported size likewise
 *   includes room for per-chunk dq sums when the token row is 512, 1024, ...
 *   bytes (bf16 rows up to 3072 bytes, fp32 rows up to 4096) and head_dim
 *   is 32, 64 or 128: the token
 *   range is then cut into equal chunks, dk and dv rows are written as k and
 *   v stream through, and sequences crossing chunk edges have their dq sums
 *   added in chunk order. Without that room the backward runs per sequence
 *   and head on the CUDA cores.
 * ------------------------------------------------------------------------ */
size_t pe_attention_workspace_size(pe_dtype dtype, int32_t num_sequences, int64_t num_tokens,
                                   int32_t num_heads, int32_t head_dim, int32_t max_seq_len,
                                   int query_is_first_token, int backward);

pe_status pe_packed_attention_fwd(pe_dtype dtype, int32_t num_sequences, int64_t num_tokens,
                                  int32_t num_heads, int32_t head_dim, int32_t max_seq_len,
                                  const void* q, const void* k, const void* v,
                                  const int32_t* cu_seqlens, float scale, int query_is_first_token,
                                  void* out, float* lse, void* workspace, size_t workspace_bytes,
                                  pe_stream_t stream);

/* ------------------------------------------------------------------------
 * Packed attention backward (the custom op gigl::varlen_attention_backward,
 * which takes the saved q, k, v, output and log-sum-exp and returns the
 * gradients in q, k and v). With P = softmax(scale q k^T) per sequence/head:
 *   Delta_r = dO_r . O_r,  dS = P o (dO v^T - Delta),
 *   dq = scale dS k,  dk = scale dS^T q,  dv = P^T dO.
 * Arguments as in the forward; out and lse are that forward's results for
 * the same inputs; dout, dq are shaped like q; dk, dv like k. Delta is formed
 * from out as passed (a bf16 out is the exact output rounded). Every element
 * of dq, dk, dv is written. The result is bitwise deterministic run to run
 * (no floating-point atomics).
 * ------------------------------------------------------------------------ */
pe_status pe_packed_attention_bwd(pe_dtype dtype, int32_t num_sequences, int64_t num_tokens,
                                  int32_t num_heads, int32_t head_dim, int32_t max_seq_len,
                                  const void* q, const void* k, const void* v,
                                  const int32_t* cu_seqlens, float scale, int query_is_first_token,
                                  const void* out, const float* lse, const void* dout,
                                  void* dq, void* dk, void* dv,
                                  void* workspace, size_t workspace_bytes, pe_stream_t stream);

/* ------------------------------------------------------------------------
 * Local (sliding-window) packed attention: the same forward and backward with
 * each query restricted to a window of key positions around its own. The
 * pages name the mode without defining it (packed-encoders README: the packed
 * kernel's "global or local-64 attention" for ModernBERT geometry, and
 * FlashAttention's sliding-window pruning); here the key at position j of a
 * sequence is visible from the query at position r of the same sequence iff
 *     r - window_left <= j <= r + window_right,
 * positions counted from the sequence start, a first-token query sitting at
 * position 0. A negative bound is unbounded, so (-1, -1) is exactly
 * pe_packed_attention_fwd / _bwd; ModernBERT's local-64 is (64, 64). Every
 * query sees at least its own key. Kernels visit only the key blocks inside
 * the band, so the work per query is O(window) rather than O(length).
 * All other arguments, layouts, workspace sizes and errors are those of
 * pe_packed_attention_fwd / pe_packed_attention_bwd (out and lse passed to
 * the backward must come from the forward with the same window).
 * ------------------------------------------------------------------------ */
pe_status pe_packed_attention_fwd_local(pe_dtype dtype, int32_t num_sequences,
                                        int64_t num_tokens, int32_t num_heads, int32_t head_dim,
                                        int32_t max_seq_len, const void* q, const void* k,
                                        const void* v, const int32_t* cu_seqlens, float scale,
                                        int32_t window_left, int32_t window_right,
                                        int query_is_first_token, void* out, float* lse,
                                        void* workspace, size_t workspace_bytes,
                                        pe_stream_t stream);
pe_status pe_packed_attention_bwd_local(pe_dtype dtype, int32_t num_sequences,
                                        int64_t num_tokens, int32_t num_heads, int32_t head_dim,
                                        int32_t max_seq_len, const void* q, const void* k,
                                        const void* v, const int32_t* cu_seqlens, float scale,
                                        int32_t window_left, int32_t window_right,
                                        int query_is_first_token, const void* out,
                                        const float* lse, const void* dout, void* dq, void* dk,
                                        void* dv, void* workspace, size_t workspace_bytes,
                                        pe_stream_t stream);

/* ------------------------------------------------------------------------
 * The packed encoder layer tail (page "packed-encoders 0.1.0": fused
 * LayerNorm / residual-LayerNorm / RoPE / GeGLU kernels on the flat token
 * buffer, the token count a runtime grid dimension; position ids restart at
 * every sequence, section "Fully packed execution"). Formulas as in
 * ModernBERT. Every call is asynchronous on `stream`, allocates nothing and
 * reads nothing back, so a layer tail can be captured in a CUDA graph. Tensors
 * are contiguous device memory in the I/O dtype (bf16 or fp32); arithmetic is
 * fp32.
 *
 * pe_packed_positions: positions[t] = t - cu_seqlens[i] for the sequence i
 *   holding token t (int32 [num_tokens]); the README's lengths 5, 3, 8 give
 *   0 1 2 3 4 0 1 2 0 1 2 3 4 5 6 7.
 * pe_rope_packed: split-half rotary embedding in place on q [N, q_heads, D]
 *   and k [N, k_heads, D] (k may be NULL): for i < D/2 and
 *   a = positions[t] * theta^(-2i/D), (x[i], x[i+D/2]) becomes
 *   (x[i] cos a - x[i+D/2] sin a, x[i+D/2] cos a + x[i] sin a). D even, <= 256,
 *   theta > 1 (ModernBERT: 160000 for global layers, 10000 for local ones).
 *   Angles are reduced modulo 2 pi in double precision.
 * pe_layernorm: y = (h - mean(h)) / sqrt(var(h) + eps) * weight (+ bias) per
 *   row of C channels, biased variance, bias nullable; h = x, or with a
 *   residual h = x + residual rounded to the I/O dtype, written to
 *   residual_out when that is non-NULL.
 * pe_geglu: y [N, F] = gelu(x[:, :F]) * x[:, F:] for x [N, 2F], exact (erf)
 *   GELU.
 * Errors: PE_ERR_INVALID_ARG for negative sizes, NULL required pointers, odd
 * D, theta <= 1 or eps <= 0; PE_ERR_UNSUPPORTED for other dtypes or devices.
 * ------------------------------------------------------------------------ */
pe_status pe_packed_positions(const int32_t* cu_seqlens, int32_t num_sequences,
                              int64_t num_tokens, int32_t* positions, pe_stream_t stream);
pe_status pe_rope_packed(pe_dtype dtype, void* q, int32_t q_heads, void* k, int32_t k_heads,
                         const int32_t* positions, int64_t num_tokens, int32_t head_dim,
                         double theta, pe_stream_t stream);
pe_status pe_layernorm(pe_dtype dtype, const void* x, const void* residual, const void* weight,
                       const void* bias, int64_t num_tokens, int32_t channels, float eps, void* y,
                       void* residual_out, pe_stream_t stream);
pe_status pe_geglu(pe_dtype dtype, const void* x, int64_t num_tokens, int32_t features, void* y,
                   pe_stream_t stream);

/* Name of the kernel family that pe_packed_attention_fwd (backward = 0) or
 * pe_packed_attention_bwd (backward = 1) runs for these arguments (full
 * attention) on an sm_103a device: "tcgen05_bf16_d64", "tcgen05_bf16_d128",
 * "tcgen05_f32_d64", "simt_ffma", "first_token_gemv", "simt_ffma_bwd",
 * "tcgen05_bf16_d64_bwd", "tcgen05_bf16_d128_bwd", "first_token_bwd", or
 * "unsupported". The two first-token families cover both of their forms
 * (streaming whole token rows when the row shape and workspace allow it, per
 * sequence and head otherwise). A static string; never NULL. */
const char* pe_attention_kernel(pe_dtype dtype, int32_t head_dim, int query_is_first_token,
                                int backward);

/* The same for pe_packed_attention_fwd_local / pe_packed_attention_bwd_local
 * with this window (window_left, window_right, max_seq_len as in those calls;
 * a window that reaches every key is full attention). Local attention changes
 * the family only for the forward of full-query calls: bf16 head_dim 64 keeps
 * its tensor-core family ("tcgen05_bf16_d64", a local instance of the same
 * kernel), every other forward runs "simt_ffma"; the backward families and
 * the first-token families are those of pe_attention_kernel. max_seq_len < 1:
 * "unsupported". A static string; never NULL. */
const char* pe_attention_kernel_local(pe_dtype dtype, int32_t head_dim, int32_t max_seq_len,
                                      int32_t window_left, int32_t window_right,
                                      int query_is_first_token, int backward);

/* ------------------------------------------------------------------------
 * Allocation-free forward. The pages have no counterpart to this call; it
 * exists for callers that cannot give the library a workspace: a host
 * runtime that owns every device allocation through its own fixed pool and
 * exposes no scratch API (a serving process, a framework plugin), or a
 * latency-critical loop where cudaMalloc/cudaFree would add implicit
 * device-wide synchronisation.
 *
 * Same arguments and results as pe_packed_attention_fwd without the
 * workspace. The scratch (status word and tile plan, and a first-token
 * forward's partial softmax states when they fit; otherwise that forward runs
 * one CTA per sequence and head) lives in a 512 KiB device array inside the
 * library that every GPU loading it holds until the process exits;
 * num_sequences may be at most 65536, larger batches return PE_ERR_WORKSPACE
 * before anything runs. The call allocates nothing.
 * The first call on a device (with that device current) looks up the
 * array's device address; make that first call before any stream capture.
 * All calls on a device share the array and it keeps the last call's
 * contents (the call clears what must start at zero itself): calls whose
 * executions overlap on the GPU race and must be serialised by the caller.
 * The array's address is cached per device for the life of the process; the
 * cache does not survive cudaDeviceReset (call nothing here after one).
 * The device-side status of the last call (the layout check and the bounded
 * pipeline waits) sits in the array too: pe_read_noalloc_status reads it.
 * ------------------------------------------------------------------------ */
pe_status pe_packed_attention_fwd_noalloc(pe_dtype dtype, int32_t num_sequences,
                                          int64_t num_tokens, int32_t num_heads, int32_t head_dim,
                                          int32_t max_seq_len, const void* q, const void* k,
                                          const void* v, const int32_t* cu_seqlens, float scale,
                                          int query_is_first_token, void* out, float* lse,
                                          pe_stream_t stream);

/* Synchronizes `stream` and returns the device-side status that the last
 * attention call on `workspace` left in its first 4 bytes (PE_OK when the
 * layout passed its check and every pipeline wait completed). */
pe_status pe_read_device_status(const void* workspace, pe_stream_t stream);

/* The same for pe_packed_attention_fwd_noalloc: synchronizes `stream` and
 * returns the device-side status of the last allocation-free call on the
 * current device (copied from the library's static array into host stack
 * memory; nothing is allocated). PE_ERR_CUDA if the array's address cannot be
 * looked up. */
pe_status pe_read_noalloc_status(pe_stream_t stream);

/* Sets the time limit of every bounded pipeline wait in the kernels launched
 * after this call, in nanoseconds, for the whole process; 0 restores the
 * default of 2 s. Returns the previous limit. A wait that exceeds the limit
 * makes its kernel record PE_ERR_DEVICE_TIMEOUT in the status word, finish
 * the copies and tensor-core operations it has in flight (each such drain
 * wait is bounded by 2 s whatever this limit), free its tensor memory and
 * exit, leaving the call's outputs incomplete; the context stays usable. A
 * diagnostic control: a limit far below a kernel's normal waits turns a valid
 * call into a reported timeout, which is how the timeout path is tested. */
uint64_t pe_set_wait_limit_ns(uint64_t ns);

#ifdef __cplusplus
}
#endif

#endif /* PE_H_ */
