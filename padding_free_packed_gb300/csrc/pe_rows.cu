// Packed rows: padded [B, S] layouts that hold several documents per row, as
// produced by packing collaters, turned into the flat token stream and
// cu_seqlens that the rest of the library consumes (page
// "nemo_automodel.components.models.common.packing"):
//   - an indexed packing mask marks document i of a row (1-based) with the
//     integer i and padding with 0 (function is_indexed_packed_mask);
//   - flatten_packed_sequence_metadata takes row-local token indices [B, S]
//     and row-local cumulative lengths [B, M+1], both -1 padded, and returns
//     flat indices into the padded [B, S] layout and flat cu_seqlens, failing
//     on inconsistent layouts, boundaries or token counts.
// Readings: padding is trailing in both layouts; documents are non-empty and
// numbered 1, 2, ... in order within a row; row-local boundaries start at 0,
// increase strictly and end at the row's token count; row-local token indices
// lie in [0, S). Rows follow each other in the flat stream.
//
// Three kernels and one host read, like pack_sequences: a validating count
// over (row, chunk of 2048 positions) pairs that adds each chunk's tokens and
// document starts into its row's totals (integer atomics: exact in any order),
// a single-CTA scan of the per-row totals, and a fill over the same chunks;
// the host then copies back 16 bytes.
#include "pe_common.cuh"

namespace pe {

namespace {

constexpr int kRowThreads = 256;
constexpr int kScanThreads = 1024;
constexpr int32_t kChunk = 2048;   // row positions per CTA work item

struct RowsResult {
  long long num_tokens;
  int32_t num_docs;
  int32_t status;
};

// Workspace: the result word, then per row the token and document counts and
// their exclusive prefixes.
struct RowsWorkspace {
  RowsResult* result;
  int32_t* n;          // [B] tokens per row
  int32_t* d;          // [B] documents per row
  int64_t* tok_off;    // [B] first flat token of the row
  int64_t* doc_off;    // [B] first document of the row
};

size_t round16(size_t x) { return (x + 15) / 16 * 16; }

size_t rows_ws_bytes(int32_t B) {
  return 16 + 2 * round16(4 * (size_t)B) + 2 * round16(8 * (size_t)B);
}

RowsWorkspace rows_ws_view(void* ws, int32_t B) {
  char* p = static_cast<char*>(ws);
  RowsWorkspace w;
  w.result = reinterpret_cast<RowsResult*>(p);
  p += 16;
  w.n = reinterpret_cast<int32_t*>(p);
  p += round16(4 * (size_t)B);
  w.d = reinterpret_cast<int32_t*>(p);
  p += round16(4 * (size_t)B);
  w.tok_off = reinterpret_cast<int64_t*>(p);
  p += round16(8 * (size_t)B);
  w.doc_off = reinterpret_cast<int64_t*>(p);
  return w;
}

__device__ __forceinline__ void flag_invalid(RowsResult* r) {
  atomicCAS(&r->status, (int32_t)PE_OK, (int32_t)PE_ERR_INVALID_ARG);
}

// Block-wide sum of two counters (blockDim.x == kRowThreads).
__device__ __forceinline__ void block_sum2(int& a, int& b, int* sh) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    a += __shfl_xor_sync(0xffffffffu, a, off);
    b += __shfl_xor_sync(0xffffffffu, b, off);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    sh[warp] = a;
    sh[32 + warp] = b;
  }
  __syncthreads();
  a = b = 0;
  for (int w = 0; w < kRowThreads / 32; ++w) {
    a += sh[w];
    b += sh[32 + w];
  }
  __syncthreads();
}

// Indexed packing mask: per row, checks every position against its left
// neighbour (a document continues or the next one starts; padding only at the
// end) and counts tokens and document starts.
__global__ void __launch_bounds__(kRowThreads)
doc_ids_count_kernel(const int32_t* __restrict__ ids, int32_t B, int32_t S, RowsWorkspace w) {
  __shared__ int sh[64];
  const int32_t chunks = (S + kChunk - 1) / kChunk;
  for (int64_t item = blockIdx.x; item < (int64_t)B * chunks; item += gridDim.x) {
    const int64_t b = item / chunks;
    const int32_t j0 = (int32_t)(item - b * chunks) * kChunk, j1 = min(j0 + kChunk, S);
    const int32_t* row = ids + b * (int64_t)S;
    int tokens = 0, starts = 0;
    bool bad = false;
    for (int32_t j = j0 + threadIdx.x; j < j1; j += kRowThreads) {
      const int32_t id = __ldg(row + j);
      const int32_t left = j > 0 ? __ldg(row + j - 1) : 0;
      if (id < 0) bad = true;
      if (id > 0) {
        ++tokens;
        if (j == 0) {
          bad |= id != 1;
          ++starts;
        } else if (left == 0) {
          bad = true;                       // a document after padding
        } else if (id == left + 1) {
          ++starts;
        } else if (id != left) {
          bad = true;                       // a skipped or repeated document number
        }
      }
    }
    if (bad) flag_invalid(w.result);
    block_sum2(tokens, starts, sh);
    if (threadIdx.x == 0) {
      atomicAdd(w.n + b, tokens);
      atomicAdd(w.d + b, starts);
    }
  }
}

// Row-local token indices and cumulative lengths (-1 padded): per row, counts
// the tokens and documents and checks the layout rules.
// The check that a row's last boundary equals its token count needs the row
// total, so it runs in the scan.
__global__ void __launch_bounds__(kRowThreads)
nemo_rows_count_kernel(const int64_t* __restrict__ tok, const int32_t* __restrict__ rcu,
                       int32_t B, int32_t S, int32_t M1, RowsWorkspace w) {
  __shared__ int sh[64];
  const int32_t chunks = (S + kChunk - 1) / kChunk;
  for (int64_t item = blockIdx.x; item < (int64_t)B * chunks; item += gridDim.x) {
    const int64_t b = item / chunks;
    const int32_t chunk = (int32_t)(item - b * chunks);
    const int32_t j0 = chunk * kChunk, j1 = min(j0 + kChunk, S);
    const int64_t* trow = tok + b * (int64_t)S;
    const int32_t* crow = rcu + b * (int64_t)M1;
    int tokens = 0, bounds = 0;
    bool bad = false;
    for (int32_t j = j0 + threadIdx.x; j < j1; j += kRowThreads) {
      const int64_t t = __ldg(trow + j);
      if (t == -1) continue;
      ++tokens;
      bad |= t < 0 || t >= S;
      bad |= j > 0 && __ldg(trow + j - 1) == -1;   // padding not trailing
    }
    for (int32_t k = threadIdx.x; chunk == 0 && k < M1; k += kRowThreads) {  // boundaries once per row
      const int32_t c = __ldg(crow + k);
      if (k == 0) {
        bad |= c != 0;
        continue;
      }
      if (c == -1) continue;
      ++bounds;
      const int32_t prev = __ldg(crow + k - 1);
      bad |= prev == -1 || c <= prev;              // padding not trailing, or an empty document
    }
    if (bad) flag_invalid(w.result);
    block_sum2(tokens, bounds, sh);
    if (threadIdx.x == 0) {
      atomicAdd(w.n + b, tokens);
      atomicAdd(w.d + b, bounds);
    }
  }
}

// Inclusive block-wide scan of one int64 per thread (blockDim.x == 1024).
__device__ __forceinline__ long long scan1024(long long x, long long* warp_sums,
                                              long long& block_total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    long long s = warp_sums[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, s, off);
      if (lane >= off) s += y;
    }
    warp_sums[lane] = s;
  }
  __syncthreads();
  const long long prefix = warp > 0 ? warp_sums[warp - 1] : 0;
  block_total = warp_sums[31];
  __syncthreads();
  return x + prefix;
}

// Exclusive prefixes of the per-row counts; totals and the closing boundary.
// With row-local boundaries (rcu non-null) it also checks that each row's last
// boundary equals the row's token count.
__global__ void __launch_bounds__(kScanThreads)
rows_scan_kernel(int32_t B, RowsWorkspace w, const int32_t* __restrict__ rcu, int32_t M1,
                 int32_t* __restrict__ cu_seqlens) {
  __shared__ long long warp_sums[32];
  long long carry_n = 0, carry_d = 0;
  for (int64_t base = 0; base < B; base += kScanThreads) {
    const int64_t b = base + threadIdx.x;
    const long long n = b < B ? w.n[b] : 0, d = b < B ? w.d[b] : 0;
    // d < M1 always: it counts boundary entries after the first of M1.
    if (rcu && b < B && __ldg(rcu + b * (int64_t)M1 + d) != n) flag_invalid(w.result);
    long long tn, td;
    const long long in = scan1024(n, warp_sums, tn);
    const long long id = scan1024(d, warp_sums, td);
    if (b < B) {
      w.tok_off[b] = carry_n + in - n;
      w.doc_off[b] = carry_d + id - d;
    }
    carry_n += tn;
    carry_d += td;
  }
  __syncthreads();   // every row's check has flagged before the status is read
  if (threadIdx.x == 0) {
    RowsResult* r = w.result;
    if (r->status == PE_OK && carry_n >= (1LL << 31)) r->status = PE_ERR_OVERFLOW;
    r->num_tokens = carry_n;
    r->num_docs = (int32_t)carry_d;
    if (r->status == PE_OK) cu_seqlens[carry_d] = (int32_t)carry_n;
  }
}

__global__ void __launch_bounds__(kRowThreads)
doc_ids_fill_kernel(const int32_t* __restrict__ ids, int32_t B, int32_t S, RowsWorkspace w,
                    int64_t* __restrict__ flat_index, int32_t* __restrict__ cu_seqlens) {
  if (w.result->status != PE_OK) return;
  const int32_t chunks = (S + kChunk - 1) / kChunk;
  for (int64_t item = blockIdx.x; item < (int64_t)B * chunks; item += gridDim.x) {
    const int64_t b = item / chunks;
    const int32_t j0 = (int32_t)(item - b * chunks) * kChunk;
    const int32_t* row = ids + b * (int64_t)S;
    const int32_t n = w.n[b], j1 = min(j0 + kChunk, n);
    const int64_t t0 = w.tok_off[b], d0 = w.doc_off[b];
    for (int32_t j = j0 + threadIdx.x; j < j1; j += kRowThreads) {  // tokens: the first n positions
      flat_index[t0 + j] = b * (int64_t)S + j;
      const int32_t id = __ldg(row + j);
      if (j == 0 || __ldg(row + j - 1) != id) cu_seqlens[d0 + id - 1] = (int32_t)(t0 + j);
    }
  }
}

__global__ void __launch_bounds__(kRowThreads)
nemo_rows_fill_kernel(const int64_t* __restrict__ tok, const int32_t* __restrict__ rcu,
                      int32_t B, int32_t S, int32_t M1, RowsWorkspace w,
                      int64_t* __restrict__ flat_index, int32_t* __restrict__ cu_seqlens) {
  if (w.result->status != PE_OK) return;
  const int32_t chunks = (S + kChunk - 1) / kChunk;
  for (int64_t item = blockIdx.x; item < (int64_t)B * chunks; item += gridDim.x) {
    const int64_t b = item / chunks;
    const int32_t chunk = (int32_t)(item - b * chunks);
    const int32_t n = w.n[b], d = w.d[b];
    const int64_t t0 = w.tok_off[b], d0 = w.doc_off[b];
    for (int32_t i = chunk * kChunk + threadIdx.x; i < min(chunk * kChunk + kChunk, n);
         i += kRowThreads)
      flat_index[t0 + i] = b * (int64_t)S + __ldg(tok + b * (int64_t)S + i);
    for (int32_t k = threadIdx.x; chunk == 0 && k < d; k += kRowThreads)
      cu_seqlens[d0 + k] = (int32_t)(t0 + __ldg(rcu + b * (int64_t)M1 + k));
  }
}

// Launch sizes and the host read shared by both entry points.
unsigned row_blocks(int32_t B, int32_t S) {
  const int64_t items = (int64_t)B * ((S + kChunk - 1) / kChunk);
  const int64_t cap = (int64_t)device_sm_count() * 8;
  return (unsigned)(items < cap ? items : cap);
}

// Zeroes the result word and the per-row totals the count kernels add into.
pe_status clear_counts(const RowsWorkspace& w, int32_t B, cudaStream_t stream) {
  PE_CUDA_TRY(cudaMemsetAsync(w.result, 0, sizeof(RowsResult), stream));
  if (B > 0)
    PE_CUDA_TRY(cudaMemsetAsync(w.n, 0, reinterpret_cast<char*>(w.tok_off) -
                                            reinterpret_cast<char*>(w.n), stream));
  return PE_OK;
}

pe_status read_result(const RowsWorkspace& w, int64_t* num_tokens, int32_t* num_documents,
                      cudaStream_t stream) {
  RowsResult host;
  PE_CUDA_TRY(cudaMemcpyAsync(&host, w.result, sizeof(host), cudaMemcpyDeviceToHost, stream));
  PE_CUDA_TRY(cudaStreamSynchronize(stream));
  if (host.status != PE_OK) return (pe_status)host.status;
  *num_tokens = host.num_tokens;
  *num_documents = host.num_docs;
  return PE_OK;
}

pe_status check_rows_args(int32_t B, int32_t S, const void* in, const int64_t* flat_index,
                          const int32_t* cu_seqlens, const int64_t* num_tokens,
                          const int32_t* num_documents, void* ws, size_t ws_bytes) {
  if (B < 0 || S < 1 || !cu_seqlens || !num_tokens || !num_documents) return PE_ERR_INVALID_ARG;
  if ((int64_t)B * S >= (1LL << 40)) return PE_ERR_INVALID_ARG;
  if (B > 0 && (!in || !flat_index)) return PE_ERR_INVALID_ARG;
  if (!ws || ws_bytes < rows_ws_bytes(B) || !aligned(ws, 16)) return PE_ERR_WORKSPACE;
  if (!device_is_sm103()) return PE_ERR_UNSUPPORTED;
  return PE_OK;
}

}  // namespace

}  // namespace pe

using namespace pe;

extern "C" size_t pe_rows_workspace_size(int32_t num_rows) {
  return num_rows < 0 ? 0 : rows_ws_bytes(num_rows);
}

extern "C" pe_status pe_pack_document_ids(const int32_t* document_ids, int32_t B, int32_t S,
                                          int64_t* flat_index, int32_t* cu_seqlens,
                                          int64_t* num_tokens, int32_t* num_documents,
                                          void* workspace, size_t workspace_bytes,
                                          pe_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  PE_TRY(check_rows_args(B, S, document_ids, flat_index, cu_seqlens, num_tokens, num_documents,
                         workspace, workspace_bytes));
  const RowsWorkspace w = rows_ws_view(workspace, B);
  PE_TRY(clear_counts(w, B, stream));
  if (B > 0) {
    doc_ids_count_kernel<<<row_blocks(B, S), kRowThreads, 0, stream>>>(document_ids, B, S, w);
    PE_CUDA_TRY(cudaGetLastError());
  }
  rows_scan_kernel<<<1, kScanThreads, 0, stream>>>(B, w, nullptr, 0, cu_seqlens);
  PE_CUDA_TRY(cudaGetLastError());
  if (B > 0) {
    doc_ids_fill_kernel<<<row_blocks(B, S), kRowThreads, 0, stream>>>(document_ids, B, S, w,
                                                                   flat_index, cu_seqlens);
    PE_CUDA_TRY(cudaGetLastError());
  }
  return read_result(w, num_tokens, num_documents, stream);
}

extern "C" pe_status pe_flatten_packed_metadata(const int64_t* token_indices,
                                                const int32_t* row_cu_seqlens, int32_t B,
                                                int32_t S, int32_t M1, int64_t* flat_index,
                                                int32_t* cu_seqlens, int64_t* num_tokens,
                                                int32_t* num_documents, void* workspace,
                                                size_t workspace_bytes, pe_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (M1 < 1 || (B > 0 && !row_cu_seqlens)) return PE_ERR_INVALID_ARG;
  PE_TRY(check_rows_args(B, S, token_indices, flat_index, cu_seqlens, num_tokens, num_documents,
                         workspace, workspace_bytes));
  const RowsWorkspace w = rows_ws_view(workspace, B);
  PE_TRY(clear_counts(w, B, stream));
  if (B > 0) {
    nemo_rows_count_kernel<<<row_blocks(B, S), kRowThreads, 0, stream>>>(token_indices,
                                                                      row_cu_seqlens, B, S, M1, w);
    PE_CUDA_TRY(cudaGetLastError());
  }
  rows_scan_kernel<<<1, kScanThreads, 0, stream>>>(B, w, row_cu_seqlens, M1, cu_seqlens);
  PE_CUDA_TRY(cudaGetLastError());
  if (B > 0) {
    nemo_rows_fill_kernel<<<row_blocks(B, S), kRowThreads, 0, stream>>>(
        token_indices, row_cu_seqlens, B, S, M1, w, flat_index, cu_seqlens);
    PE_CUDA_TRY(cudaGetLastError());
  }
  return read_result(w, num_tokens, num_documents, stream);
}
