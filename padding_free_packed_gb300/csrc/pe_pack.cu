// Pack index builder, padded<->packed row movers and the attention tile plan.
//
// pack_sequences (page "Source code for gigl.nn.packed_attention", module
// docstring, "Data flow of a packed forward" and "Example") is two kernels and
// one host read: a single-CTA validating scan writes cu_seqlens and the token
// count, a fill kernel writes flat_index, then the host copies back 16 bytes.
#include "pe_common.cuh"

namespace pe {

namespace {

constexpr int kScanThreads = 1024;

// Result of the validating scan, read back by the host in one copy.
struct PackResult {
  long long num_tokens;
  int32_t status;
  int32_t pad;
};

// Inclusive block-wide scan of one int64 per thread (blockDim.x == 1024).
__device__ __forceinline__ long long block_inclusive_scan(long long x, long long* warp_sums,
                                                          long long& block_total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    long long y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    long long w = warp_sums[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      long long y = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += y;
    }
    warp_sums[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const long long prefix = warp > 0 ? warp_sums[warp - 1] : 0;
  block_total = warp_sums[31];
  __syncthreads();  // warp_sums is reused by the next call
  return x + prefix;
}

// Validates 1 <= L_i <= S, writes cu_seqlens and the token count.
__global__ void __launch_bounds__(kScanThreads)
pack_scan_kernel(const int32_t* __restrict__ lengths, int32_t B, int32_t S,
                 int32_t* __restrict__ cu_seqlens, PackResult* __restrict__ result) {
  __shared__ long long warp_sums[32];
  __shared__ int bad;
  if (threadIdx.x == 0) bad = 0;
  __syncthreads();
  long long carry = 0;
  if (threadIdx.x == 0) cu_seqlens[0] = 0;
  for (int64_t base = 0; base < B; base += kScanThreads) {
    const int64_t i = base + threadIdx.x;
    long long len = 0;
    if (i < B) {
      len = lengths[i];
      if (len < 1 || len > S) bad = 1;  // benign race: every writer stores 1
    }
    long long total;
    const long long incl = block_inclusive_scan(len, warp_sums, total);
    if (i < B) cu_seqlens[i + 1] = (int32_t)(carry + incl);
    carry += total;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int32_t st = PE_OK;
    if (bad) st = PE_ERR_BAD_LENGTH;
    else if (carry >= (1LL << 31)) st = PE_ERR_OVERFLOW;
    result->num_tokens = carry;
    result->status = st;
  }
}

// flat_index[cu_i + j] = i * S + j: one block per sequence (grid-stride).
__global__ void pack_fill_kernel(const int32_t* __restrict__ cu_seqlens, int32_t B, int32_t S,
                                 const PackResult* __restrict__ result,
                                 int64_t* __restrict__ flat_index) {
  if (result->status != PE_OK) return;
  for (int64_t i = blockIdx.x; i < B; i += gridDim.x) {
    const int32_t start = cu_seqlens[i];
    const int32_t len = cu_seqlens[i + 1] - start;
    const int64_t row0 = i * (int64_t)S;
    for (int32_t j = threadIdx.x; j < len; j += blockDim.x) flat_index[start + j] = row0 + j;
  }
}

// ---------------------------------------------------------------------------
// Row movers: one warp per destination row; lanes move 16-, 4- or 1-byte words.
// Each lane issues up to four loads before its stores to keep bytes in flight.
// ---------------------------------------------------------------------------
template <typename W>
__device__ __forceinline__ void copy_row(const W* __restrict__ src, W* __restrict__ dst,
                                         int64_t words, int lane) {
  int64_t c = lane;
  for (; c + 96 < words; c += 128) {
    W a = src[c], b = src[c + 32], d = src[c + 64], e = src[c + 96];
    dst[c] = a;
    dst[c + 32] = b;
    dst[c + 64] = d;
    dst[c + 96] = e;
  }
  for (; c < words; c += 32) dst[c] = src[c];
}

template <typename W>
__device__ __forceinline__ void zero_row(W* __restrict__ dst, int64_t words, int lane) {
  W z;
  memset(&z, 0, sizeof(W));
  for (int64_t c = lane; c < words; c += 32) dst[c] = z;
}

template <typename W>
__global__ void gather_rows_kernel(const W* __restrict__ padded, const int64_t* __restrict__ flat,
                                   int64_t N, int64_t words, W* __restrict__ packed) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < N;
       t += warps) {
    const int64_t src_row = __ldg(flat + t);
    copy_row(padded + src_row * words, packed + t * words, words, lane);
  }
}

template <typename W>
__global__ void scatter_rows_kernel(const W* __restrict__ packed, const int32_t* __restrict__ cu,
                                    int32_t B, int32_t S, int64_t words, W* __restrict__ padded) {
  const int lane = threadIdx.x & 31;
  const int64_t rows = (int64_t)B * S;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t p = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); p < rows;
       p += warps) {
    const int64_t i = p / S;
    const int32_t j = (int32_t)(p - i * S);
    const int32_t start = __ldg(cu + i);
    const int32_t len = __ldg(cu + i + 1) - start;
    if (j < len)
      copy_row(packed + (int64_t)(start + j) * words, padded + p * words, words, lane);
    else
      zero_row(padded + p * words, words, lane);
  }
}

template <typename W>
pe_status launch_gather(const void* padded, const int64_t* flat, int64_t N, int64_t row_bytes,
                        void* packed, cudaStream_t stream) {
  const int64_t words = row_bytes / (int64_t)sizeof(W);
  const int threads = 256;
  int64_t blocks = ceil_div(N, threads / 32);
  const int64_t cap = (int64_t)device_sm_count() * 8;
  if (blocks > cap) blocks = cap;
  gather_rows_kernel<W><<<(unsigned)blocks, threads, 0, stream>>>(
      static_cast<const W*>(padded), flat, N, words, static_cast<W*>(packed));
  PE_CUDA_TRY(cudaGetLastError());
  return PE_OK;
}

template <typename W>
pe_status launch_scatter(const void* packed, const int32_t* cu, int32_t B, int32_t S,
                         int64_t row_bytes, void* padded, cudaStream_t stream) {
  const int64_t words = row_bytes / (int64_t)sizeof(W);
  const int threads = 256;
  int64_t blocks = ceil_div((int64_t)B * S, threads / 32);
  const int64_t cap = (int64_t)device_sm_count() * 8;
  if (blocks > cap) blocks = cap;
  scatter_rows_kernel<W><<<(unsigned)blocks, threads, 0, stream>>>(
      static_cast<const W*>(packed), cu, B, S, words, static_cast<W*>(padded));
  PE_CUDA_TRY(cudaGetLastError());
  return PE_OK;
}

// ---------------------------------------------------------------------------
// Layout check of a caller's cu_seqlens (one CTA of kScanThreads threads):
// cu[0] = 0, cu[B] = N, 1 <= cu[i+1] - cu[i] <= S. Reads only cu[0 .. B].
// Returns PE_OK or the error code, the same in every thread; *detail gets the
// first sequence whose length is out of range, or -1 for an end.
// ---------------------------------------------------------------------------
__device__ int32_t check_layout_cta(const int32_t* __restrict__ cu, int32_t B,
                                    const LayoutCheck& chk, int32_t* detail) {
  __shared__ int32_t bad_seq;
  __shared__ int32_t bad_end;
  if (threadIdx.x == 0) {
    bad_seq = 0x7fffffff;
    bad_end = (__ldg(cu) != 0 || (int64_t)__ldg(cu + B) != chk.num_tokens) ? 1 : 0;
  }
  __syncthreads();
  for (int64_t i = threadIdx.x; i < B; i += blockDim.x) {
    const int64_t len = (int64_t)__ldg(cu + i + 1) - __ldg(cu + i);
    if (len < 1 || len > chk.max_seq_len) atomicMin(&bad_seq, (int32_t)i);
  }
  __syncthreads();
  const int32_t seq = bad_seq, end = bad_end;
  __syncthreads();  // the shared flags may be reused by a later call in this CTA
  *detail = seq != 0x7fffffff ? seq : -1;
  if (seq != 0x7fffffff) return PE_ERR_BAD_LENGTH;
  return end ? PE_ERR_INVALID_ARG : PE_OK;
}

__global__ void __launch_bounds__(kScanThreads)
layout_check_kernel(const int32_t* __restrict__ cu, int32_t B, LayoutCheck chk) {
  griddep_launch_dependents();  // the next kernel may be scheduled; it waits for this one
  int32_t detail;
  const int32_t code = check_layout_cta(cu, B, chk, &detail);
  if (threadIdx.x == 0) {
    chk.status->code = code;
    chk.status->detail = code == PE_OK ? 0 : detail;
  }
}

// ---------------------------------------------------------------------------
// Tile plan: counting sort of sequences by tile length (longest first), then
// the inclusive prefix of tiles in that order. One CTA; no host read.
// ---------------------------------------------------------------------------
constexpr int kPlanBins = 2048;

__global__ void __launch_bounds__(kScanThreads)
tile_plan_kernel(const int32_t* __restrict__ cu, int32_t B, int32_t heads, int32_t rows_per_tile,
                 int32_t pair_heads_rows, int32_t quad_heads_rows, TilePlan plan,
                 LayoutCheck chk, int32_t pair_odd_tails) {
  griddep_launch_dependents();  // the kernel that consumes the plan waits for it on the device
  __shared__ int32_t start[kPlanBins];
  __shared__ long long warp_sums[32];
  const int tid = threadIdx.x;
  // An invalid layout (or an error already recorded by an earlier pass of the
  // same call) leaves a plan without tiles: nothing below reads through cu.
  {
    int32_t detail;
    const int32_t prior = *reinterpret_cast<volatile int32_t*>(&chk.status->code);
    const int32_t code = check_layout_cta(cu, B, chk, &detail);
    if (code != PE_OK || prior != PE_OK) {
      if (tid == 0) {
        if (code != PE_OK && atomicCAS(&chk.status->code, (int)PE_OK, code) == PE_OK)
          chk.status->detail = detail;
        *plan.total_tiles = 0;
        *plan.counter = 0;
      }
      return;
    }
  }
  for (int k = tid; k < kPlanBins; k += kScanThreads) start[k] = 0;
  __syncthreads();
  for (int64_t i = tid; i < B; i += kScanThreads) {
    const int32_t blocks = (int32_t)ceil_div(__ldg(cu + i + 1) - __ldg(cu + i), rows_per_tile);
    atomicAdd(&start[min(blocks, kPlanBins - 1)], 1);
  }
  __syncthreads();
  // Exclusive scan in descending key order: start[k] = #sequences with key > k.
  {
    long long total;
    const int k0 = kPlanBins - 1 - 2 * tid, k1 = k0 - 1;
    const long long a = start[k0], b = start[k1];
    const long long incl = block_inclusive_scan(a + b, warp_sums, total);
    __syncthreads();
    start[k0] = (int32_t)(incl - a - b);
    start[k1] = (int32_t)(incl - b);
  }
  __syncthreads();
  for (int64_t i = tid; i < B; i += kScanThreads) {
    const int32_t blocks = (int32_t)ceil_div(__ldg(cu + i + 1) - __ldg(cu + i), rows_per_tile);
    const int32_t pos = atomicAdd(&start[min(blocks, kPlanBins - 1)], 1);
    plan.order[pos] = (int32_t)i;
  }
  __syncthreads();
  long long carry = 0;
  for (int64_t base = 0; base < B; base += kScanThreads) {
    const int64_t pos = base + tid;
    long long tiles = 0;
    if (pos < B) {
      const int32_t i = plan.order[pos];
      const int32_t len = __ldg(cu + i + 1) - __ldg(cu + i);
      const long long pairs = ceil_div(len, rows_per_tile);
      const bool odd_tail = pair_odd_tails && (ceil_div(len, rows_per_tile / 2) & 1);
      tiles = len <= quad_heads_rows   ? (long long)(heads + 3) / 4
              : len <= pair_heads_rows ? (long long)(heads + 1) / 2
              : odd_tail               ? (long long)heads * (pairs - 1) + (heads + 1) / 2
                                       : (long long)heads * pairs;
    }
    long long total;
    const long long incl = block_inclusive_scan(tiles, warp_sums, total);
    if (pos < B) plan.tile_end[pos] = (int32_t)(carry + incl);
    carry += total;
  }
  if (tid == 0) {
    *plan.total_tiles = (int32_t)carry;
    *plan.counter = 0;
  }
}

}  // namespace

pe_status launch_tile_plan(const int32_t* cu_seqlens, int32_t B, int32_t heads,
                           int32_t rows_per_tile, int32_t pair_heads_rows,
                           int32_t quad_heads_rows, TilePlan plan, LayoutCheck check,
                           cudaStream_t stream, int32_t pair_odd_tails) {
  static_assert(kPlanBins == 2 * kScanThreads, "plan scan covers two bins per thread");
  if (!check.status) return PE_ERR_INVALID_ARG;
  tile_plan_kernel<<<1, kScanThreads, 0, stream>>>(cu_seqlens, B, heads, rows_per_tile,
                                                   pair_heads_rows, quad_heads_rows, plan, check,
                                                   pair_odd_tails);
  PE_CUDA_TRY(cudaGetLastError());
  return PE_OK;
}

pe_status launch_layout_check(const int32_t* cu_seqlens, int32_t B, LayoutCheck check,
                              cudaStream_t stream) {
  if (!check.status) return PE_ERR_INVALID_ARG;
  layout_check_kernel<<<1, kScanThreads, 0, stream>>>(cu_seqlens, B, check);
  PE_CUDA_TRY(cudaGetLastError());
  return PE_OK;
}

}  // namespace pe

using namespace pe;

extern "C" size_t pe_pack_workspace_size(int32_t /*num_sequences*/) { return sizeof(PackResult); }

extern "C" pe_status pe_pack_sequences(const int32_t* lengths, int32_t B, int32_t S,
                                       int64_t* flat_index, int32_t* cu_seqlens,
                                       int64_t* num_tokens, void* workspace,
                                       size_t workspace_bytes, pe_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (B < 0 || S < 1 || !cu_seqlens || !num_tokens) return PE_ERR_INVALID_ARG;
  if (B > 0 && (!lengths || !flat_index)) return PE_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < sizeof(PackResult) || !aligned(workspace, 16))
    return PE_ERR_WORKSPACE;
  if (!device_is_sm103()) return PE_ERR_UNSUPPORTED;
  PackResult* result = static_cast<PackResult*>(workspace);
  pack_scan_kernel<<<1, kScanThreads, 0, stream>>>(lengths, B, S, cu_seqlens, result);
  PE_CUDA_TRY(cudaGetLastError());
  if (B > 0) {
    const int blocks = (int)(B < 65535 ? B : 65535);
    pack_fill_kernel<<<blocks, 256, 0, stream>>>(cu_seqlens, B, S, result, flat_index);
    PE_CUDA_TRY(cudaGetLastError());
  }
  PackResult host;
  PE_CUDA_TRY(cudaMemcpyAsync(&host, result, sizeof(host), cudaMemcpyDeviceToHost, stream));
  PE_CUDA_TRY(cudaStreamSynchronize(stream));
  if (host.status != PE_OK) return (pe_status)host.status;
  *num_tokens = host.num_tokens;
  return PE_OK;
}

extern "C" pe_status pe_gather_packed(const void* padded, const int64_t* flat_index,
                                      int64_t N, int64_t row_bytes, void* packed,
                                      pe_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (N < 0 || row_bytes < 1) return PE_ERR_INVALID_ARG;
  if (N == 0) return PE_OK;
  if (!padded || !flat_index || !packed) return PE_ERR_INVALID_ARG;
  if (!device_is_sm103()) return PE_ERR_UNSUPPORTED;
  if (row_bytes % 16 == 0 && aligned(padded, 16) && aligned(packed, 16))
    return launch_gather<uint4>(padded, flat_index, N, row_bytes, packed, stream);
  if (row_bytes % 4 == 0 && aligned(padded, 4) && aligned(packed, 4))
    return launch_gather<uint32_t>(padded, flat_index, N, row_bytes, packed, stream);
  return launch_gather<uint8_t>(padded, flat_index, N, row_bytes, packed, stream);
}

extern "C" pe_status pe_scatter_padded(const void* packed, const int32_t* cu_seqlens, int32_t B,
                                       int32_t S, int64_t row_bytes, void* padded,
                                       pe_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (B < 0 || S < 1 || row_bytes < 1) return PE_ERR_INVALID_ARG;
  if (B == 0) return PE_OK;
  if (!packed || !cu_seqlens || !padded) return PE_ERR_INVALID_ARG;
  if (!device_is_sm103()) return PE_ERR_UNSUPPORTED;
  if (row_bytes % 16 == 0 && aligned(padded, 16) && aligned(packed, 16))
    return launch_scatter<uint4>(packed, cu_seqlens, B, S, row_bytes, padded, stream);
  if (row_bytes % 4 == 0 && aligned(padded, 4) && aligned(packed, 4))
    return launch_scatter<uint32_t>(packed, cu_seqlens, B, S, row_bytes, padded, stream);
  return launch_scatter<uint8_t>(packed, cu_seqlens, B, S, row_bytes, padded, stream);
}

// Host-resident padded grid -> packed device buffer with the copy engines:
// sequence i's rows are one contiguous run in both layouts, so each is one
// asynchronous copy (no SM work; overlaps kernels on other streams).
extern "C" pe_status pe_upload_packed(const void* padded_host, const int32_t* lengths_host,
                                      int32_t B, int32_t S, int64_t row_bytes, void* packed,
                                      pe_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (B < 0 || S < 1 || row_bytes < 1) return PE_ERR_INVALID_ARG;
  if (B == 0) return PE_OK;
  if (!padded_host || !lengths_host || !packed) return PE_ERR_INVALID_ARG;
  int64_t total = 0;
  for (int32_t i = 0; i < B; ++i) {
    if (lengths_host[i] < 1 || lengths_host[i] > S) return PE_ERR_BAD_LENGTH;
    total += lengths_host[i];
  }
  if (total >= (1LL << 31)) return PE_ERR_OVERFLOW;
  const char* src = static_cast<const char*>(padded_host);
  char* dst = static_cast<char*>(packed);
  int64_t t = 0;
  for (int32_t i = 0; i < B; ++i) {
    PE_CUDA_TRY(cudaMemcpyAsync(dst + t * row_bytes, src + (int64_t)i * S * row_bytes,
                                (size_t)lengths_host[i] * row_bytes, cudaMemcpyHostToDevice,
                                stream));
    t += lengths_host[i];
  }
  return PE_OK;
}

// Packed device buffer -> host-resident padded grid with the copy engines,
// the mirror of pe_upload_packed; pad rows are left as they are.
extern "C" pe_status pe_download_padded(const void* packed, const int32_t* lengths_host,
                                        int32_t B, int32_t S, int64_t row_bytes,
                                        void* padded_host, pe_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (B < 0 || S < 1 || row_bytes < 1) return PE_ERR_INVALID_ARG;
  if (B == 0) return PE_OK;
  if (!padded_host || !lengths_host || !packed) return PE_ERR_INVALID_ARG;
  int64_t total = 0;
  for (int32_t i = 0; i < B; ++i) {
    if (lengths_host[i] < 1 || lengths_host[i] > S) return PE_ERR_BAD_LENGTH;
    total += lengths_host[i];
  }
  if (total >= (1LL << 31)) return PE_ERR_OVERFLOW;
  const char* src = static_cast<const char*>(packed);
  char* dst = static_cast<char*>(padded_host);
  int64_t t = 0;
  for (int32_t i = 0; i < B; ++i) {
    PE_CUDA_TRY(cudaMemcpyAsync(dst + (int64_t)i * S * row_bytes, src + t * row_bytes,
                                (size_t)lengths_host[i] * row_bytes, cudaMemcpyDeviceToHost,
                                stream));
    t += lengths_host[i];
  }
  return PE_OK;
}
