// Allocation-free variant of the packed attention forward.
//
// Some callers cannot hand this library a workspace: a host runtime that owns
// every device allocation through its own fixed pool and exposes no scratch
// API (a serving process or a framework plugin), or a latency-critical loop
// where a cudaMalloc/cudaFree pair would add implicit device-wide
// synchronisation. For them this entry point keeps the forward's scratch (the
// device status word and the longest-first tile plan, plus a first-token
// forward's partial softmax states when they fit) in a file-scope device
// array that every GPU loading the library holds until the process exits. A
// first-token call whose partial states do not fit runs the same forward
// without them (one CTA per sequence and head).
//
// Set-up: the first call on a device, with that device current, looks up the
// array's device address with cudaGetSymbolAddress and caches it for the life
// of the process (the cache does not survive cudaDeviceReset); make that
// first call before any stream capture. No call allocates memory. The array
// is shared by every call on a device and keeps the last call's contents; the
// forward clears the parts that must start at zero (the status word and the
// work counter) itself. Calls whose executions overlap on the GPU (two
// streams, or two host threads) race on the array and must be serialised by
// the caller.
#include <atomic>

#include "pe_kernels.cuh"

namespace {

constexpr int32_t kNoAllocMaxSequences = 65536;
// Status word + counters (32 bytes) + LPT order and cumulative tiles (4 bytes
// per sequence each) for the largest accepted batch.
constexpr size_t kNoAllocScratchBytes = 32 + 2 * sizeof(int32_t) * kNoAllocMaxSequences;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_address[kMaxDevices];

pe_status scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PE_ERR_CUDA;
  void* p = g_scratch_address[dev].load();
  if (!p) {
    // The symbol's name is a host-side stand-in; only this lookup yields the
    // array's address on the current device.
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return PE_ERR_CUDA;
    g_scratch_address[dev].store(p);
  }
  *out = p;
  return PE_OK;
}

}  // namespace

extern "C" pe_status pe_packed_attention_fwd_noalloc(
    pe_dtype dtype, int32_t num_sequences, int64_t num_tokens, int32_t num_heads,
    int32_t head_dim, int32_t max_seq_len, const void* q, const void* k, const void* v,
    const int32_t* cu_seqlens, float scale, int query_is_first_token, void* out, float* lse,
    pe_stream_t stream) {
  if (num_sequences > kNoAllocMaxSequences) return PE_ERR_WORKSPACE;
  // What the forward requires; first-token calls use more (chunk partials)
  // only when it fits, and otherwise run without it.
  const size_t need = pe_attention_workspace_size(dtype, num_sequences, num_tokens, num_heads,
                                                  head_dim, max_seq_len, 0, 0);
  if (need > kNoAllocScratchBytes) return PE_ERR_WORKSPACE;
  void* scratch = nullptr;
  pe_status st = scratch_for_current_device(&scratch);
  if (st != PE_OK) return st;
  return pe_packed_attention_fwd(dtype, num_sequences, num_tokens, num_heads, head_dim,
                                 max_seq_len, q, k, v, cu_seqlens, scale, query_is_first_token,
                                 out, lse, scratch, kNoAllocScratchBytes, stream);
}

// The device status word of the last allocation-free call on the current
// device lives at the head of the array, where the caller cannot address it.
extern "C" pe_status pe_read_noalloc_status(pe_stream_t stream) {
  void* scratch = nullptr;
  pe_status st = scratch_for_current_device(&scratch);
  if (st != PE_OK) return st;
  return pe_read_device_status(scratch, stream);
}
