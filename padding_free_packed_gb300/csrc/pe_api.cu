// C-ABI entry points of libpe: host-side argument checks, workspace layout and
// dispatch to the kernel families. Every check runs before any launch.
#include <cstring>
#include <math.h>

#include <atomic>

#include "pe_kernels.cuh"

namespace pe {

namespace {
constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;
std::atomic<uint64_t> g_wait_limit_ns{kDefaultWaitLimitNs};
}  // namespace

uint64_t wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }

namespace {
constexpr int kMaxDevices = 64;
int g_sm_count[kMaxDevices];
int g_is_sm103[kMaxDevices];  // 0 unknown, 1 yes, 2 no

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  return dev;
}
}  // namespace

int device_sm_count() {
  const int dev = current_device();
  if (dev < 0) return 1;
  if (g_sm_count[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    g_sm_count[dev] = n > 0 ? n : 1;
  }
  return g_sm_count[dev];
}

bool device_is_sm103() {
  const int dev = current_device();
  if (dev < 0) return false;
  if (g_is_sm103[dev] == 0) {
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    g_is_sm103[dev] = (major == 10 && minor == 3) ? 1 : 2;
  }
  return g_is_sm103[dev] == 1;
}

namespace {

inline size_t round16(size_t x) { return (x + 15) / 16 * 16; }

// Bytes a call requires. First-token forwards may also use
// first_token_partial_bytes() more (reported by pe_attention_workspace_size)
// to split long sequences over several CTAs; without them they run one CTA
// per (sequence, head).
size_t attention_ws_bytes(int32_t B, int64_t N, int32_t H, int query_is_first_token,
                          int backward) {
  size_t bytes = plan_bytes(B);
  if (backward) {
    const int64_t nq = query_is_first_token ? B : N;
    bytes += round16((size_t)H * (size_t)nq * sizeof(float));
  }
  return bytes;
}

pe_status check_common(pe_dtype dtype, int32_t B, int64_t N, int32_t H, int32_t D, int32_t S,
                       float scale) {
  if (dtype != PE_BF16 && dtype != PE_FP32) return PE_ERR_INVALID_ARG;
  if (B < 0 || N < 0 || H < 1 || S < 1) return PE_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return PE_ERR_INVALID_ARG;
  if (D < 8 || D % 8 != 0 || D > kMaxHeadDim) return PE_ERR_UNSUPPORTED;
  if (N >= (1LL << 31)) return PE_ERR_OVERFLOW;
  if ((N == 0) != (B == 0)) return PE_ERR_INVALID_ARG;  // every sequence holds >= 1 token
  // Tile counts are int32 on the device: bound them on the host.
  const int64_t tiles = (int64_t)H * (N / 64 + B + 1);
  if (tiles >= (1LL << 31)) return PE_ERR_OVERFLOW;
  return PE_OK;
}

pe_status check_tensor(const void* p, int64_t elems) {
  if (elems == 0) return PE_OK;
  if (!p) return PE_ERR_INVALID_ARG;
  if (!aligned(p, 16)) return PE_ERR_UNSUPPORTED;
  return PE_OK;
}

pe_status check_workspace(void* ws, size_t have, size_t need) {
  if (!ws || have < need || !aligned(ws, 16)) return PE_ERR_WORKSPACE;
  return PE_OK;
}

}  // namespace
}  // namespace pe

using namespace pe;

extern "C" const char* pe_status_string(int status) {
  switch (status) {
    case PE_OK: return "ok";
    case PE_ERR_INVALID_ARG: return "invalid argument";
    case PE_ERR_BAD_LENGTH: return "sequence length < 1 or > max_seq_len";
    case PE_ERR_OVERFLOW: return "token or tile count does not fit in int32";
    case PE_ERR_UNSUPPORTED: return "unsupported head_dim, dtype, alignment or device";
    case PE_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case PE_ERR_CUDA: return "CUDA runtime error";
    case PE_ERR_DEVICE_TIMEOUT: return "a kernel gave up waiting on its pipeline";
    default: return "unknown status";
  }
}

extern "C" int pe_abi_version(void) { return 3; }

extern "C" size_t pe_attention_workspace_size(pe_dtype dtype, int32_t B, int64_t N,
                                              int32_t H, int32_t D, int32_t S,
                                              int query_is_first_token, int backward) {
  if (B < 0 || N < 0 || H < 1 || D < 0 || S < 1) return 0;
  size_t bytes = attention_ws_bytes(B, N, H, query_is_first_token, backward);
  if (query_is_first_token && !backward)
    bytes += first_token_stream_supported(dtype, H, D) ? first_token_stream_partial_bytes(N, H, D)
                                                       : first_token_partial_bytes(B, H, D, S);
  if (query_is_first_token && backward && first_token_bwd_stream_supported(dtype, H, D))
    bytes += first_token_bwd_stream_partial_bytes(N, H, D);
  return bytes;
}

extern "C" pe_status pe_packed_attention_fwd_local(
    pe_dtype dtype, int32_t B, int64_t N, int32_t H, int32_t D, int32_t S, const void* q,
    const void* k, const void* v, const int32_t* cu_seqlens, float scale, int32_t window_left,
    int32_t window_right, int query_is_first_token, void* out, float* lse, void* workspace,
    size_t workspace_bytes, pe_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  PE_TRY(check_common(dtype, B, N, H, D, S, scale));
  const int64_t nq = query_is_first_token ? B : N;
  PE_TRY(check_tensor(q, nq));
  PE_TRY(check_tensor(k, N));
  PE_TRY(check_tensor(v, N));
  PE_TRY(check_tensor(out, nq));
  if (B > 0 && !cu_seqlens) return PE_ERR_INVALID_ARG;
  if (lse && !aligned(lse, 4)) return PE_ERR_UNSUPPORTED;
  PE_TRY(check_workspace(workspace, workspace_bytes,
                         attention_ws_bytes(B, N, H, query_is_first_token, 0)));
  if (query_is_first_token && !first_token_supported(D)) return PE_ERR_UNSUPPORTED;
  if (!device_is_sm103()) return PE_ERR_UNSUPPORTED;
  const Window win = make_window(window_left, window_right, S);
  DeviceStatus* status = static_cast<DeviceStatus*>(workspace);
  const LayoutCheck chk = {S, N, status};
  if (B == 0) {
    PE_CUDA_TRY(cudaMemsetAsync(workspace, 0, sizeof(DeviceStatus), stream));
    return PE_OK;
  }
  const TilePlan plan = plan_view(workspace, B);
  if (query_is_first_token) {
    // No tile plan: the layout check writes the status word (its reset).
    PE_TRY(launch_layout_check(cu_seqlens, B, chk, stream));
    // Streaming form (whole token rows, equal token chunks per CTA) when the
    // row shape allows it and the workspace holds its chunk partials.
    if (first_token_stream_supported(dtype, H, D) &&
        workspace_bytes >= plan_bytes(B) + first_token_stream_partial_bytes(N, H, D)) {
      float* part = reinterpret_cast<float*>(static_cast<char*>(workspace) + plan_bytes(B));
      return fwd_first_token_stream(dtype, D, q, k, v, cu_seqlens, B, H, N, S, scale, win, out,
                                    lse, part, status, stream);
    }
    // Otherwise one CTA per (sequence, head), split over key chunks when
    // sequences are long on average (more than two chunks) and the workspace
    // has room for those chunk partials.
    const size_t part_bytes = first_token_partial_bytes(B, H, D, S);
    float* part = nullptr;
    if (part_bytes > 0 && N > 2LL * kFirstTokenChunk * B &&
        workspace_bytes >= plan_bytes(B) + part_bytes)
      part = reinterpret_cast<float*>(static_cast<char*>(workspace) + plan_bytes(B));
    return fwd_first_token(dtype, D, q, k, v, cu_seqlens, B, H, S, scale, win, out, lse, part,
                           status, stream);
  }
  PE_CUDA_TRY(cudaMemsetAsync(workspace, 0, sizeof(DeviceStatus), stream));
  if (dtype == PE_BF16 && D == 64) {
    PE_TRY(launch_tile_plan(cu_seqlens, B, H, sm103_fwd_rows_per_item(),
                            sm103_fwd_pair_heads_rows(win), sm103_fwd_quad_heads_rows(win), plan,
                            chk, stream, sm103_fwd_pair_odd_tails(win)));
    return fwd_sm103(q, k, v, cu_seqlens, B, H, N, scale, win, out, lse, plan, status, stream);
  }
  if (dtype == PE_BF16 && D == 128 && !win.active()) {
    PE_TRY(launch_tile_plan(cu_seqlens, B, H, sm103_d128_fwd_rows_per_item(),
                            sm103_d128_fwd_pair_heads_rows(), sm103_d128_fwd_quad_heads_rows(),
                            plan, chk, stream, sm103_d128_fwd_pair_odd_tails()));
    return fwd_sm103_d128(q, k, v, cu_seqlens, B, H, N, scale, out, lse, plan, status, stream);
  }
  if (dtype == PE_FP32 && D == 64 && !win.active()) {
    PE_TRY(launch_tile_plan(cu_seqlens, B, H, sm103_f32_fwd_rows_per_item(),
                            sm103_f32_fwd_pair_heads_rows(), sm103_f32_fwd_quad_heads_rows(),
                            plan, chk, stream));
    return fwd_sm103_f32(q, k, v, cu_seqlens, B, H, N, scale, out, lse, plan, status, stream);
  }
  PE_TRY(launch_tile_plan(cu_seqlens, B, H, simt_rows_per_item(), 0, 0, plan, chk, stream));
  return fwd_simt(dtype, D, q, k, v, cu_seqlens, B, H, scale, win, out, lse, N, plan, stream);
}

extern "C" pe_status pe_packed_attention_fwd(pe_dtype dtype, int32_t B, int64_t N, int32_t H,
                                             int32_t D, int32_t S, const void* q, const void* k,
                                             const void* v, const int32_t* cu_seqlens,
                                             float scale, int query_is_first_token, void* out,
                                             float* lse, void* workspace, size_t workspace_bytes,
                                             pe_stream_t stream) {
  return pe_packed_attention_fwd_local(dtype, B, N, H, D, S, q, k, v, cu_seqlens, scale, -1, -1,
                                       query_is_first_token, out, lse, workspace,
                                       workspace_bytes, stream);
}

extern "C" pe_status pe_packed_attention_bwd_local(
    pe_dtype dtype, int32_t B, int64_t N, int32_t H, int32_t D, int32_t S, const void* q,
    const void* k, const void* v, const int32_t* cu_seqlens, float scale, int32_t window_left,
    int32_t window_right, int query_is_first_token, const void* out, const float* lse,
    const void* dout, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
    pe_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  PE_TRY(check_common(dtype, B, N, H, D, S, scale));
  const int64_t nq = query_is_first_token ? B : N;
  PE_TRY(check_tensor(q, nq));
  PE_TRY(check_tensor(k, N));
  PE_TRY(check_tensor(v, N));
  PE_TRY(check_tensor(out, nq));
  PE_TRY(check_tensor(dout, nq));
  PE_TRY(check_tensor(dq, nq));
  PE_TRY(check_tensor(dk, N));
  PE_TRY(check_tensor(dv, N));
  if (B > 0 && (!cu_seqlens || !lse)) return PE_ERR_INVALID_ARG;
  if (lse && !aligned(lse, 4)) return PE_ERR_UNSUPPORTED;
  PE_TRY(check_workspace(workspace, workspace_bytes,
                         attention_ws_bytes(B, N, H, query_is_first_token, 1)));
  if (!device_is_sm103()) return PE_ERR_UNSUPPORTED;
  const Window win = make_window(window_left, window_right, S);
  DeviceStatus* status = static_cast<DeviceStatus*>(workspace);
  const LayoutCheck chk = {S, N, status};
  const size_t base_bytes = attention_ws_bytes(B, N, H, query_is_first_token, 1);
  if (B > 0 && query_is_first_token && first_token_bwd_stream_supported(dtype, H, D) &&
      workspace_bytes >= base_bytes + first_token_bwd_stream_partial_bytes(N, H, D)) {
    // Streaming form: the layout check writes the status word (its reset).
    PE_TRY(launch_layout_check(cu_seqlens, B, chk, stream));
    float* part = reinterpret_cast<float*>(static_cast<char*>(workspace) + base_bytes);
    return bwd_first_token_stream(dtype, D, q, k, v, out, dout, lse, cu_seqlens, B, H, N, S,
                                  scale, win, dq, dk, dv, part, status, stream);
  }
  PE_CUDA_TRY(cudaMemsetAsync(workspace, 0, sizeof(DeviceStatus), stream));
  if (B == 0) return PE_OK;
  TilePlan plan = plan_view(workspace, B);
  float* delta = reinterpret_cast<float*>(static_cast<char*>(workspace) + plan_bytes(B));
  if (dtype == PE_BF16 && D == 64 && !query_is_first_token) {
    PE_TRY(bwd_preprocess(dtype, D, out, dout, N, H, delta, stream));
    return bwd_sm103(q, k, v, cu_seqlens, B, H, N, scale, win, lse, dout, delta, dq, dk, dv,
                     plan, chk, stream);
  }
  if (dtype == PE_BF16 && D == 128 && !query_is_first_token) {
    PE_TRY(bwd_preprocess(dtype, D, out, dout, N, H, delta, stream));
    return bwd_sm103_d128(q, k, v, cu_seqlens, B, H, N, scale, win, lse, dout, delta, dq, dk,
                          dv, plan, chk, stream);
  }
  return bwd_simt(dtype, D, q, k, v, cu_seqlens, B, H, nq, scale, query_is_first_token, win, out,
                  lse, dout, dq, dk, dv, delta, plan, chk, stream);
}

extern "C" pe_status pe_packed_attention_bwd(pe_dtype dtype, int32_t B, int64_t N, int32_t H,
                                             int32_t D, int32_t S, const void* q, const void* k,
                                             const void* v, const int32_t* cu_seqlens,
                                             float scale, int query_is_first_token,
                                             const void* out, const float* lse, const void* dout,
                                             void* dq, void* dk, void* dv, void* workspace,
                                             size_t workspace_bytes, pe_stream_t stream) {
  return pe_packed_attention_bwd_local(dtype, B, N, H, D, S, q, k, v, cu_seqlens, scale, -1, -1,
                                       query_is_first_token, out, lse, dout, dq, dk, dv,
                                       workspace, workspace_bytes, stream);
}

extern "C" const char* pe_attention_kernel(pe_dtype dtype, int32_t D, int query_is_first_token,
                                          int backward) {
  if ((dtype != PE_BF16 && dtype != PE_FP32) || D < 8 || D % 8 != 0 || D > kMaxHeadDim)
    return "unsupported";
  if (backward) {
    if (query_is_first_token)
      return (D == 32 || D == 64 || D == 128) ? "first_token_bwd" : "simt_ffma_bwd";
    if (dtype == PE_BF16 && D == 64) return "tcgen05_bf16_d64_bwd";
    if (dtype == PE_BF16 && D == 128) return "tcgen05_bf16_d128_bwd";
    return "simt_ffma_bwd";
  }
  if (query_is_first_token) return first_token_supported(D) ? "first_token_gemv" : "unsupported";
  if (dtype == PE_BF16 && D == 64) return "tcgen05_bf16_d64";
  if (dtype == PE_BF16 && D == 128) return "tcgen05_bf16_d128";
  if (dtype == PE_FP32 && D == 64) return "tcgen05_f32_d64";
  return "simt_ffma";
}

extern "C" const char* pe_attention_kernel_local(pe_dtype dtype, int32_t D, int32_t S,
                                                int32_t window_left, int32_t window_right,
                                                int query_is_first_token, int backward) {
  const char* family = pe_attention_kernel(dtype, D, query_is_first_token, backward);
  if (S < 1) return "unsupported";
  // A window that reaches every key is full attention; first-token calls and
  // the backward families take windows in their own kernels. Of the forward's
  // tensor-core families only bf16 head_dim 64 has a local instance.
  if (!make_window(window_left, window_right, S).active() || query_is_first_token || backward)
    return family;
  if (dtype == PE_BF16 && D == 64) return family;
  return std::strcmp(family, "unsupported") == 0 ? family : "simt_ffma";
}

extern "C" uint64_t pe_set_wait_limit_ns(uint64_t ns) {
  return g_wait_limit_ns.exchange(ns == 0 ? kDefaultWaitLimitNs : ns);
}

extern "C" pe_status pe_read_device_status(const void* workspace, pe_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (!workspace) return PE_ERR_INVALID_ARG;
  DeviceStatus host;
  PE_CUDA_TRY(cudaMemcpyAsync(&host, workspace, sizeof(host), cudaMemcpyDeviceToHost, stream));
  PE_CUDA_TRY(cudaStreamSynchronize(stream));
  return (pe_status)host.code;
}
