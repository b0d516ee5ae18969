// Shared device/host helpers of libpe (internal header).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pe.h"

namespace pe {

constexpr int kMaxHeadDim = 128;

// Host-side check of a CUDA runtime call; returns PE_ERR_CUDA from the caller.
#define PE_CUDA_TRY(expr)                                   \
  do {                                                      \
    cudaError_t pe_err_ = (expr);                           \
    if (pe_err_ != cudaSuccess) return PE_ERR_CUDA;         \
  } while (0)

#define PE_TRY(expr)                                        \
  do {                                                      \
    pe_status pe_st_ = (expr);                              \
    if (pe_st_ != PE_OK) return pe_st_;                     \
  } while (0)

__host__ __device__ inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

inline bool aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

// Element conversions to and from the fp32 compute type.
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// log2(e): scores are kept in the base-2 domain so that exp(x) = 2^(x log2 e)
// maps onto the hardware ex2 instruction.
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Programmatic dependent launch (a kernel launched with
// launch_after_previous): griddep_wait blocks until the previous kernel in
// the stream has completed and its writes are visible (at once for a kernel
// launched without it); griddep_launch_dependents lets the next such kernel
// be scheduled before this one ends.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Device-side status word at the head of every attention workspace.
struct DeviceStatus {
  int32_t code;       // pe_status
  int32_t detail;     // diagnostics: where a wait gave up (role id), or the
                      // first sequence of a layout that failed its check
  int32_t pad[2];
};

__device__ __forceinline__ void report_timeout(DeviceStatus* st, int detail) {
  if (st) {
    atomicCAS(&st->code, (int)PE_OK, (int)PE_ERR_DEVICE_TIMEOUT);
    st->detail = detail;
  }
}

// ---------------------------------------------------------------------------
// Tile plan: longest-processing-time-first order of sequences and the
// cumulative tile count in that order (built on the device, no host read).
// ---------------------------------------------------------------------------
struct TilePlan {
  int32_t* counter;        // work counter claimed with atomicAdd (reset by the plan)
  int32_t* total_tiles;    // number of tiles
  int32_t* order;          // [B] sequence index at each position (longest first)
  int32_t* tile_end;       // [B] inclusive prefix of tiles over positions
};

// Local (sliding-window) attention: the key at position j of a sequence is
// visible from the query at position r iff r - left <= j <= r + right. Both
// bounds are >= 0; kUnbounded stands for no bound (full attention).
constexpr int32_t kUnbounded = 0x7fffffff;
struct Window {
  int32_t left, right;
  __host__ __device__ bool active() const { return left != kUnbounded || right != kUnbounded; }
};
// The ABI's (left, right) with a negative bound meaning unbounded; a bound of
// max_seq_len - 1 or more reaches every key, so it is unbounded too.
inline Window make_window(int32_t left, int32_t right, int32_t max_seq_len) {
  Window w;
  w.left = (left < 0 || left >= max_seq_len - 1) ? kUnbounded : left;
  w.right = (right < 0 || right >= max_seq_len - 1) ? kUnbounded : right;
  return w;
}
constexpr Window kFullWindow = {kUnbounded, kUnbounded};
// First visible key position of the query at position r (r >= 0).
__host__ __device__ __forceinline__ int32_t window_lo(Window w, int32_t r) {
  return r - (w.left < r ? w.left : r);
}
// Last visible key position of the query at position r < len in a sequence of
// len keys (len - 1 for r >= len, rows that are computed but never stored).
__host__ __device__ __forceinline__ int32_t window_hi(Window w, int32_t r, int32_t len) {
  const int32_t room = len - 1 - r;
  return r + (w.right < room ? w.right : room);
}

// Workspace layout shared by the attention entry points:
//   [0, 16)        DeviceStatus
//   [16, 32)       counter, total_tiles
//   [32, ...)      order[B], tile_end[B] (each rounded to 16 bytes)
//   [...]          kernel-specific scratch (16-byte aligned)
inline size_t plan_bytes(int32_t B) {
  size_t per = ((size_t)B * 4 + 15) / 16 * 16;
  return 32 + 2 * per;
}

inline TilePlan plan_view(void* ws, int32_t B) {
  char* base = static_cast<char*>(ws);
  size_t per = ((size_t)B * 4 + 15) / 16 * 16;
  TilePlan p;
  p.counter = reinterpret_cast<int32_t*>(base + 16);
  p.total_tiles = reinterpret_cast<int32_t*>(base + 20);
  p.order = reinterpret_cast<int32_t*>(base + 32);
  p.tile_end = reinterpret_cast<int32_t*>(base + 32 + per);
  return p;
}

// Decodes tile t of a plan into (sequence, local tile index) by binary search
// over the inclusive prefix; local < tiles of that sequence.
__device__ __forceinline__ void plan_decode(const int32_t* __restrict__ order,
                                            const int32_t* __restrict__ tile_end, int32_t B,
                                            int32_t t, int32_t& seq, int32_t& local) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    int mid = (lo + hi) >> 1;
    if (__ldg(tile_end + mid) > t) hi = mid; else lo = mid + 1;
  }
  seq = __ldg(order + lo);
  local = t - (lo > 0 ? __ldg(tile_end + lo - 1) : 0);
}

// What a caller's cu_seqlens must satisfy before any kernel reads through it:
// cu[0] = 0, cu[B] = N and 1 <= cu[i+1] - cu[i] <= S for every i (so every
// entry lies in [0, N] and every sequence is non-empty). A violation is
// recorded in `status` (PE_ERR_BAD_LENGTH for a length, PE_ERR_INVALID_ARG for
// an end; detail = the first offending sequence, or -1 for an end) and no
// attention kernel of the call reads q, k or v.
struct LayoutCheck {
  int32_t max_seq_len;
  int64_t num_tokens;
  DeviceStatus* status;
};

// Launches the plan kernel: tiles of sequence i = heads * ceil(L_i / rows_per_tile),
// or ceil(heads / 4) when L_i <= quad_heads_rows and ceil(heads / 2) when
// L_i <= pair_heads_rows (kernels that run four or two heads of such a sequence
// in one work item; 0 turns either off). The kernel first checks the layout
// (LayoutCheck); when the check fails, or when the status word already holds an
// error (an earlier pass of the same call), the plan has no tiles, so the
// persistent kernels that consume it claim no work. With pair_odd_tails, a
// longer sequence whose last item would hold only one of its two half-tiles
// (ceil(L_i / (rows_per_tile / 2)) odd) has those last half-tiles of two heads
// share one item: heads * (ceil(L_i / rows_per_tile) - 1) + ceil(heads / 2)
// tiles.
pe_status launch_tile_plan(const int32_t* cu_seqlens, int32_t B, int32_t heads,
                           int32_t rows_per_tile, int32_t pair_heads_rows,
                           int32_t quad_heads_rows, TilePlan plan, LayoutCheck check,
                           cudaStream_t stream, int32_t pair_odd_tails = 0);

// The same check for calls without a tile plan (first-token queries): writes
// the whole status word (code 0 when the layout is valid), so it also serves as
// the call's reset of that word. Kernels launched after it read the code at
// entry and return when it is not PE_OK.
pe_status launch_layout_check(const int32_t* cu_seqlens, int32_t B, LayoutCheck check,
                              cudaStream_t stream);

// Limit of every bounded pipeline wait in the kernels launched from now on
// (pe_set_wait_limit_ns; 2 s by default).
uint64_t wait_limit_ns();

// First-token queries split each sequence's keys into chunks of this many keys
// (one CTA each) when sequences are long (see the forward entry point); chunk
// partials are merged after.
constexpr int32_t kFirstTokenChunk = 1024;
inline int32_t first_token_splits(int32_t max_seq_len) {
  return max_seq_len <= kFirstTokenChunk
             ? 1
             : static_cast<int32_t>((max_seq_len + kFirstTokenChunk - 1) / kFirstTokenChunk);
}
// Bytes of chunk partials (m, l, o[D] per chunk) of a first-token call.
inline size_t first_token_partial_bytes(int32_t B, int32_t H, int32_t D, int32_t max_seq_len) {
  const int32_t ns = first_token_splits(max_seq_len);
  if (ns == 1) return 0;
  return ((size_t)B * H * ns * (D + 2) * sizeof(float) + 15) / 16 * 16;
}

// Number of SMs of the current device (cached per device).
int device_sm_count();

// Launches `kernel` so that it may be scheduled while the previous kernel in
// the stream is still running (programmatic stream serialisation); the kernel
// must call griddep_wait() before it reads anything that kernel wrote.
template <typename... KArgs, typename... Args>
pe_status launch_after_previous(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kernel, args...) != cudaSuccess) return PE_ERR_CUDA;
  return PE_OK;
}
// True if the current device is compute capability 10.3.
bool device_is_sm103();

}  // namespace pe
