// Streaming of whole token rows for the first-token query kernels.
//
// In first-token mode each sequence has a single query row, so both the
// forward and the backward are bound by moving the key and value rows once
// (page "Source code for gigl.nn.packed_attention", function
// `packed_attention`, `query_is_first_token`). The packed buffers are
// token-major [N, H, D]: one token's keys for all heads are one contiguous row
// of H*D elements, so the kernels stream whole rows in order:
//
//  * the token range [0, N) is cut into equal chunks, one CTA each;
//  * one producer thread per CTA walks the sequences that overlap its chunk and
//    copies their visible k and v rows into a five-stage shared-memory ring
//    with bulk asynchronous copies (cp.async.bulk, completion counted in bytes
//    on an mbarrier per stage), running ahead across sequence boundaries;
//  * four consumer warps read each row with 16-byte shared loads: lane l owns
//    vectors l, l + 32, ..., l + 32 (VPL - 1) of a row, and a head's D
//    elements are LPH consecutive lanes, so per-head dot products reduce with
//    xor shuffles inside a lane group.
//
// A row is supported when it is a whole number of 512-byte warp loads and a
// head spans a power of two of lanes (D in {32, 64, 128}).
#pragma once

#include "pe_common.cuh"
#include "pe_sm103.cuh"

namespace pe {
namespace stream {

using namespace sm103;

constexpr int kWarps = 4;                  // consumer warps
constexpr int kThreads = kWarps * 32;      // consumer threads
constexpr int kBlock = kThreads + 32;      // + one producer warp
constexpr int kStages = 5;
constexpr int kStageBytes = 8192;          // of k (and as much of v) per stage

template <typename T, int D, int VPL>
struct Shape {
  static constexpr int kEPV = 16 / (int)sizeof(T);  // elements per 16-byte vector
  static constexpr int kLPH = D / kEPV;              // lanes per head
  static constexpr int kRow = 32 * VPL * kEPV;       // elements of one token row (H * D)
  static constexpr int kRowBytes = kRow * (int)sizeof(T);
  static constexpr int kH = kRow / D;                // heads
  static constexpr int kRows = kStageBytes / kRowBytes > 0 ? kStageBytes / kRowBytes : 1;
  static constexpr int kStageElems = kRows * kRow;   // of k (or v) per stage
  static constexpr size_t kRingBytes = (size_t)kStages * 2 * kStageElems * sizeof(T);
  static_assert(32 % kLPH == 0 && kLPH >= 1, "a head must span a power of two of lanes");
  static_assert(kRowBytes % 16 == 0, "bulk copies move multiples of 16 bytes");
};

// Token row width in 512-byte warp loads (vectors per lane), 0 if the row is
// not a whole number of them.
inline int vectors_per_lane(pe_dtype dtype, int32_t H, int32_t D) {
  const int64_t row_bytes = (int64_t)H * D * (dtype == PE_FP32 ? 4 : 2);
  return row_bytes % 512 == 0 ? (int)(row_bytes / 512) : 0;
}

template <typename T>
__device__ __forceinline__ void unpack16(const uint4& r, float (&x)[16 / sizeof(T)]) {
  if constexpr (sizeof(T) == 4) {
    x[0] = __uint_as_float(r.x);
    x[1] = __uint_as_float(r.y);
    x[2] = __uint_as_float(r.z);
    x[3] = __uint_as_float(r.w);
  } else {
    // bf16 element 2j is the low half of word j; a bf16 is the top half of an fp32.
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      x[2 * j] = __uint_as_float(w[j] << 16);
      x[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
    }
  }
}

// The inverse of unpack16, rounding to nearest even for bf16.
template <typename T>
__device__ __forceinline__ uint4 pack16(const float (&x)[16 / sizeof(T)]) {
  if constexpr (sizeof(T) == 4) {
    return make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]),
                      __float_as_uint(x[3]));
  } else {
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(x[2 * j], x[2 * j + 1]);  // .x low half
      w[j] = *reinterpret_cast<const uint32_t*>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
}

__device__ __forceinline__ uint4 load16(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

__device__ __forceinline__ void store16(void* p, const uint4& x) {
  *reinterpret_cast<uint4*>(p) = x;
}

// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned) from
// global to shared memory, counted on the mbarrier `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

// Barrier of the consumer warps only (the producer warp never joins it).
__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory");
}
// The same barrier (another id) that also returns the OR of `x` over the
// consumer threads, so that they all take the same branch after it.
__device__ __forceinline__ bool consumers_sync_or(bool x) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\t"
      "bar.red.or.pred p, 2, %2, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(x ? 1u : 0u), "n"(kThreads)
      : "memory");
  return r != 0;
}

// Largest i in [0, B) with cu[i] <= t (cu[0] = 0 <= t), found by the whole
// warp: each round probes 32 evenly spaced entries and keeps the interval the
// last true probe opens.
__device__ __forceinline__ int32_t find_sequence(const int32_t* __restrict__ cu, int32_t B,
                                                 int32_t t, int lane) {
  int32_t lo = 0, hi = B;  // answer in [lo, hi)
  while (hi - lo > 32) {
    const int32_t step = (hi - lo + 31) / 32;
    const int32_t idx = lo + lane * step;
    const bool le = idx < hi && __ldg(cu + idx) <= t;
    const int n = __popc(__ballot_sync(0xffffffffu, le));  // >= 1: cu[lo] <= t
    lo += (n - 1) * step;
    hi = min(hi, lo + step);
  }
  const int32_t idx = lo + lane;
  const bool le = idx < hi && __ldg(cu + idx) <= t;
  return lo + __popc(__ballot_sync(0xffffffffu, le)) - 1;
}

// The rows of one sequence inside a chunk [c0, c1): [a, next) lie in the
// chunk, [a, vis_end) of them are keys its query sees, and [s0, e1) are all
// the keys its query sees.
struct Segment {
  int64_t s0, e1, a, vis_end, next;
};

__device__ __forceinline__ Segment segment_of(const int32_t* __restrict__ cu, int32_t i,
                                              int64_t a, int64_t c1, int32_t key_limit) {
  Segment g;
  g.s0 = __ldg(cu + i);
  const int64_t s1 = __ldg(cu + i + 1);
  g.next = min(s1, c1);
  g.e1 = min(s1, g.s0 + key_limit);
  g.a = a;
  g.vis_end = min(g.next, g.e1);
  return g;
}

// Producer of a chunk (one thread): copies the visible k and v rows of every
// sequence overlapping [c0, c1) into the ring, at most kRows rows of one
// sequence per stage, in the order the consumers walk them. A wait that gives
// up stops the stream; the copies still in flight land in this CTA's shared
// memory, so they are waited for (bounded) before the thread returns.
template <class Sh, typename T>
__device__ __forceinline__ void produce_rows(const T* __restrict__ k, const T* __restrict__ v,
                                             const int32_t* __restrict__ cu, int32_t first,
                                             int64_t c0, int64_t c1, int32_t key_limit, T* ks,
                                             T* vs, uint64_t* full, uint64_t* empty,
                                             volatile WaitGuard* guard, DeviceStatus* status,
                                             int site) {
  constexpr int R = Sh::kRows, ROW = Sh::kRow;
  uint32_t g = 0;  // stages issued
  bool ok = true;
  int32_t i = first;
  for (int64_t a = c0; ok && a < c1; ++i) {
    const Segment sg = segment_of(cu, i, a, c1, key_limit);
    for (int64_t r0 = sg.a; r0 < sg.vis_end; r0 += R, ++g) {
      const int s = g % kStages;
      if (!mbar_wait(smem_u32(&empty[s]), ((g / kStages) & 1) ^ 1, guard, status, site)) {
        ok = false;
        break;
      }
      const uint32_t bytes = (uint32_t)(min((int64_t)R, sg.vis_end - r0) * Sh::kRowBytes);
      mbar_arrive_expect_tx(smem_u32(&full[s]), 2 * bytes);
      bulk_load(smem_u32(ks + s * Sh::kStageElems), k + r0 * ROW, bytes, smem_u32(&full[s]));
      bulk_load(smem_u32(vs + s * Sh::kStageElems), v + r0 * ROW, bytes, smem_u32(&full[s]));
    }
    a = sg.next;
  }
  if (!ok) {
    for (uint32_t j = g > kStages ? g - kStages : 0; j < g; ++j)
      mbar_drain_wait(smem_u32(&full[j % kStages]), (j / kStages) & 1);
  }
}

}  // namespace stream
}  // namespace pe
