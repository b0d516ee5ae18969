// CUDA-core packed attention forward entry points and the first-token-query
// kernel. The full-query FFMA kernel is in pe_fwd_simt.cuh (its fp32
// instances here, its bf16 instances in pe_fwd_simt_bf16.cu).
//
// First-token mode: the query of sequence i is one row, so the work is a
// matrix-vector product bounded by reading k and v once. One CTA per
// (sequence, head); lanes are grouped so that each group reads whole 16-byte
// slices of one key row; groups keep private online-softmax states that are
// merged at the end.
#include "pe_fwd_simt.cuh"

namespace pe {

using namespace fwd_simt_impl;

namespace {

// ---------------------------------------------------------------------------
// First-token query: one CTA per (sequence, head).
// ---------------------------------------------------------------------------
constexpr int kFtThreads = 256;

template <typename T, int D>
struct FtShape {
  static constexpr int kVec = 16 / sizeof(T);                       // elements per lane load
  static constexpr int kEPL = D < kVec ? D : kVec;                 // elements per lane
  static constexpr int kLPK = D / kEPL;                             // lanes per key row
  static constexpr int kGroups = 32 / kLPK;                         // key groups per warp
};

template <typename T, int EPL>
__device__ __forceinline__ void load_slice(const T* __restrict__ p, float (&x)[EPL]) {
  if constexpr (EPL * sizeof(T) == 16) {
    uint4 raw = __ldg(reinterpret_cast<const uint4*>(p));
    const T* e = reinterpret_cast<const T*>(&raw);
#pragma unroll
    for (int u = 0; u < EPL; ++u) x[u] = to_f32(e[u]);
  } else {
#pragma unroll
    for (int u = 0; u < EPL; ++u) x[u] = to_f32(p[u]);
  }
}

// One CTA per (sequence, head, chunk of `chunk` keys), grid-stride. With one
// chunk per sequence (nsplit == 1) it writes the output and lse directly;
// otherwise it writes the chunk's unnormalised partial state (m, l, o[D]) to
// `part` ([B][H][nsplit]), and first_token_merge_kernel combines the chunks
// in chunk order. Chunks past a sequence's end leave an empty state (l = 0).
template <typename T, int D>
__global__ void __launch_bounds__(kFtThreads)
fwd_first_token_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                       const int32_t* __restrict__ cu, int32_t B, int32_t H, float scale_log2,
                       int32_t key_limit, T* __restrict__ out, float* __restrict__ lse,
                       int32_t nsplit, int32_t chunk, float* __restrict__ part,
                       const DeviceStatus* __restrict__ status) {
  // A layout that failed its check (nothing else writes the word while this
  // kernel runs, so every thread reads the same code).
  if (status->code != PE_OK) return;
  using S = FtShape<T, D>;
  constexpr int EPL = S::kEPL, LPK = S::kLPK, G = S::kGroups;
  constexpr int kWarps = kFtThreads / 32;
  __shared__ float s_m[kWarps * G], s_l[kWarps * G];
  __shared__ float s_o[kWarps * G][D];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int group = lane / LPK, sub = lane % LPK;
  const int64_t row_stride = (int64_t)H * D;

  const int64_t items = (int64_t)B * H * nsplit;
  for (int64_t item = blockIdx.x; item < items; item += gridDim.x) {
    const int64_t ih = item / nsplit;
    const int32_t split = (int32_t)(item - ih * nsplit);
    const int32_t i = (int32_t)(ih / H), h = (int32_t)(ih - (int64_t)i * H);
    const int32_t seq_start = __ldg(cu + i);
    // The query sits at position 0: with a window it sees keys 0 .. key_limit-1.
    const int32_t seq_len = min(__ldg(cu + i + 1) - seq_start, key_limit);
    const int32_t key0 = split * chunk;
    const int32_t start = seq_start + key0;
    const int32_t len = max(0, min(chunk, seq_len - key0));  // keys of this chunk
    float qv[EPL];
    load_slice<T, EPL>(q + ((int64_t)i * H + h) * D + sub * EPL, qv);
#pragma unroll
    for (int u = 0; u < EPL; ++u) qv[u] *= scale_log2;
    float m = -INFINITY, l = 0.f, o[EPL];
#pragma unroll
    for (int u = 0; u < EPL; ++u) o[u] = 0.f;
    const T* kbase = k + (int64_t)start * row_stride + (int64_t)h * D + sub * EPL;
    const T* vbase = v + (int64_t)start * row_stride + (int64_t)h * D + sub * EPL;
    const int step = kWarps * G;
    // The trip count depends only on the warp, never on the lane group, so the
    // full-warp shuffles below always see all 32 lanes.
    for (int32_t base = warp * G; base < len; base += 2 * step) {
      const int32_t j0 = base + group, j1 = j0 + step;
      const bool has0 = j0 < len, has1 = j1 < len;
      float k0[EPL], k1[EPL], v0[EPL], v1[EPL];
      if (has0) {
        load_slice<T, EPL>(kbase + (int64_t)j0 * row_stride, k0);
        load_slice<T, EPL>(vbase + (int64_t)j0 * row_stride, v0);
      }
      if (has1) {
        load_slice<T, EPL>(kbase + (int64_t)j1 * row_stride, k1);
        load_slice<T, EPL>(vbase + (int64_t)j1 * row_stride, v1);
      }
      float d0 = 0.f, d1 = 0.f;
#pragma unroll
      for (int u = 0; u < EPL; ++u) {
        if (has0) d0 = fmaf(qv[u], k0[u], d0);
        if (has1) d1 = fmaf(qv[u], k1[u], d1);
      }
#pragma unroll
      for (int off = 1; off < LPK; off <<= 1) {
        d0 += __shfl_xor_sync(0xffffffffu, d0, off);
        d1 += __shfl_xor_sync(0xffffffffu, d1, off);
      }
      if (!has0) d0 = -INFINITY;
      if (!has1) d1 = -INFINITY;
      const float m_new = fmaxf(m, fmaxf(d0, d1));
      if (m_new == -INFINITY) continue;  // this group holds no key yet
      const float corr = ex2(m - m_new);
      const float p0 = ex2(d0 - m_new), p1 = ex2(d1 - m_new);
      l = l * corr + p0 + p1;
#pragma unroll
      for (int u = 0; u < EPL; ++u)
        o[u] = o[u] * corr + (has0 ? p0 * v0[u] : 0.f) + (has1 ? p1 * v1[u] : 0.f);
      m = m_new;
    }
    // Merge the per-group states of the CTA.
    const int slot = warp * G + group;
    if (sub == 0) {
      s_m[slot] = m;
      s_l[slot] = l;
    }
#pragma unroll
    for (int u = 0; u < EPL; ++u) s_o[slot][sub * EPL + u] = o[u];
    __syncthreads();
    if (threadIdx.x < D) {
      const int c = threadIdx.x;
      float gm = -INFINITY;
      for (int s2 = 0; s2 < kWarps * G; ++s2) gm = fmaxf(gm, s_m[s2]);
      float gl = 0.f, go = 0.f;
      for (int s2 = 0; s2 < kWarps * G; ++s2) {
        const float w = s_l[s2] > 0.f ? ex2(s_m[s2] - gm) : 0.f;
        gl += s_l[s2] * w;
        go += s_o[s2][c] * w;
      }
      if (nsplit == 1) {
        out[((int64_t)i * H + h) * D + c] = from_f32<T>(go / gl);
        if (lse && c == 0) lse[(int64_t)h * B + i] = (gm + __log2f(gl)) * kLn2;
      } else {
        float* dst = part + item * (D + 2);
        dst[2 + c] = go;
        if (c == 0) {
          dst[0] = gm;  // -inf, with l = 0, for a chunk past the sequence end
          dst[1] = gl;
        }
      }
    }
    __syncthreads();
  }
}

// Combines the chunk partials of each (sequence, head), one warp each, in
// chunk order: m = max m_s, l = sum l_s 2^(m_s - m), o = sum o_s 2^(m_s - m) / l.
template <typename T, int D>
__global__ void first_token_merge_kernel(const float* __restrict__ part, int32_t B, int32_t H,
                                         int32_t nsplit, T* __restrict__ out,
                                         float* __restrict__ lse,
                                         const DeviceStatus* __restrict__ status) {
  if (status->code != PE_OK) return;
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t ih = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
       ih < (int64_t)B * H; ih += warps) {
    const float* base = part + ih * nsplit * (D + 2);
    float gm = -INFINITY;
    for (int32_t s2 = 0; s2 < nsplit; ++s2) gm = fmaxf(gm, base[(int64_t)s2 * (D + 2)]);
    float gl = 0.f;
    for (int32_t s2 = 0; s2 < nsplit; ++s2) {
      const float* ps = base + (int64_t)s2 * (D + 2);
      if (ps[1] > 0.f) gl += ps[1] * ex2(ps[0] - gm);
    }
    const int32_t i = (int32_t)(ih / H), h = (int32_t)(ih - (int64_t)i * H);
    for (int c = lane; c < D; c += 32) {
      float go = 0.f;
      for (int32_t s2 = 0; s2 < nsplit; ++s2) {
        const float* ps = base + (int64_t)s2 * (D + 2);
        if (ps[1] > 0.f) go += ps[2 + c] * ex2(ps[0] - gm);
      }
      out[((int64_t)i * H + h) * D + c] = from_f32<T>(go / gl);
    }
    if (lse && lane == 0) lse[(int64_t)h * B + i] = (gm + __log2f(gl)) * kLn2;
  }
}

template <typename T, int D>
pe_status launch_first(const void* q, const void* k, const void* v, const int32_t* cu, int32_t B,
                       int32_t H, int32_t S, float scale, Window win, void* out, float* lse,
                       float* part, const DeviceStatus* status, cudaStream_t stream) {
  // With a window the query sees at most right + 1 keys.
  const int32_t key_limit = win.right == kUnbounded ? S : min(S, win.right + 1);
  // Without room for chunk partials every sequence is a single chunk.
  const int32_t nsplit = part ? first_token_splits(key_limit) : 1;
  const int64_t cap = (int64_t)device_sm_count() * 16;
  int64_t blocks = (int64_t)B * H * nsplit;
  if (blocks > cap) blocks = cap;
  fwd_first_token_kernel<T, D><<<(unsigned)blocks, kFtThreads, 0, stream>>>(
      static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v), cu, B, H,
      scale * kLog2e, key_limit, static_cast<T*>(out), lse, nsplit,
      nsplit == 1 ? key_limit : kFirstTokenChunk, part, status);
  PE_CUDA_TRY(cudaGetLastError());
  if (nsplit > 1) {
    int64_t mblocks = ceil_div((int64_t)B * H, 8);
    if (mblocks > cap) mblocks = cap;
    first_token_merge_kernel<T, D><<<(unsigned)mblocks, 256, 0, stream>>>(
        part, B, H, nsplit, static_cast<T*>(out), lse, status);
    PE_CUDA_TRY(cudaGetLastError());
  }
  return PE_OK;
}

template <typename T>
pe_status dispatch_first(int D, const void* q, const void* k, const void* v, const int32_t* cu,
                         int32_t B, int32_t H, int32_t S, float scale, Window win, void* out,
                         float* lse, float* part, const DeviceStatus* status,
                         cudaStream_t stream) {
  switch (D) {
#define PE_CASE(d)                                                                            \
  case d:                                                                                     \
    return launch_first<T, d>(q, k, v, cu, B, H, S, scale, win, out, lse, part, status, stream);
    PE_CASE(8) PE_CASE(16) PE_CASE(32) PE_CASE(64) PE_CASE(128)
#undef PE_CASE
    default: return PE_ERR_UNSUPPORTED;
  }
}

}  // namespace

int simt_rows_per_item() { return kItemRows; }

pe_status fwd_simt(pe_dtype dtype, int D, const void* q, const void* k, const void* v,
                   const int32_t* cu, int32_t B, int32_t H, float scale, Window win, void* out,
                   float* lse, int64_t N, TilePlan plan, cudaStream_t stream) {
  if (dtype == PE_FP32)
    return dispatch_full<float>(D, q, k, v, cu, B, H, scale, win, out, lse, N, plan, stream);
  return full_bf16(D, q, k, v, cu, B, H, scale, win, out, lse, N, plan, stream);
}

bool first_token_supported(int D) { return D == 8 || D == 16 || D == 32 || D == 64 || D == 128; }

pe_status fwd_first_token(pe_dtype dtype, int D, const void* q, const void* k, const void* v,
                          const int32_t* cu, int32_t B, int32_t H, int32_t S, float scale,
                          Window win, void* out, float* lse, float* part,
                          const DeviceStatus* status, cudaStream_t stream) {
  if (dtype == PE_FP32)
    return dispatch_first<float>(D, q, k, v, cu, B, H, S, scale, win, out, lse, part, status,
                                 stream);
  return dispatch_first<__nv_bfloat16>(D, q, k, v, cu, B, H, S, scale, win, out, lse, part,
                                       status, stream);
}

}  // namespace pe
