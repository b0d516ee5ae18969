// CUDA-core (FFMA) packed attention forward and the first-token-query kernel.
//
// The full-mode kernel serves fp32 inputs (the pages keep attention in fp32
// because inference needs the accuracy: page "Source code for
// gigl.nn.packed_attention", function _varlen_attention) and bf16 inputs whose
// head_dim has no tensor-core kernel. Every sequence attends only to its own
// keys (module docstring, "Data flow of a packed forward").
//
// Full mode: a persistent grid claims tiles of 64 query rows of one
// (sequence, head) from the longest-first tile plan. Each CTA runs 256 threads
// as a 16 x 16 grid: thread (ty, tx) owns query rows ty + 16*ii and, per key
// block of 64, key columns tx + 16*jj (ii, jj < 4) of the score tile and output
// columns tx*CPT .. tx*CPT+CPT-1. Softmax is online, in the base-2 domain, with
// the row statistics reduced across the 16 tx lanes by warp shuffles.
//
// Local attention (a window of key positions around each query position)
// restricts the key blocks a tile visits to those its rows can see and masks
// the rest of those blocks per element.
//
// First-token mode: the query of sequence i is one row, so the work is a
// matrix-vector product bounded by reading k and v once. One CTA per
// (sequence, head); lanes are grouped so that each group reads whole 16-byte
// slices of one key row; groups keep private online-softmax states that are
// merged at the end.
#include "pe_common.cuh"

namespace pe {

namespace {

constexpr int kBM = 64;        // query rows per tile
constexpr int kBN = 64;        // keys per block
constexpr int kThreads = 256;  // 16 x 16

template <int D>
struct SimtShape {
  static constexpr int kPitch = D + 4;                 // fp32 words per staged row
  static constexpr int kCPT = (D + 15) / 16;           // output columns per thread
  static constexpr size_t kSmemBytes =
      sizeof(float) * ((size_t)kBM * kPitch + 2 * (size_t)kBN * kPitch + (size_t)kBM * (kBN + 4));
};

// Stages `rows` rows (row stride `stride` elements) of D elements into
// smem[r * pitch + c] as fp32; rows >= rows_valid are zero-filled.
template <typename T, int D>
__device__ __forceinline__ void stage_rows(float* __restrict__ smem, const T* __restrict__ g,
                                           int64_t stride, int rows_valid) {
  constexpr int kPitch = SimtShape<D>::kPitch;
  constexpr int kVec = 16 / sizeof(T);  // elements per 16-byte load
  constexpr int kVecPerRow = D / kVec > 0 ? D / kVec : 1;
  constexpr int kElems = D < kVec ? D : kVec;
  for (int idx = threadIdx.x; idx < kBM * kVecPerRow; idx += kThreads) {
    const int r = idx / kVecPerRow, v = idx % kVecPerRow;
    float vals[kVec];
    if (r < rows_valid) {
      const T* src = g + (int64_t)r * stride + v * kVec;
      if constexpr (D >= kVec) {
        uint4 raw = *reinterpret_cast<const uint4*>(src);
        const T* e = reinterpret_cast<const T*>(&raw);
#pragma unroll
        for (int u = 0; u < kVec; ++u) vals[u] = to_f32(e[u]);
      } else {
#pragma unroll
        for (int u = 0; u < kElems; ++u) vals[u] = to_f32(src[u]);
      }
    } else {
#pragma unroll
      for (int u = 0; u < kVec; ++u) vals[u] = 0.f;
    }
#pragma unroll
    for (int u = 0; u < kElems; ++u) smem[r * kPitch + v * kVec + u] = vals[u];
  }
}

// kLocal selects the local-attention variant (key range and window masks);
// full attention compiles without them.
template <typename T, int D, bool kLocal>
__global__ void __launch_bounds__(kThreads)
fwd_simt_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                const int32_t* __restrict__ cu, int32_t B, int32_t H, float scale_log2,
                Window win, T* __restrict__ out, float* __restrict__ lse, int64_t lse_stride,
                TilePlan plan) {
  using Shape = SimtShape<D>;
  constexpr int P = Shape::kPitch;
  constexpr int CPT = Shape::kCPT;
  extern __shared__ float4 smem_raw[];
  float* Qs = reinterpret_cast<float*>(smem_raw);
  float* Ks = Qs + kBM * P;
  float* Vs = Ks + kBN * P;
  float* Ps = Vs + kBN * P;  // [kBM][kBN + 4]
  __shared__ int32_t s_tile;

  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int64_t row_stride = (int64_t)H * D;
  const int32_t total = *plan.total_tiles;
  const bool col_active = tx * CPT < D;

  for (;;) {
    if (threadIdx.x == 0) s_tile = atomicAdd(plan.counter, 1);
    __syncthreads();
    const int32_t t = s_tile;
    if (t >= total) break;
    int32_t seq, local;
    plan_decode(plan.order, plan.tile_end, B, t, seq, local);
    const int32_t start = __ldg(cu + seq), len = __ldg(cu + seq + 1) - start;
    const int32_t nqb = (len + kBM - 1) / kBM;
    const int32_t h = local / nqb, qb = local - h * nqb;
    const int32_t q0 = qb * kBM;
    const int rows_valid = min(kBM, len - q0);

    stage_rows<T, D>(Qs, q + ((int64_t)(start + q0) * H + h) * D, row_stride, rows_valid);

    float m[4], l[4], o[4][CPT];
    int32_t vis_lo[4], vis_hi[4];  // visible key positions of each row (local attention)
#pragma unroll
    for (int ii = 0; ii < 4; ++ii) {
      m[ii] = -INFINITY;
      l[ii] = 0.f;
#pragma unroll
      for (int c = 0; c < CPT; ++c) o[ii][c] = 0.f;
      vis_lo[ii] = window_lo(win, q0 + ty + 16 * ii);
      vis_hi[ii] = window_hi(win, q0 + ty + 16 * ii, len);
    }
    // Keys any real row of the tile can see: from the first row's first
    // visible key to the last row's last one.
    constexpr bool windowed = kLocal;
    const int32_t kb_begin = windowed ? window_lo(win, q0) : 0;
    const int32_t kb_end = windowed ? window_hi(win, q0 + rows_valid - 1, len) + 1 : len;

    for (int32_t kb = kb_begin; kb < kb_end; kb += kBN) {
      const int keys_valid = min(kBN, kb_end - kb);
      __syncthreads();  // previous block's Ks/Vs/Ps fully consumed
      stage_rows<T, D>(Ks, k + ((int64_t)(start + kb) * H + h) * D, row_stride, keys_valid);
      stage_rows<T, D>(Vs, v + ((int64_t)(start + kb) * H + h) * D, row_stride, keys_valid);
      __syncthreads();

      // S = Q K^T for rows ty+16ii, keys tx+16jj.
      float s[4][4];
#pragma unroll
      for (int ii = 0; ii < 4; ++ii)
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) s[ii][jj] = 0.f;
#pragma unroll 4
      for (int c = 0; c < D; c += 4) {
        float4 qv[4], kv[4];
#pragma unroll
        for (int ii = 0; ii < 4; ++ii)
          qv[ii] = *reinterpret_cast<const float4*>(Qs + (ty + 16 * ii) * P + c);
#pragma unroll
        for (int jj = 0; jj < 4; ++jj)
          kv[jj] = *reinterpret_cast<const float4*>(Ks + (tx + 16 * jj) * P + c);
#pragma unroll
        for (int ii = 0; ii < 4; ++ii)
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            s[ii][jj] = fmaf(qv[ii].x, kv[jj].x, s[ii][jj]);
            s[ii][jj] = fmaf(qv[ii].y, kv[jj].y, s[ii][jj]);
            s[ii][jj] = fmaf(qv[ii].z, kv[jj].z, s[ii][jj]);
            s[ii][jj] = fmaf(qv[ii].w, kv[jj].w, s[ii][jj]);
          }
      }

      // Online softmax (base 2). Keys past the sequence end, or outside a
      // row's window, are excluded.
#pragma unroll
      for (int ii = 0; ii < 4; ++ii) {
        float bmax = -INFINITY;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int32_t kp = kb + tx + 16 * jj;
          const bool vis = (tx + 16 * jj < keys_valid) &&
                           (!windowed || (kp >= vis_lo[ii] && kp <= vis_hi[ii]));
          s[ii][jj] = vis ? s[ii][jj] * scale_log2 : -INFINITY;
          bmax = fmaxf(bmax, s[ii][jj]);
        }
#pragma unroll
        for (int off = 1; off < 16; off <<= 1)
          bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, off));
        // -inf while a row has seen no visible key (possible with a window):
        // then exponents are taken against 0 and stay exactly 0. Without a
        // window every block holds a real key for every row.
        const float m_new = fmaxf(m[ii], bmax);
        const float m_use = (kLocal && m_new == -INFINITY) ? 0.f : m_new;
        const float corr = ex2(m[ii] - m_use);   // 0 while m = -inf
        float bsum = 0.f;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const float p = ex2(s[ii][jj] - m_use);
          bsum += p;
          Ps[(ty + 16 * ii) * (kBN + 4) + tx + 16 * jj] = p;
        }
#pragma unroll
        for (int off = 1; off < 16; off <<= 1) bsum += __shfl_xor_sync(0xffffffffu, bsum, off);
        l[ii] = l[ii] * corr + bsum;
        m[ii] = m_new;
#pragma unroll
        for (int c = 0; c < CPT; ++c) o[ii][c] *= corr;
      }
      __syncthreads();

      // O += P V for rows ty+16ii, columns tx*CPT + c.
      if (col_active) {
#pragma unroll 2
        for (int j = 0; j < kBN; j += 4) {
          float4 pv[4];
#pragma unroll
          for (int ii = 0; ii < 4; ++ii)
            pv[ii] = *reinterpret_cast<const float4*>(Ps + (ty + 16 * ii) * (kBN + 4) + j);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            float vv[CPT];
#pragma unroll
            for (int c = 0; c < CPT; ++c) vv[c] = Vs[(j + u) * P + tx * CPT + c];
#pragma unroll
            for (int ii = 0; ii < 4; ++ii) {
              const float pw = u == 0 ? pv[ii].x : u == 1 ? pv[ii].y : u == 2 ? pv[ii].z : pv[ii].w;
#pragma unroll
              for (int c = 0; c < CPT; ++c) o[ii][c] = fmaf(pw, vv[c], o[ii][c]);
            }
          }
        }
      }
    }

    // Epilogue: normalise, store real rows, write the natural-log lse.
#pragma unroll
    for (int ii = 0; ii < 4; ++ii) {
      const int r = ty + 16 * ii;
      if (r < rows_valid) {
        const int64_t tok = start + q0 + r;
        const float inv = 1.f / l[ii];
        if (col_active) {
          T* dst = out + (tok * H + h) * D + tx * CPT;
#pragma unroll
          for (int c = 0; c < CPT; ++c)
            if (tx * CPT + c < D) dst[c] = from_f32<T>(o[ii][c] * inv);
        }
        if (lse && tx == 0) lse[(int64_t)h * lse_stride + tok] = (m[ii] + __log2f(l[ii])) * kLn2;
      }
    }
  }
}

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
                       int32_t nsplit, int32_t chunk, float* __restrict__ part) {
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
                                         float* __restrict__ lse) {
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
pe_status launch_full(const void* q, const void* k, const void* v, const int32_t* cu, int32_t B,
                      int32_t H, float scale, Window win, void* out, float* lse, int64_t N,
                      TilePlan plan, cudaStream_t stream) {
  auto kernel = win.active() ? fwd_simt_kernel<T, D, true> : fwd_simt_kernel<T, D, false>;
  const size_t smem = SimtShape<D>::kSmemBytes;
  PE_CUDA_TRY(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  int per_sm = 0;
  PE_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, smem));
  if (per_sm < 1) return PE_ERR_UNSUPPORTED;
  kernel<<<device_sm_count() * per_sm, kThreads, smem, stream>>>(
      static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v), cu, B, H,
      scale * kLog2e, win, static_cast<T*>(out), lse, N, plan);
  PE_CUDA_TRY(cudaGetLastError());
  return PE_OK;
}

template <typename T, int D>
pe_status launch_first(const void* q, const void* k, const void* v, const int32_t* cu, int32_t B,
                       int32_t H, int32_t S, float scale, Window win, void* out, float* lse,
                       float* part, cudaStream_t stream) {
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
      nsplit == 1 ? key_limit : kFirstTokenChunk, part);
  PE_CUDA_TRY(cudaGetLastError());
  if (nsplit > 1) {
    int64_t mblocks = ceil_div((int64_t)B * H, 8);
    if (mblocks > cap) mblocks = cap;
    first_token_merge_kernel<T, D><<<(unsigned)mblocks, 256, 0, stream>>>(
        part, B, H, nsplit, static_cast<T*>(out), lse);
    PE_CUDA_TRY(cudaGetLastError());
  }
  return PE_OK;
}

template <typename T>
pe_status dispatch_full(int D, const void* q, const void* k, const void* v, const int32_t* cu,
                        int32_t B, int32_t H, float scale, Window win, void* out, float* lse,
                        int64_t N, TilePlan plan, cudaStream_t stream) {
  switch (D) {
#define PE_CASE(d) \
  case d: return launch_full<T, d>(q, k, v, cu, B, H, scale, win, out, lse, N, plan, stream);
    PE_CASE(8) PE_CASE(16) PE_CASE(24) PE_CASE(32) PE_CASE(40) PE_CASE(48) PE_CASE(56)
    PE_CASE(64) PE_CASE(72) PE_CASE(80) PE_CASE(88) PE_CASE(96) PE_CASE(104) PE_CASE(112)
    PE_CASE(120) PE_CASE(128)
#undef PE_CASE
    default: return PE_ERR_UNSUPPORTED;
  }
}

template <typename T>
pe_status dispatch_first(int D, const void* q, const void* k, const void* v, const int32_t* cu,
                         int32_t B, int32_t H, int32_t S, float scale, Window win, void* out,
                         float* lse, float* part, cudaStream_t stream) {
  switch (D) {
#define PE_CASE(d) \
  case d: return launch_first<T, d>(q, k, v, cu, B, H, S, scale, win, out, lse, part, stream);
    PE_CASE(8) PE_CASE(16) PE_CASE(32) PE_CASE(64) PE_CASE(128)
#undef PE_CASE
    default: return PE_ERR_UNSUPPORTED;
  }
}

}  // namespace

int simt_rows_per_tile() { return kBM; }

pe_status fwd_simt(pe_dtype dtype, int D, const void* q, const void* k, const void* v,
                   const int32_t* cu, int32_t B, int32_t H, float scale, Window win, void* out,
                   float* lse, int64_t N, TilePlan plan, cudaStream_t stream) {
  if (dtype == PE_FP32)
    return dispatch_full<float>(D, q, k, v, cu, B, H, scale, win, out, lse, N, plan, stream);
  return dispatch_full<__nv_bfloat16>(D, q, k, v, cu, B, H, scale, win, out, lse, N, plan,
                                      stream);
}

bool first_token_supported(int D) { return D == 8 || D == 16 || D == 32 || D == 64 || D == 128; }

pe_status fwd_first_token(pe_dtype dtype, int D, const void* q, const void* k, const void* v,
                          const int32_t* cu, int32_t B, int32_t H, int32_t S, float scale,
                          Window win, void* out, float* lse, float* part, TilePlan /*plan*/,
                          cudaStream_t stream) {
  if (dtype == PE_FP32)
    return dispatch_first<float>(D, q, k, v, cu, B, H, S, scale, win, out, lse, part, stream);
  return dispatch_first<__nv_bfloat16>(D, q, k, v, cu, B, H, S, scale, win, out, lse, part,
                                       stream);
}

}  // namespace pe
