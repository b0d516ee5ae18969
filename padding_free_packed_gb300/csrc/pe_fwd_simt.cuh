// CUDA-core (FFMA) packed attention forward, full-query mode: the kernel
// template shared by the fp32 and bf16 translation units.
//
// The kernel serves fp32 inputs (the pages keep attention in fp32 because
// inference needs the accuracy: page "Source code for
// gigl.nn.packed_attention", function _varlen_attention) and bf16 inputs whose
// head_dim has no tensor-core kernel. Every sequence attends only to its own
// keys (module docstring, "Data flow of a packed forward").
//
// A persistent grid claims work items of 128 query rows of one (sequence,
// head) from the longest-first tile plan and runs them as two tiles of 64
// rows; when all of the sequence's keys fit in the staging buffers (at most
// two blocks of 64 for fp32, one for bf16), the second tile reuses the first
// tile's staged K and V instead of loading them again. Each CTA runs 256 threads as a 16 x 16 grid:
// thread (ty, tx) owns query rows ty + 16*ii and, per key block of 64, key
// columns tx + 16*jj (ii, jj < 4) of the score tile and output columns
// tx*CPT .. tx*CPT+CPT-1. Softmax is online, in the base-2 domain, with the
// row statistics reduced across the 16 tx lanes by warp shuffles.
//
// Short sequences: a tile with at most 32 real rows runs only ii < 2, and a
// key block with at most 32 real keys only jj < 2 (and P V only over its real
// keys rounded up to 4), so a sequence of ~90 tokens computes ~96 x 96 score
// elements instead of 128 x 128. The skipped products are those of padding
// rows and keys, whose results are never stored or are exactly zero.
//
// fp32 rows are copied to shared memory with cp.async into two K/V stages:
// block j+1 loads while block j is computed. bf16 rows are converted to fp32
// in registers into one stage.
//
// Local attention (a window of key positions around each query position)
// restricts the key blocks a tile visits to those its rows can see and masks
// the rest of those blocks per element.
#pragma once

#include <type_traits>

#include "pe_common.cuh"

namespace pe {
namespace fwd_simt_impl {

constexpr int kBM = 64;          // query rows per tile
constexpr int kItemRows = 2 * kBM;  // query rows per work item (two tiles)
constexpr int kBN = 64;          // keys per block
constexpr int kThreads = 256;    // 16 x 16
constexpr int kPsPitch = kBN + 16;  // fp32 words per row of P: a warp's two rows sit 16 banks apart

template <typename T, int D>
struct SimtShape {
  static constexpr int kPitch = D + 4;        // fp32 words per staged row
  static constexpr int kCPT = (D + 15) / 16;  // output columns per thread
  static constexpr bool kAsync = std::is_same<T, float>::value;
  static constexpr int kStages = kAsync ? 2 : 1;
  static constexpr size_t kSmemBytes =
      sizeof(float) * ((size_t)kBM * kPitch + 2 * kStages * (size_t)kBN * kPitch +
                       (size_t)kBM * kPsPitch);
};

__device__ __forceinline__ void cp_async16(float* smem, const float* gmem, bool valid) {
  const unsigned dst = (unsigned)__cvta_generic_to_shared(smem);
  // src-size 0 writes 16 zero bytes and reads nothing.
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(gmem),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_group 0;\n" ::: "memory");
}

// Copies 64 fp32 rows (row stride `stride` elements, D elements each) into
// smem[r * (D + 4) + c] asynchronously; rows >= rows_valid (>= 1) are zeroes.
template <int D>
__device__ __forceinline__ void stage_rows_async(float* __restrict__ smem,
                                                 const float* __restrict__ g, int64_t stride,
                                                 int rows_valid) {
  constexpr int kPitch = D + 4;
  constexpr int kVecPerRow = D / 4;
  for (int idx = threadIdx.x; idx < kBM * kVecPerRow; idx += kThreads) {
    const int r = idx / kVecPerRow, c = idx - r * kVecPerRow;
    const bool valid = r < rows_valid;
    cp_async16(smem + r * kPitch + c * 4, g + (int64_t)(valid ? r : 0) * stride + c * 4, valid);
  }
}

// Stages 64 rows (row stride `stride` elements) of D elements into
// smem[r * (D + 4) + c] as fp32 through registers; rows >= rows_valid are
// zero-filled. D is a multiple of 8, so every row is whole 16-byte loads.
template <typename T, int D>
__device__ __forceinline__ void stage_rows(float* __restrict__ smem, const T* __restrict__ g,
                                           int64_t stride, int rows_valid) {
  constexpr int kPitch = D + 4;
  constexpr int kVec = 16 / sizeof(T);  // elements per 16-byte load
  constexpr int kVecPerRow = D / kVec;
  static_assert(D % kVec == 0, "rows are whole 16-byte loads");
  for (int idx = threadIdx.x; idx < kBM * kVecPerRow; idx += kThreads) {
    const int r = idx / kVecPerRow, v = idx % kVecPerRow;
    float vals[kVec];
    if (r < rows_valid) {
      uint4 raw = *reinterpret_cast<const uint4*>(g + (int64_t)r * stride + v * kVec);
      const T* e = reinterpret_cast<const T*>(&raw);
#pragma unroll
      for (int u = 0; u < kVec; ++u) vals[u] = to_f32(e[u]);
    } else {
#pragma unroll
      for (int u = 0; u < kVec; ++u) vals[u] = 0.f;
    }
#pragma unroll
    for (int u = 0; u < kVec; u += 4)
      *reinterpret_cast<float4*>(smem + r * kPitch + v * kVec + u) =
          make_float4(vals[u], vals[u + 1], vals[u + 2], vals[u + 3]);
  }
}

// One key block of a tile: S = Q K^T over rows ii < NI and key columns
// jj < NJ, the online-softmax update, then O += P V over the block's real keys
// (rounded up to 4; P and V are zero past them).
template <int D, bool kLocal, int NI, int NJ>
__device__ __forceinline__ void attend_block(const float* __restrict__ Qs,
                                             const float* __restrict__ Ks,
                                             const float* __restrict__ Vs, float* __restrict__ Ps,
                                             int32_t kb, int keys_valid, float scale_log2,
                                             const int32_t (&vis_lo)[4], const int32_t (&vis_hi)[4],
                                             float (&m)[4], float (&l)[4],
                                             float (&o)[4][(D + 15) / 16], int tx, int ty,
                                             bool col_active) {
  constexpr int P = D + 4;
  constexpr int CPT = (D + 15) / 16;
  float s[NI][NJ];
#pragma unroll
  for (int ii = 0; ii < NI; ++ii)
#pragma unroll
    for (int jj = 0; jj < NJ; ++jj) s[ii][jj] = 0.f;
#pragma unroll 4
  for (int c = 0; c < D; c += 4) {
    float4 qv[NI], kv[NJ];
#pragma unroll
    for (int ii = 0; ii < NI; ++ii)
      qv[ii] = *reinterpret_cast<const float4*>(Qs + (ty + 16 * ii) * P + c);
#pragma unroll
    for (int jj = 0; jj < NJ; ++jj)
      kv[jj] = *reinterpret_cast<const float4*>(Ks + (tx + 16 * jj) * P + c);
#pragma unroll
    for (int ii = 0; ii < NI; ++ii)
#pragma unroll
      for (int jj = 0; jj < NJ; ++jj) {
        s[ii][jj] = fmaf(qv[ii].x, kv[jj].x, s[ii][jj]);
        s[ii][jj] = fmaf(qv[ii].y, kv[jj].y, s[ii][jj]);
        s[ii][jj] = fmaf(qv[ii].z, kv[jj].z, s[ii][jj]);
        s[ii][jj] = fmaf(qv[ii].w, kv[jj].w, s[ii][jj]);
      }
  }

  // Online softmax (base 2). Keys past the sequence end, or outside a row's
  // window, are excluded.
#pragma unroll
  for (int ii = 0; ii < NI; ++ii) {
    float bmax = -INFINITY;
#pragma unroll
    for (int jj = 0; jj < NJ; ++jj) {
      const int32_t kp = kb + tx + 16 * jj;
      const bool vis = (tx + 16 * jj < keys_valid) &&
                       (!kLocal || (kp >= vis_lo[ii] && kp <= vis_hi[ii]));
      s[ii][jj] = vis ? s[ii][jj] * scale_log2 : -INFINITY;
      bmax = fmaxf(bmax, s[ii][jj]);
    }
#pragma unroll
    for (int off = 1; off < 16; off <<= 1)
      bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, off));
    // -inf while a row has seen no visible key (possible with a window): then
    // exponents are taken against 0 and stay exactly 0. Without a window every
    // block holds a real key for every row.
    const float m_new = fmaxf(m[ii], bmax);
    const float m_use = (kLocal && m_new == -INFINITY) ? 0.f : m_new;
    const float corr = ex2(m[ii] - m_use);  // 0 while m = -inf
    float bsum = 0.f;
#pragma unroll
    for (int jj = 0; jj < NJ; ++jj) {
      const float p = ex2(s[ii][jj] - m_use);
      bsum += p;
      Ps[(ty + 16 * ii) * kPsPitch + tx + 16 * jj] = p;
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
    const int keys4 = (keys_valid + 3) & ~3;
#pragma unroll 2
    for (int j = 0; j < keys4; j += 4) {
      float4 pv[NI];
#pragma unroll
      for (int ii = 0; ii < NI; ++ii)
        pv[ii] = *reinterpret_cast<const float4*>(Ps + (ty + 16 * ii) * kPsPitch + j);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        float vv[CPT];
        const float* vrow = Vs + (j + u) * P + tx * CPT;
        if constexpr (CPT % 4 == 0) {
#pragma unroll
          for (int c = 0; c < CPT; c += 4) {
            const float4 x = *reinterpret_cast<const float4*>(vrow + c);
            vv[c] = x.x; vv[c + 1] = x.y; vv[c + 2] = x.z; vv[c + 3] = x.w;
          }
        } else {
#pragma unroll
          for (int c = 0; c < CPT; ++c) vv[c] = vrow[c];
        }
#pragma unroll
        for (int ii = 0; ii < NI; ++ii) {
          const float pw = u == 0 ? pv[ii].x : u == 1 ? pv[ii].y : u == 2 ? pv[ii].z : pv[ii].w;
#pragma unroll
          for (int c = 0; c < CPT; ++c) o[ii][c] = fmaf(pw, vv[c], o[ii][c]);
        }
      }
    }
  }
}

// One 64-row query tile of (sequence, head) with NI x 16 rows computed. With
// kv_resident the key blocks are already in the stages, in block order from
// stage 0 (full attention with at most kStages blocks), and are not staged again.
template <typename T, int D, bool kLocal, int NI>
__device__ __forceinline__ void attend_tile(const T* __restrict__ q, const T* __restrict__ k,
                                            const T* __restrict__ v, int32_t H, float scale_log2,
                                            Window win, T* __restrict__ out,
                                            float* __restrict__ lse, int64_t lse_stride,
                                            float* Qs, float* Ks0, float* Vs0, float* Ps,
                                            int32_t start, int32_t len, int32_t h, int32_t q0,
                                            int rows_valid, bool kv_resident) {
  using Shape = SimtShape<T, D>;
  constexpr int P = Shape::kPitch;
  constexpr int CPT = Shape::kCPT;
  constexpr int kStageFloats = kBN * P;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const bool col_active = tx * CPT < D;
  const int64_t row_stride = (int64_t)H * D;
  const T* kh = k + (int64_t)start * row_stride + (int64_t)h * D;
  const T* vh = v + (int64_t)start * row_stride + (int64_t)h * D;
  const T* qt = q + ((int64_t)(start + q0) * H + h) * D;

  // Keys any real row of the tile can see: from the first row's first
  // visible key to the last row's last one.
  const int32_t kb_begin = kLocal ? window_lo(win, q0) : 0;
  const int32_t kb_end = kLocal ? window_hi(win, q0 + rows_valid - 1, len) + 1 : len;

  if constexpr (Shape::kAsync) {
    stage_rows_async<D>(Qs, qt, row_stride, rows_valid);
    if (!kv_resident) {
      const int kv0 = min(kBN, kb_end - kb_begin);
      stage_rows_async<D>(Ks0, kh + (int64_t)kb_begin * row_stride, row_stride, kv0);
      stage_rows_async<D>(Vs0, vh + (int64_t)kb_begin * row_stride, row_stride, kv0);
    }
    cp_async_commit();
  } else {
    stage_rows<T, D>(Qs, qt, row_stride, rows_valid);
  }

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

  int stage = 0;
  for (int32_t kb = kb_begin; kb < kb_end; kb += kBN) {
    const int keys_valid = min(kBN, kb_end - kb);
    float* Ks = Ks0 + stage * kStageFloats;
    float* Vs = Vs0 + stage * kStageFloats;
    if constexpr (Shape::kAsync) {
      cp_async_wait_all();
      // This block's rows landed for every thread; the other stage and P are
      // no longer read by the previous block.
      __syncthreads();
      const int32_t nb = kb + kBN;
      if (!kv_resident && nb < kb_end) {
        const int nv = min(kBN, kb_end - nb);
        float* Kn = Ks0 + (stage ^ 1) * kStageFloats;
        float* Vn = Vs0 + (stage ^ 1) * kStageFloats;
        stage_rows_async<D>(Kn, kh + (int64_t)nb * row_stride, row_stride, nv);
        stage_rows_async<D>(Vn, vh + (int64_t)nb * row_stride, row_stride, nv);
      }
      cp_async_commit();
      stage ^= 1;
    } else {
      __syncthreads();  // previous block's Ks/Vs/Ps fully consumed
      if (!kv_resident) {
        stage_rows<T, D>(Ks, kh + (int64_t)kb * row_stride, row_stride, keys_valid);
        stage_rows<T, D>(Vs, vh + (int64_t)kb * row_stride, row_stride, keys_valid);
      }
      __syncthreads();
    }
    if (keys_valid > 32)
      attend_block<D, kLocal, NI, 4>(Qs, Ks, Vs, Ps, kb, keys_valid, scale_log2, vis_lo, vis_hi,
                                     m, l, o, tx, ty, col_active);
    else
      attend_block<D, kLocal, NI, 2>(Qs, Ks, Vs, Ps, kb, keys_valid, scale_log2, vis_lo, vis_hi,
                                     m, l, o, tx, ty, col_active);
  }

  // Epilogue: normalise, store real rows, write the natural-log lse.
#pragma unroll
  for (int ii = 0; ii < NI; ++ii) {
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

// kLocal selects the local-attention variant (key range and window masks);
// full attention compiles without them.
template <typename T, int D, bool kLocal>
__global__ void __launch_bounds__(kThreads)
fwd_simt_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                const int32_t* __restrict__ cu, int32_t B, int32_t H, float scale_log2,
                Window win, T* __restrict__ out, float* __restrict__ lse, int64_t lse_stride,
                TilePlan plan) {
  using Shape = SimtShape<T, D>;
  constexpr int P = Shape::kPitch;
  extern __shared__ float4 smem_raw[];
  float* Qs = reinterpret_cast<float*>(smem_raw);
  float* Ks0 = Qs + kBM * P;                          // [kStages][kBN][P]
  float* Vs0 = Ks0 + Shape::kStages * kBN * P;        // [kStages][kBN][P]
  float* Ps = Vs0 + Shape::kStages * kBN * P;         // [kBM][kPsPitch]
  __shared__ int32_t s_tile;

  const int32_t total = *plan.total_tiles;
  for (;;) {
    // The barrier also orders the previous tile's last reads of shared
    // memory before this tile's first writes.
    if (threadIdx.x == 0) s_tile = atomicAdd(plan.counter, 1);
    __syncthreads();
    const int32_t t = s_tile;
    if (t >= total) break;
    int32_t seq, local;
    plan_decode(plan.order, plan.tile_end, B, t, seq, local);
    const int32_t start = __ldg(cu + seq), len = __ldg(cu + seq + 1) - start;
    const int32_t nqb = (len + kItemRows - 1) / kItemRows;
    const int32_t h = local / nqb, qb = local - h * nqb;
    // The item's second tile keeps the staged keys when they are all of the
    // sequence's (full attention, at most kStages blocks).
    const bool reuse = !kLocal && len <= Shape::kStages * kBN;
    for (int32_t q0 = qb * kItemRows; q0 < min(len, (qb + 1) * kItemRows); q0 += kBM) {
      const int rows_valid = min(kBM, len - q0);
      const bool resident = reuse && q0 > qb * kItemRows;
      if (rows_valid > 32)
        attend_tile<T, D, kLocal, 4>(q, k, v, H, scale_log2, win, out, lse, lse_stride, Qs, Ks0,
                                     Vs0, Ps, start, len, h, q0, rows_valid, resident);
      else
        attend_tile<T, D, kLocal, 2>(q, k, v, H, scale_log2, win, out, lse, lse_stride, Qs, Ks0,
                                     Vs0, Ps, start, len, h, q0, rows_valid, resident);
    }
  }
}

template <typename T, int D>
pe_status launch_full(const void* q, const void* k, const void* v, const int32_t* cu, int32_t B,
                      int32_t H, float scale, Window win, void* out, float* lse, int64_t N,
                      TilePlan plan, cudaStream_t stream) {
  auto kernel = win.active() ? fwd_simt_kernel<T, D, true> : fwd_simt_kernel<T, D, false>;
  const size_t smem = SimtShape<T, D>::kSmemBytes;
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

// bf16 instantiation, compiled in its own translation unit.
pe_status full_bf16(int D, const void* q, const void* k, const void* v, const int32_t* cu,
                    int32_t B, int32_t H, float scale, Window win, void* out, float* lse,
                    int64_t N, TilePlan plan, cudaStream_t stream);

}  // namespace fwd_simt_impl
}  // namespace pe
