// CUDA-core (FFMA) packed attention backward kernels: the gradients in q, k and v that
// the custom op gigl::varlen_attention_backward returns (page "Source code for
// gigl.nn.packed_attention"), computed without floating-point atomics so the
// result is bitwise deterministic.
//
// With P = softmax(scale q k^T) recomputed from the saved log-sum-exp:
//   preprocess:  Delta_r = dO_r . O_r                      [H, Nq] fp32
//   key pass:    per (sequence, head, 64-key block), over the sequence's
//                query blocks: dV += P^T dO, dK += scale dS^T q
//   query pass:  per (sequence, head, 64-row query block), over key blocks:
//                dq += scale dS k
// where dS = P o (dO v^T - Delta). Both passes run 256 threads as a 16 x 16
// grid with 4 x 4 register micro-tiles over 64 x 64 score tiles staged in
// shared memory, and claim tiles from the longest-first plan. With local
// attention each pass visits only the blocks inside the window band and masks
// P (and so dS) to zero outside it.
//
// This header holds the two pass kernels, templated on head_dim and on the
// local-attention variant; pe_bwd_simt.cu instantiates full attention and the
// Delta preprocess, pe_bwd_simt_local.cu local attention.
#pragma once

#include "pe_common.cuh"

namespace pe {
namespace bwd_simt_impl {

constexpr int kB = 64;          // rows per block (queries or keys)
constexpr int kThreads = 256;   // 16 x 16
constexpr int kSP = kB + 4;     // pitch of the staged score tiles

template <int D>
struct BwdShape {
  static constexpr int kPitch = D + 4;
  static constexpr int kCPT = (D + 15) / 16;
  static constexpr size_t kSmemBytes =
      sizeof(float) * (4 * (size_t)kB * kPitch + 2 * (size_t)kB * kSP + 2 * (size_t)kB);
};

template <typename T, int D>
__device__ __forceinline__ void stage(float* __restrict__ smem, const T* __restrict__ g,
                                      int64_t stride, int rows_valid) {
  constexpr int kPitch = D + 4;
  constexpr int kVec = 16 / sizeof(T);
  constexpr int kVecPerRow = D / kVec;
  for (int idx = threadIdx.x; idx < kB * kVecPerRow; idx += kThreads) {
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
    for (int u = 0; u < kVec; ++u) smem[r * kPitch + v * kVec + u] = vals[u];
  }
}

// acc[a][b] += X[xa + 16a] . Y[yb + 16b] over D (rows of pitch D+4).
template <int D>
__device__ __forceinline__ void micro_dot(const float* __restrict__ X, int xa,
                                          const float* __restrict__ Y, int yb, float (&acc)[4][4]) {
  constexpr int P = D + 4;
#pragma unroll 4
  for (int c = 0; c < D; c += 4) {
    float4 xv[4], yv[4];
#pragma unroll
    for (int a = 0; a < 4; ++a) xv[a] = *reinterpret_cast<const float4*>(X + (xa + 16 * a) * P + c);
#pragma unroll
    for (int b = 0; b < 4; ++b) yv[b] = *reinterpret_cast<const float4*>(Y + (yb + 16 * b) * P + c);
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        acc[a][b] = fmaf(xv[a].x, yv[b].x, acc[a][b]);
        acc[a][b] = fmaf(xv[a].y, yv[b].y, acc[a][b]);
        acc[a][b] = fmaf(xv[a].z, yv[b].z, acc[a][b]);
        acc[a][b] = fmaf(xv[a].w, yv[b].w, acc[a][b]);
      }
  }
}

// out[a][c] += sum_r W[(wa + 16a) * kSP + r] * Z[r * P + zc + c], r < kB.
template <int D>
__device__ __forceinline__ void micro_acc(const float* __restrict__ W, int wa,
                                          const float* __restrict__ Z, int zc,
                                          float (&out)[4][BwdShape<D>::kCPT]) {
  constexpr int P = D + 4;
  constexpr int CPT = BwdShape<D>::kCPT;
#pragma unroll 2
  for (int r = 0; r < kB; r += 4) {
    float4 w4[4];
#pragma unroll
    for (int a = 0; a < 4; ++a) w4[a] = *reinterpret_cast<const float4*>(W + (wa + 16 * a) * kSP + r);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      float z[CPT];
#pragma unroll
      for (int c = 0; c < CPT; ++c) z[c] = Z[(r + u) * P + zc + c];
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const float w = u == 0 ? w4[a].x : u == 1 ? w4[a].y : u == 2 ? w4[a].z : w4[a].w;
#pragma unroll
        for (int c = 0; c < CPT; ++c) out[a][c] = fmaf(w, z[c], out[a][c]);
      }
    }
  }
}

struct BwdArgs {
  const void *q, *k, *v, *dout;
  const float *lse, *delta;
  void *dq, *dk, *dv;
  const int32_t* cu;
  int32_t B, H;
  int64_t Nq;
  float scale, scale_log2;
  int first_token;
  Window win;
  TilePlan plan;
  LayoutCheck check;  // for the tile plans (host side only)
};

// Visibility of key position kp from the query at position rp (local attention).
__device__ __forceinline__ bool visible(const Window& w, int32_t rp, int32_t kp, int32_t len) {
  return kp >= window_lo(w, rp) && kp <= window_hi(w, rp, len);
}

// Key pass: dK and dV for one 64-key block of one (sequence, head) per tile.
// kLocal selects the local-attention variant (block ranges and window masks).
template <typename T, int D, bool kLocal>
__global__ void __launch_bounds__(kThreads) bwd_dkdv_kernel(BwdArgs a) {
  constexpr int P = D + 4;
  constexpr int CPT = BwdShape<D>::kCPT;
  extern __shared__ float4 smem_raw[];
  float* Ks = reinterpret_cast<float*>(smem_raw);
  float* Vs = Ks + kB * P;
  float* Qs = Vs + kB * P;
  float* Gs = Qs + kB * P;     // dO
  float* PT = Gs + kB * P;     // P^T  [key][query]
  float* ST = PT + kB * kSP;   // dS^T [key][query]
  float* lse_s = ST + kB * kSP;
  float* dlt_s = lse_s + kB;
  __shared__ int32_t s_tile;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int64_t rs = (int64_t)a.H * D;
  const T* q = static_cast<const T*>(a.q);
  const T* k = static_cast<const T*>(a.k);
  const T* v = static_cast<const T*>(a.v);
  const T* g = static_cast<const T*>(a.dout);
  const int32_t total = *a.plan.total_tiles;
  const bool col_active = tx * CPT < D;

  for (;;) {
    if (threadIdx.x == 0) s_tile = atomicAdd(a.plan.counter, 1);
    __syncthreads();
    const int32_t t = s_tile;
    if (t >= total) break;
    int32_t seq, local;
    plan_decode(a.plan.order, a.plan.tile_end, a.B, t, seq, local);
    const int32_t start = __ldg(a.cu + seq), len = __ldg(a.cu + seq + 1) - start;
    const int32_t nkb = (len + kB - 1) / kB;
    const int32_t h = local / nkb, kb = local - h * nkb;
    const int32_t k0 = kb * kB;
    const int keys_valid = min(kB, len - k0);
    const int64_t q_first = a.first_token ? seq : start;   // first query row of the sequence
    const int32_t q_len = a.first_token ? 1 : len;
    // Query positions that can see a key of this block: [k0 - right, k_last + left]
    // (a first-token query sits at position 0).
    constexpr bool windowed = kLocal;
    int32_t qb_begin = 0, qb_end = q_len;
    if (windowed) {
      const int32_t k_last = k0 + keys_valid - 1;
      if (a.first_token) {
        qb_end = window_hi(a.win, 0, len) >= k0 ? 1 : 0;
      } else {
        const Window rev = {a.win.right, a.win.left};  // r sees kp  <=>  kp sees r reversed
        qb_begin = window_lo(rev, k0);
        qb_end = window_hi(rev, k_last, len) + 1;
      }
    }

    stage<T, D>(Ks, k + ((int64_t)(start + k0) * a.H + h) * D, rs, keys_valid);
    stage<T, D>(Vs, v + ((int64_t)(start + k0) * a.H + h) * D, rs, keys_valid);
    float dk[4][CPT], dv[4][CPT];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int c = 0; c < CPT; ++c) dk[i][c] = dv[i][c] = 0.f;

    for (int32_t qb = qb_begin; qb < qb_end; qb += kB) {
      const int rows_valid = min(kB, qb_end - qb);
      __syncthreads();
      stage<T, D>(Qs, q + ((q_first + qb) * a.H + h) * D, rs, rows_valid);
      stage<T, D>(Gs, g + ((q_first + qb) * a.H + h) * D, rs, rows_valid);
      if (threadIdx.x < kB) {
        const int r = threadIdx.x;
        const int64_t row = q_first + qb + r;
        lse_s[r] = r < rows_valid ? a.lse[(int64_t)h * a.Nq + row] * kLog2e : 0.f;
        dlt_s[r] = r < rows_valid ? a.delta[(int64_t)h * a.Nq + row] : 0.f;
      }
      __syncthreads();
      // Transposed tiles: key rows ty+16jj, query rows tx+16ii.
      float st[4][4] = {}, dpt[4][4] = {};
      micro_dot<D>(Ks, ty, Qs, tx, st);
      micro_dot<D>(Vs, ty, Gs, tx, dpt);
#pragma unroll
      for (int jj = 0; jj < 4; ++jj)
#pragma unroll
        for (int ii = 0; ii < 4; ++ii) {
          const int j = ty + 16 * jj, r = tx + 16 * ii;
          float p = 0.f, ds = 0.f;
          if (j < keys_valid && r < rows_valid &&
              (!windowed || visible(a.win, a.first_token ? 0 : qb + r, k0 + j, len))) {
            p = ex2(st[jj][ii] * a.scale_log2 - lse_s[r]);
            ds = p * (dpt[jj][ii] - dlt_s[r]);
          }
          PT[j * kSP + r] = p;
          ST[j * kSP + r] = ds;
        }
      __syncthreads();
      if (col_active) {
        micro_acc<D>(PT, ty, Gs, tx * CPT, dv);
        micro_acc<D>(ST, ty, Qs, tx * CPT, dk);
      }
    }
    T* dkp = static_cast<T*>(a.dk);
    T* dvp = static_cast<T*>(a.dv);
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      const int j = ty + 16 * jj;
      if (j < keys_valid && col_active) {
        const int64_t base = ((int64_t)(start + k0 + j) * a.H + h) * D + tx * CPT;
#pragma unroll
        for (int c = 0; c < CPT; ++c)
          if (tx * CPT + c < D) {
            dkp[base + c] = from_f32<T>(dk[jj][c] * a.scale);
            dvp[base + c] = from_f32<T>(dv[jj][c]);
          }
      }
    }
  }
}

// Query pass: dq for one 64-row query block of one (sequence, head) per tile.
template <typename T, int D, bool kLocal>
__global__ void __launch_bounds__(kThreads) bwd_dq_kernel(BwdArgs a) {
  constexpr int P = D + 4;
  constexpr int CPT = BwdShape<D>::kCPT;
  extern __shared__ float4 smem_raw[];
  float* Qs = reinterpret_cast<float*>(smem_raw);
  float* Gs = Qs + kB * P;
  float* Ks = Gs + kB * P;
  float* Vs = Ks + kB * P;
  float* Ss = Vs + kB * P;     // dS [query][key]
  float* lse_s = Ss + 2 * kB * kSP;
  float* dlt_s = lse_s + kB;
  __shared__ int32_t s_tile;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int64_t rs = (int64_t)a.H * D;
  const T* q = static_cast<const T*>(a.q);
  const T* k = static_cast<const T*>(a.k);
  const T* v = static_cast<const T*>(a.v);
  const T* g = static_cast<const T*>(a.dout);
  const int32_t total = *a.plan.total_tiles;
  const bool col_active = tx * CPT < D;

  for (;;) {
    if (threadIdx.x == 0) s_tile = atomicAdd(a.plan.counter, 1);
    __syncthreads();
    const int32_t t = s_tile;
    if (t >= total) break;
    int32_t seq, local;
    plan_decode(a.plan.order, a.plan.tile_end, a.B, t, seq, local);
    const int32_t start = __ldg(a.cu + seq), len = __ldg(a.cu + seq + 1) - start;
    const int32_t q_len = a.first_token ? 1 : len;
    const int32_t nqb = (q_len + kB - 1) / kB;
    const int32_t h = local / nqb, qb = local - h * nqb;
    const int64_t q_first = (a.first_token ? seq : start) + (int64_t)qb * kB;
    const int rows_valid = min(kB, q_len - qb * kB);

    stage<T, D>(Qs, q + (q_first * a.H + h) * D, rs, rows_valid);
    stage<T, D>(Gs, g + (q_first * a.H + h) * D, rs, rows_valid);
    if (threadIdx.x < kB) {
      const int r = threadIdx.x;
      lse_s[r] = r < rows_valid ? a.lse[(int64_t)h * a.Nq + q_first + r] * kLog2e : 0.f;
      dlt_s[r] = r < rows_valid ? a.delta[(int64_t)h * a.Nq + q_first + r] : 0.f;
    }
    float dq[4][CPT];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int c = 0; c < CPT; ++c) dq[i][c] = 0.f;
    // Keys the block's rows can see (query positions qb*64 .. , or 0 for a
    // first-token query).
    constexpr bool windowed = kLocal;
    const int32_t p0 = a.first_token ? 0 : qb * kB;
    const int32_t kb_begin = windowed ? window_lo(a.win, p0) : 0;
    const int32_t kb_end = windowed ? window_hi(a.win, p0 + rows_valid - 1, len) + 1 : len;

    for (int32_t kb = kb_begin; kb < kb_end; kb += kB) {
      const int keys_valid = min(kB, kb_end - kb);
      __syncthreads();
      stage<T, D>(Ks, k + ((int64_t)(start + kb) * a.H + h) * D, rs, keys_valid);
      stage<T, D>(Vs, v + ((int64_t)(start + kb) * a.H + h) * D, rs, keys_valid);
      __syncthreads();
      float s[4][4] = {}, dp[4][4] = {};
      micro_dot<D>(Qs, ty, Ks, tx, s);
      micro_dot<D>(Gs, ty, Vs, tx, dp);
#pragma unroll
      for (int ii = 0; ii < 4; ++ii)
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int r = ty + 16 * ii, j = tx + 16 * jj;
          float ds = 0.f;
          if (j < keys_valid && r < rows_valid &&
              (!windowed || visible(a.win, p0 + r, kb + j, len))) {
            const float p = ex2(s[ii][jj] * a.scale_log2 - lse_s[r]);
            ds = p * (dp[ii][jj] - dlt_s[r]);
          }
          Ss[r * kSP + j] = ds;
        }
      __syncthreads();
      if (col_active) micro_acc<D>(Ss, ty, Ks, tx * CPT, dq);
    }
    T* dqp = static_cast<T*>(a.dq);
#pragma unroll
    for (int ii = 0; ii < 4; ++ii) {
      const int r = ty + 16 * ii;
      if (r < rows_valid && col_active) {
        const int64_t base = ((q_first + r) * a.H + h) * D + tx * CPT;
#pragma unroll
        for (int c = 0; c < CPT; ++c)
          if (tx * CPT + c < D) dqp[base + c] = from_f32<T>(dq[ii][c] * a.scale);
      }
    }
  }
}

// The key pass and the query pass (Delta is already in place).
template <typename T, int D, bool kLocal>
pe_status launch_passes(const BwdArgs& a, TilePlan plan, int32_t B, cudaStream_t stream) {
  const size_t smem = BwdShape<D>::kSmemBytes;
  // Key pass.
  {
    auto kernel = bwd_dkdv_kernel<T, D, kLocal>;
    PE_CUDA_TRY(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    int per_sm = 0;
    PE_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, smem));
    if (per_sm < 1) return PE_ERR_UNSUPPORTED;
    PE_TRY(launch_tile_plan(a.cu, B, a.H, kB, 0, 0, plan, a.check, stream));
    kernel<<<device_sm_count() * per_sm, kThreads, smem, stream>>>(a);
    PE_CUDA_TRY(cudaGetLastError());
  }
  // Query pass (first-token mode: one single-row block per sequence and head).
  {
    auto kernel = bwd_dq_kernel<T, D, kLocal>;
    PE_CUDA_TRY(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    int per_sm = 0;
    PE_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, smem));
    if (per_sm < 1) return PE_ERR_UNSUPPORTED;
    PE_TRY(launch_tile_plan(a.cu, B, a.H, a.first_token ? 0x7fffffff : kB, 0, 0, plan, a.check,
                            stream));
    kernel<<<device_sm_count() * per_sm, kThreads, smem, stream>>>(a);
    PE_CUDA_TRY(cudaGetLastError());
  }
  return PE_OK;
}

template <typename T, bool kLocal>
pe_status dispatch_passes(int D, const BwdArgs& a, TilePlan plan, int32_t B, cudaStream_t stream) {
  switch (D) {
#define PE_CASE(d) case d: return launch_passes<T, d, kLocal>(a, plan, B, stream);
    PE_CASE(8) PE_CASE(16) PE_CASE(24) PE_CASE(32) PE_CASE(40) PE_CASE(48) PE_CASE(56)
    PE_CASE(64) PE_CASE(72) PE_CASE(80) PE_CASE(88) PE_CASE(96) PE_CASE(104) PE_CASE(112)
    PE_CASE(120) PE_CASE(128)
#undef PE_CASE
    default: return PE_ERR_UNSUPPORTED;
  }
}

// Local-attention passes, instantiated in their own translation unit
// (pe_bwd_simt_local.cu) so that the two variants compile in parallel.
pe_status passes_local(pe_dtype dtype, int D, const BwdArgs& a, TilePlan plan, int32_t B,
                       cudaStream_t stream);

}  // namespace bwd_simt_impl
}  // namespace pe
