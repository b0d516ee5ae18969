// The packed encoder layer tail on the flat [N, ...] token buffer (page
// "packed-encoders 0.1.0": fused LayerNorm / residual-LayerNorm / RoPE / GeGLU
// kernels whose token count is a runtime grid dimension; position ids restart
// at every sequence, section "Fully packed execution"). The formulas are
// ModernBERT's:
//   RoPE (split-half): for i < D/2 and a = pos * theta^(-2i/D),
//     out[i] = x[i] cos a - x[i+D/2] sin a, out[i+D/2] = x[i+D/2] cos a + x[i] sin a;
//   LayerNorm: y = (h - mean) / sqrt(var + eps) * w (+ b), biased variance;
//     residual-LayerNorm: h = x + residual, stored (rounded to the I/O type)
//     and normalised as stored;
//   GeGLU: y[f] = gelu(x[f]) * x[F + f], exact (erf) GELU.
// Every call is asynchronous on its stream, allocates nothing and reads
// nothing back, so a whole layer tail can be captured in a CUDA graph. All
// are bandwidth kernels: each element is read once from HBM and written once.
#include <math.h>

#include "pe_common.cuh"

namespace pe {

namespace {

constexpr int kThreads = 256;

// pos[cu_i + j] = j: one block per sequence (grid-stride).
__global__ void packed_positions_kernel(const int32_t* __restrict__ cu, int32_t B,
                                        int32_t* __restrict__ pos) {
  for (int64_t i = blockIdx.x; i < B; i += gridDim.x) {
    const int32_t start = __ldg(cu + i), len = __ldg(cu + i + 1) - start;
    for (int32_t j = threadIdx.x; j < len; j += blockDim.x) pos[start + j] = j;
  }
}

// Vectors of V elements, moved as 16 bytes when V * sizeof(T) == 16.
template <typename T, int V>
struct Vec {
  T e[V];
};

template <typename T, int V>
__device__ __forceinline__ Vec<T, V> load_vec(const T* p) {
  Vec<T, V> v;
  if constexpr (V * sizeof(T) == 16) {
    *reinterpret_cast<uint4*>(v.e) = *reinterpret_cast<const uint4*>(p);
  } else {
#pragma unroll
    for (int u = 0; u < V; ++u) v.e[u] = p[u];
  }
  return v;
}

template <typename T, int V>
__device__ __forceinline__ void store_vec(T* p, const Vec<T, V>& v) {
  if constexpr (V * sizeof(T) == 16) {
    *reinterpret_cast<uint4*>(p) = *reinterpret_cast<const uint4*>(v.e);
  } else {
#pragma unroll
    for (int u = 0; u < V; ++u) p[u] = v.e[u];
  }
}

// One warp per token. The angle pos * theta^(-2i/D) of each frequency i is
// reduced modulo 2 pi in double precision once per token (lane i), shared by
// all heads of q and k through a per-warp table of cosines and sines, so the
// fp32 sine and cosine keep full accuracy at long positions (an fp32 product
// alone would be off by ~pos * 2^-24 radians). The frequencies in turns per
// position, theta^(-2i/D) / (2 pi), come from the host in double precision.
// Lanes then move V consecutive pairs of one head at a time (16-byte vectors
// from both halves of the row when the half-width allows it, else V = 1).
constexpr int kMaxHalf = 128;         // head_dim <= 256

struct RopeTurns {
  double t[kMaxHalf];
};

template <typename T, int V>
__global__ void __launch_bounds__(kThreads)
rope_kernel(T* __restrict__ q, int32_t hq, T* __restrict__ k, int32_t hk,
            const int32_t* __restrict__ pos, int64_t N, int32_t D, const RopeTurns turns) {
  __shared__ float table[kThreads / 32][2][kMaxHalf];   // per warp: cos, sin
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int32_t half = D / 2, chunks = half / V, items = (hq + hk) * chunks;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  constexpr double kTwoPi = 6.283185307179586476925;
  float* cs = table[warp][0];
  float* sn = table[warp][1];
  for (int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + warp; t < N; t += warps) {
    const double p = (double)__ldg(pos + t);
    for (int32_t i = lane; i < half; i += 32) {
      const double a = p * turns.t[i];                      // in turns
      const float r = (float)((a - rint(a)) * kTwoPi);      // in radians, |r| <= pi
      sincosf(r, &sn[i], &cs[i]);
    }
    __syncwarp();
    for (int32_t item = lane; item < items; item += 32) {
      const int32_t h = item / chunks, i0 = (item - h * chunks) * V;
      T* v = h < hq ? q + (t * hq + h) * D : k + (t * hk + (h - hq)) * D;
      Vec<T, V> x1 = load_vec<T, V>(v + i0), x2 = load_vec<T, V>(v + i0 + half);
#pragma unroll
      for (int u = 0; u < V; ++u) {
        const float a1 = to_f32(x1.e[u]), a2 = to_f32(x2.e[u]);
        const float c = cs[i0 + u], s2 = sn[i0 + u];
        x1.e[u] = from_f32<T>(a1 * c - a2 * s2);
        x2.e[u] = from_f32<T>(a2 * c + a1 * s2);
      }
      store_vec<T, V>(v + i0, x1);
      store_vec<T, V>(v + i0 + half, x2);
    }
    __syncwarp();                                           // the table is rewritten next token
  }
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

// One warp per row of C channels. h = x (+ residual, rounded to T); the mean,
// then the variance as the mean of squared deviations, then the output - three
// passes over the row, of which only the first reaches HBM. Lanes move V
// consecutive channels at a time (16-byte vectors when C and the pointers
// allow, else V = 1).
template <typename T, int V>
__global__ void __launch_bounds__(kThreads)
layernorm_kernel(const T* __restrict__ x, const T* __restrict__ res, const T* __restrict__ w,
                 const T* __restrict__ b, int64_t N, int32_t C, float eps, T* __restrict__ y,
                 T* __restrict__ res_out) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < N;
       t += warps) {
    const T* xr = x + t * C;
    const T* rr = res ? res + t * C : nullptr;
    // h of channels c .. c+V-1, as stored in res_out.
    auto h_at = [&](int32_t c, float (&h)[V]) {
      const Vec<T, V> xv = load_vec<T, V>(xr + c);
      if (rr) {
        const Vec<T, V> rv = load_vec<T, V>(rr + c);
#pragma unroll
        for (int u = 0; u < V; ++u) h[u] = to_f32(from_f32<T>(to_f32(xv.e[u]) + to_f32(rv.e[u])));
      } else {
#pragma unroll
        for (int u = 0; u < V; ++u) h[u] = to_f32(xv.e[u]);
      }
    };
    float sum = 0.f;
    for (int32_t c = lane * V; c < C; c += 32 * V) {
      float h[V];
      h_at(c, h);
      if (res_out) {
        Vec<T, V> hv;
#pragma unroll
        for (int u = 0; u < V; ++u) hv.e[u] = from_f32<T>(h[u]);
        store_vec<T, V>(res_out + t * C + c, hv);
      }
#pragma unroll
      for (int u = 0; u < V; ++u) sum += h[u];
    }
    const float mean = warp_sum(sum) / (float)C;
    float sq = 0.f;
    for (int32_t c = lane * V; c < C; c += 32 * V) {
      float h[V];
      h_at(c, h);
#pragma unroll
      for (int u = 0; u < V; ++u) {
        const float d = h[u] - mean;
        sq = fmaf(d, d, sq);
      }
    }
    const float rstd = rsqrtf(warp_sum(sq) / (float)C + eps);
    for (int32_t c = lane * V; c < C; c += 32 * V) {
      float h[V];
      h_at(c, h);
      const Vec<T, V> wv = load_vec<T, V>(w + c);
      Vec<T, V> out;
#pragma unroll
      for (int u = 0; u < V; ++u)
        out.e[u] = from_f32<T>((h[u] - mean) * rstd * to_f32(wv.e[u]) +
                               (b ? to_f32(b[c + u]) : 0.f));
      store_vec<T, V>(y + t * C + c, out);
    }
  }
}

// Rows of C = 32 * V * kIter channels held in registers: every load of the
// row (and residual) is issued before any arithmetic, then mean, variance and
// output come from registers, so a row costs one round trip to memory.
template <typename T, int V, int kIter>
__global__ void __launch_bounds__(kThreads)
layernorm_row_kernel(const T* __restrict__ x, const T* __restrict__ res, const T* __restrict__ w,
                     const T* __restrict__ b, int64_t N, float eps, T* __restrict__ y,
                     T* __restrict__ res_out) {
  constexpr int32_t C = 32 * V * kIter;
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < N;
       t += warps) {
    Vec<T, V> xv[kIter], rv[kIter];
#pragma unroll
    for (int it = 0; it < kIter; ++it) xv[it] = load_vec<T, V>(x + t * C + (it * 32 + lane) * V);
    if (res) {
#pragma unroll
      for (int it = 0; it < kIter; ++it)
        rv[it] = load_vec<T, V>(res + t * C + (it * 32 + lane) * V);
    }
    // h (= x, or x + residual rounded to T as stored in res_out) is kept in
    // T: exact, and half the registers for bf16.
    float sum = 0.f;
#pragma unroll
    for (int it = 0; it < kIter; ++it) {
      if (res) {
#pragma unroll
        for (int u = 0; u < V; ++u)
          xv[it].e[u] = from_f32<T>(to_f32(xv[it].e[u]) + to_f32(rv[it].e[u]));
      }
      if (res_out) store_vec<T, V>(res_out + t * C + (it * 32 + lane) * V, xv[it]);
#pragma unroll
      for (int u = 0; u < V; ++u) sum += to_f32(xv[it].e[u]);
    }
    const float mean = warp_sum(sum) / (float)C;
    float sq = 0.f;
#pragma unroll
    for (int it = 0; it < kIter; ++it)
#pragma unroll
      for (int u = 0; u < V; ++u) {
        const float d = to_f32(xv[it].e[u]) - mean;
        sq = fmaf(d, d, sq);
      }
    const float rstd = rsqrtf(warp_sum(sq) / (float)C + eps);
#pragma unroll
    for (int it = 0; it < kIter; ++it) {
      const int32_t c = (it * 32 + lane) * V;
      const Vec<T, V> wv = load_vec<T, V>(w + c);
      Vec<T, V> bv;
      if (b) bv = load_vec<T, V>(b + c);
      Vec<T, V> out;
#pragma unroll
      for (int u = 0; u < V; ++u)
        out.e[u] = from_f32<T>((to_f32(xv[it].e[u]) - mean) * rstd * to_f32(wv.e[u]) +
                               (b ? to_f32(bv.e[u]) : 0.f));
      store_vec<T, V>(y + t * C + c, out);
    }
  }
}

// Exact (erf) GELU, gelu(a) = a/2 (1 + erf(a / sqrt 2)), with erf from
// Abramowitz and Stegun, Handbook of Mathematical Functions, formula 7.1.26:
// for z >= 0, erf(z) = 1 - (a1 t + a2 t^2 + a3 t^3 + a4 t^4 + a5 t^5) e^(-z^2)
// with t = 1 / (1 + p z) and an absolute error of at most 1.5e-7. With
// q = (a1 t + ... + a5 t^5) e^(-z^2) and z = |a| / sqrt 2, 1 + erf is 2 - q for
// a >= 0 and q for a < 0 (no cancellation; the error stays absolute, as with
// 1 + erff). One reciprocal and one exponential replace the longer erff
// evaluation, which made this kernel issue-bound.
__device__ __forceinline__ float gelu_exact(float a) {
  constexpr float kP = 0.3275911f;
  constexpr float kA1 = 0.254829592f, kA2 = -0.284496736f, kA3 = 1.421413741f,
                  kA4 = -1.453152027f, kA5 = 1.061405429f;
  const float z = fabsf(a) * 0.70710678118654752f;
  const float t = __fdividef(1.f, fmaf(kP, z, 1.f));
  const float poly = t * fmaf(t, fmaf(t, fmaf(t, fmaf(t, kA5, kA4), kA3), kA2), kA1);
  const float q = poly * ex2(-(z * z) * kLog2e);
  return 0.5f * a * (a >= 0.f ? 2.f - q : q);
}

// y[t, f] = gelu(x[t, f]) * x[t, F + f]; V consecutive features per thread
// (16-byte vectors when the row and pointers allow it, else V = 1). With
// vectors a thread loads two of them (two grid strides apart) before it
// computes either, to keep more bytes in flight.
// Idx is the index type: 32-bit when N * F / V fits, so that splitting a
// vector index into (token, feature) is a 32-bit division.
template <typename T, int V, typename Idx>
__global__ void __launch_bounds__(kThreads)
geglu_kernel(const T* __restrict__ x, Idx N, int32_t F, T* __restrict__ y) {
  const Idx per_row = (Idx)(F / V);
  const Idx total = N * per_row;
  const Idx stride = (Idx)gridDim.x * blockDim.x;
  Idx e = (Idx)blockIdx.x * blockDim.x + threadIdx.x;
  if constexpr (V > 1) {
    for (; e < total - min(total, stride); e += 2 * stride) {  // e + stride < total
      const Idx e2 = e + stride;
      const Idx q1 = e / per_row, q2 = e2 / per_row;
      const int32_t f1 = (int32_t)(e - q1 * per_row) * V, f2 = (int32_t)(e2 - q2 * per_row) * V;
      const int64_t t1 = q1, t2 = q2;
      const T* a1 = x + t1 * 2 * F + f1;
      const T* a2 = x + t2 * 2 * F + f2;
      const uint4 av1 = *reinterpret_cast<const uint4*>(a1);
      const uint4 gv1 = *reinterpret_cast<const uint4*>(a1 + F);
      const uint4 av2 = *reinterpret_cast<const uint4*>(a2);
      const uint4 gv2 = *reinterpret_cast<const uint4*>(a2 + F);
      T o1[V], o2[V];
      const T* ae1 = reinterpret_cast<const T*>(&av1);
      const T* ge1 = reinterpret_cast<const T*>(&gv1);
      const T* ae2 = reinterpret_cast<const T*>(&av2);
      const T* ge2 = reinterpret_cast<const T*>(&gv2);
#pragma unroll
      for (int u = 0; u < V; ++u) {
        o1[u] = from_f32<T>(gelu_exact(to_f32(ae1[u])) * to_f32(ge1[u]));
        o2[u] = from_f32<T>(gelu_exact(to_f32(ae2[u])) * to_f32(ge2[u]));
      }
      *reinterpret_cast<uint4*>(y + t1 * F + f1) = *reinterpret_cast<const uint4*>(o1);
      *reinterpret_cast<uint4*>(y + t2 * F + f2) = *reinterpret_cast<const uint4*>(o2);
    }
  }
  for (; e < total; e += stride) {
    const Idx q = e / per_row;
    const int32_t f = (int32_t)(e - q * per_row) * V;
    const int64_t t = q;
    const T* a = x + t * 2 * F + f;
    const T* g = a + F;
    T out[V];
    if constexpr (V > 1) {
      uint4 av = *reinterpret_cast<const uint4*>(a), gv = *reinterpret_cast<const uint4*>(g);
      const T* ae = reinterpret_cast<const T*>(&av);
      const T* ge = reinterpret_cast<const T*>(&gv);
#pragma unroll
      for (int u = 0; u < V; ++u) out[u] = from_f32<T>(gelu_exact(to_f32(ae[u])) * to_f32(ge[u]));
      *reinterpret_cast<uint4*>(y + t * F + f) = *reinterpret_cast<const uint4*>(out);
    } else {
      y[t * F + f] = from_f32<T>(gelu_exact(to_f32(a[0])) * to_f32(g[0]));
    }
  }
}

unsigned grid_for(int64_t units_per_block_work, int64_t units) {
  int64_t blocks = ceil_div(units, units_per_block_work);
  const int64_t cap = (int64_t)device_sm_count() * 16;
  if (blocks > cap) blocks = cap;
  return (unsigned)(blocks > 0 ? blocks : 1);
}

template <typename T>
pe_status launch_rope(void* q, int32_t hq, void* k, int32_t hk, const int32_t* pos, int64_t N,
                      int32_t D, double theta, cudaStream_t stream) {
  RopeTurns turns;
  const double two_pi = 6.283185307179586476925;
  for (int i = 0; i < kMaxHalf; ++i)
    turns.t[i] = i < D / 2 ? pow(theta, -2.0 * i / D) / two_pi : 0.0;
  constexpr int V = 16 / sizeof(T);
  const unsigned grid = grid_for(kThreads / 32, N);
  const bool vec = (D / 2) % V == 0 && aligned(q, 16) && (!k || aligned(k, 16));
  if (vec)
    rope_kernel<T, V><<<grid, kThreads, 0, stream>>>(static_cast<T*>(q), hq, static_cast<T*>(k),
                                                      hk, pos, N, D, turns);
  else
    rope_kernel<T, 1><<<grid, kThreads, 0, stream>>>(static_cast<T*>(q), hq, static_cast<T*>(k),
                                                      hk, pos, N, D, turns);
  PE_CUDA_TRY(cudaGetLastError());
  return PE_OK;
}

template <typename T>
pe_status launch_layernorm(const void* x, const void* res, const void* w, const void* b,
                           int64_t N, int32_t C, float eps, void* y, void* res_out,
                           cudaStream_t stream) {
  constexpr int V = 16 / sizeof(T);
  const bool vec = C % V == 0 && aligned(x, 16) && aligned(w, 16) && aligned(y, 16) &&
                   (!res || aligned(res, 16)) && (!res_out || aligned(res_out, 16));
  // Whole rows in registers when a row is 1..8 warp-wide vectors.
  const int32_t iters = C / (32 * V);
  if (vec && C % (32 * V) == 0 && iters >= 1 && iters <= 8 && (!b || aligned(b, 16))) {
    const unsigned grid = grid_for(kThreads / 32, N);
    const T* xt = static_cast<const T*>(x);
    const T* rt = static_cast<const T*>(res);
    const T* wt = static_cast<const T*>(w);
    const T* bt = static_cast<const T*>(b);
    T* yt = static_cast<T*>(y);
    T* ot = static_cast<T*>(res_out);
    switch (iters) {
#define PE_CASE(n)                                                                          \
  case n:                                                                                   \
    layernorm_row_kernel<T, V, n><<<grid, kThreads, 0, stream>>>(xt, rt, wt, bt, N, eps, yt, \
                                                                 ot);                       \
    break;
      PE_CASE(1) PE_CASE(2) PE_CASE(3) PE_CASE(4) PE_CASE(5) PE_CASE(6) PE_CASE(7) PE_CASE(8)
#undef PE_CASE
    }
    PE_CUDA_TRY(cudaGetLastError());
    return PE_OK;
  }
  auto kernel = vec ? layernorm_kernel<T, V> : layernorm_kernel<T, 1>;
  kernel<<<grid_for(kThreads / 32, N), kThreads, 0, stream>>>(
      static_cast<const T*>(x), static_cast<const T*>(res), static_cast<const T*>(w),
      static_cast<const T*>(b), N, C, eps, static_cast<T*>(y), static_cast<T*>(res_out));
  PE_CUDA_TRY(cudaGetLastError());
  return PE_OK;
}

template <typename T>
pe_status launch_geglu(const void* x, int64_t N, int32_t F, void* y, cudaStream_t stream) {
  constexpr int V = 16 / sizeof(T);
  // 32-bit indices while every vector index and the grid stride past it fit.
  const bool idx32 = N * F < (1LL << 31);
  if (F % V == 0 && aligned(x, 16) && aligned(y, 16)) {
    const unsigned grid = grid_for(kThreads, N * (F / V));
    if (idx32)
      geglu_kernel<T, V, uint32_t><<<grid, kThreads, 0, stream>>>(
          static_cast<const T*>(x), (uint32_t)N, F, static_cast<T*>(y));
    else
      geglu_kernel<T, V, int64_t><<<grid, kThreads, 0, stream>>>(
          static_cast<const T*>(x), N, F, static_cast<T*>(y));
  } else {
    const unsigned grid = grid_for(kThreads, N * F);
    if (idx32)
      geglu_kernel<T, 1, uint32_t><<<grid, kThreads, 0, stream>>>(
          static_cast<const T*>(x), (uint32_t)N, F, static_cast<T*>(y));
    else
      geglu_kernel<T, 1, int64_t><<<grid, kThreads, 0, stream>>>(
          static_cast<const T*>(x), N, F, static_cast<T*>(y));
  }
  PE_CUDA_TRY(cudaGetLastError());
  return PE_OK;
}

bool dtype_ok(pe_dtype d) { return d == PE_BF16 || d == PE_FP32; }

}  // namespace

}  // namespace pe

using namespace pe;

extern "C" pe_status pe_packed_positions(const int32_t* cu_seqlens, int32_t B, int64_t N,
                                         int32_t* positions, pe_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (B < 0 || N < 0 || N >= (1LL << 31)) return PE_ERR_INVALID_ARG;
  if (B == 0 || N == 0) return PE_OK;
  if (!cu_seqlens || !positions) return PE_ERR_INVALID_ARG;
  if (!device_is_sm103()) return PE_ERR_UNSUPPORTED;
  const int64_t cap = (int64_t)device_sm_count() * 16;
  packed_positions_kernel<<<(unsigned)(B < cap ? B : cap), kThreads, 0, stream>>>(cu_seqlens, B,
                                                                                 positions);
  PE_CUDA_TRY(cudaGetLastError());
  return PE_OK;
}

extern "C" pe_status pe_rope_packed(pe_dtype dtype, void* q, int32_t q_heads, void* k,
                                    int32_t k_heads, const int32_t* positions, int64_t N,
                                    int32_t head_dim, double theta, pe_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (!dtype_ok(dtype)) return PE_ERR_UNSUPPORTED;
  if (N < 0 || q_heads < 0 || k_heads < 0 || head_dim < 2 || head_dim % 2 != 0 ||
      head_dim > 2 * kMaxHalf ||
      !(theta > 1.0) || !isfinite(theta))
    return PE_ERR_INVALID_ARG;
  if (!k) k_heads = 0;
  if (N == 0 || (q_heads == 0 && k_heads == 0)) return PE_OK;
  if (!positions || (q_heads > 0 && !q)) return PE_ERR_INVALID_ARG;
  if (!device_is_sm103()) return PE_ERR_UNSUPPORTED;
  if (dtype == PE_FP32)
    return launch_rope<float>(q, q_heads, k, k_heads, positions, N, head_dim, theta, stream);
  return launch_rope<__nv_bfloat16>(q, q_heads, k, k_heads, positions, N, head_dim, theta, stream);
}

extern "C" pe_status pe_layernorm(pe_dtype dtype, const void* x, const void* residual,
                                  const void* weight, const void* bias, int64_t N, int32_t C,
                                  float eps, void* y, void* residual_out, pe_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (!dtype_ok(dtype)) return PE_ERR_UNSUPPORTED;
  if (N < 0 || C < 1 || !(eps > 0.f) || !isfinite(eps)) return PE_ERR_INVALID_ARG;
  if (N == 0) return PE_OK;
  if (!x || !weight || !y || (residual_out && !residual)) return PE_ERR_INVALID_ARG;
  if (!device_is_sm103()) return PE_ERR_UNSUPPORTED;
  if (dtype == PE_FP32)
    return launch_layernorm<float>(x, residual, weight, bias, N, C, eps, y, residual_out, stream);
  return launch_layernorm<__nv_bfloat16>(x, residual, weight, bias, N, C, eps, y, residual_out,
                                         stream);
}

extern "C" pe_status pe_geglu(pe_dtype dtype, const void* x, int64_t N, int32_t F, void* y,
                              pe_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (!dtype_ok(dtype)) return PE_ERR_UNSUPPORTED;
  if (N < 0 || F < 1) return PE_ERR_INVALID_ARG;
  if (N == 0) return PE_OK;
  if (!x || !y) return PE_ERR_INVALID_ARG;
  if (!device_is_sm103()) return PE_ERR_UNSUPPORTED;
  if (dtype == PE_FP32) return launch_geglu<float>(x, N, F, y, stream);
  return launch_geglu<__nv_bfloat16>(x, N, F, y, stream);
}
