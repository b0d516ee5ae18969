// CUDA-core (FFMA) packed attention backward: the gradients in q, k and v that
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
// This file holds the Delta preprocess and the full-attention instantiation
// of the two passes (kernels in pe_bwd_simt.cuh).
#include "pe_bwd_simt.cuh"

namespace pe {

using namespace bwd_simt_impl;

namespace {

// Delta[h, r] = sum_c dO[r, h, c] * O[r, h, c]; one warp per (row, head).
template <typename T>
__global__ void bwd_preprocess_kernel(const T* __restrict__ out, const T* __restrict__ dout,
                                      int64_t Nq, int32_t H, int D, float* __restrict__ delta) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); w < Nq * H;
       w += warps) {
    const T* o = out + w * D;
    const T* g = dout + w * D;
    float acc = 0.f;
    for (int c = lane; c < D; c += 32) acc = fmaf(to_f32(o[c]), to_f32(g[c]), acc);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) {
      const int64_t r = w / H;
      const int32_t h = (int32_t)(w - r * H);
      delta[(int64_t)h * Nq + r] = acc;
    }
  }
}

}  // namespace

// Delta for bf16 rows of D (64 or 128): D/8 lanes per (row, head), each
// reading 16 bytes of O and of dO, 256/D rows per warp per step; the row loop
// is warp-uniform so the group reduction always sees all 32 lanes.
template <int D>
__global__ void bwd_preprocess_bf16_kernel(const __nv_bfloat16* __restrict__ out,
                                           const __nv_bfloat16* __restrict__ dout, int64_t Nq,
                                           int32_t H, float* __restrict__ delta) {
  constexpr int kLanes = D / 8, kRowsPerWarp = 32 / kLanes;
  const int lane = threadIdx.x & 31, group = lane / kLanes, sub = lane % kLanes;
  const int64_t rows = Nq * H;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t base = ((int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * kRowsPerWarp;
       base < rows; base += warps * kRowsPerWarp) {
    const int64_t w = base + group;
    float acc = 0.f;
    if (w < rows) {
      const uint4 a = __ldg(reinterpret_cast<const uint4*>(out + w * D) + sub);
      const uint4 b = __ldg(reinterpret_cast<const uint4*>(dout + w * D) + sub);
      const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&a);
      const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float2 fa = __bfloat1622float2(pa[u]), fb = __bfloat1622float2(pb[u]);
        acc = fmaf(fa.x, fb.x, acc);
        acc = fmaf(fa.y, fb.y, acc);
      }
    }
#pragma unroll
    for (int off = 1; off < kLanes; off <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (w < rows && sub == 0) {
      const int64_t r = w / H;
      const int32_t h = (int32_t)(w - r * H);
      delta[(int64_t)h * Nq + r] = acc;
    }
  }
}

pe_status bwd_preprocess(pe_dtype dtype, int D, const void* out, const void* dout, int64_t Nq,
                         int32_t H, float* delta, cudaStream_t stream) {
  if (dtype != PE_BF16 || (D != 64 && D != 128)) return PE_ERR_UNSUPPORTED;
  const int64_t rows_per_block = 8 * (256 / D);  // 8 warps
  int64_t blocks = ceil_div(Nq * H, rows_per_block);
  const int64_t cap = (int64_t)device_sm_count() * 8;
  if (blocks > cap) blocks = cap;
  if (blocks <= 0) return PE_OK;
  const auto* o = static_cast<const __nv_bfloat16*>(out);
  const auto* g = static_cast<const __nv_bfloat16*>(dout);
  if (D == 64)
    bwd_preprocess_bf16_kernel<64><<<(unsigned)blocks, 256, 0, stream>>>(o, g, Nq, H, delta);
  else
    bwd_preprocess_bf16_kernel<128><<<(unsigned)blocks, 256, 0, stream>>>(o, g, Nq, H, delta);
  PE_CUDA_TRY(cudaGetLastError());
  return PE_OK;
}

pe_status bwd_simt(pe_dtype dtype, int D, const void* q, const void* k, const void* v,
                   const int32_t* cu, int32_t B, int32_t H, int64_t Nq, float scale,
                   int first_token, Window win, const void* out, const float* lse,
                   const void* dout, void* dq, void* dk, void* dv, float* delta, TilePlan plan,
                   LayoutCheck check, cudaStream_t stream) {
  BwdArgs a;
  a.q = q; a.k = k; a.v = v; a.dout = dout;
  a.lse = lse; a.delta = delta;
  a.dq = dq; a.dk = dk; a.dv = dv;
  a.cu = cu; a.B = B; a.H = H; a.Nq = Nq;
  a.scale = scale; a.scale_log2 = scale * kLog2e;
  a.first_token = first_token;
  a.win = win;
  a.plan = plan;
  a.check = check;
  // Delta.
  int64_t blocks = ceil_div(Nq * H, 8);
  const int64_t cap = (int64_t)device_sm_count() * 8;
  if (blocks > cap) blocks = cap;
  if (blocks > 0) {
    if (dtype == PE_FP32)
      bwd_preprocess_kernel<float><<<(unsigned)blocks, 256, 0, stream>>>(
          static_cast<const float*>(out), static_cast<const float*>(dout), Nq, H, D, delta);
    else
      bwd_preprocess_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, 0, stream>>>(
          static_cast<const __nv_bfloat16*>(out), static_cast<const __nv_bfloat16*>(dout), Nq, H,
          D, delta);
    PE_CUDA_TRY(cudaGetLastError());
  }
  if (win.active()) return passes_local(dtype, D, a, plan, B, stream);
  if (dtype == PE_FP32) return dispatch_passes<float, false>(D, a, plan, B, stream);
  return dispatch_passes<__nv_bfloat16, false>(D, a, plan, B, stream);
}

}  // namespace pe

