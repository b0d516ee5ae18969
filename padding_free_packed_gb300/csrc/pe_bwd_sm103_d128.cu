// Packed attention backward on the sm_103a tensor cores, head_dim 128, full
// or local attention (the kernel, templated on head_dim, is in
// pe_bwd_sm103.cuh).
#include "pe_bwd_sm103.cuh"

namespace pe {

pe_status bwd_sm103_d128(const void* q, const void* k, const void* v, const int32_t* cu,
                         int32_t B, int32_t H, int64_t N, float scale, Window win,
                         const float* lse, const void* dout, const float* delta, void* dq,
                         void* dk, void* dv, TilePlan plan, LayoutCheck check,
                         cudaStream_t stream) {
  return bwd_sm103_impl<128>(q, k, v, cu, B, H, N, scale, win, lse, dout, delta, dq, dk, dv,
                             plan, check, stream);
}

}  // namespace pe
