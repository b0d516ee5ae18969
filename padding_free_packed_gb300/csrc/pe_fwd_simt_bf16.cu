// bf16 instances of the full-query FFMA attention forward (pe_fwd_simt.cuh),
// for head dimensions without a tensor-core kernel; a translation unit of
// their own so they compile in parallel with the fp32 instances.
#include "pe_fwd_simt.cuh"

namespace pe {
namespace fwd_simt_impl {

pe_status full_bf16(int D, const void* q, const void* k, const void* v, const int32_t* cu,
                    int32_t B, int32_t H, float scale, Window win, void* out, float* lse,
                    int64_t N, TilePlan plan, cudaStream_t stream) {
  return dispatch_full<__nv_bfloat16>(D, q, k, v, cu, B, H, scale, win, out, lse, N, plan,
                                      stream);
}

}  // namespace fwd_simt_impl
}  // namespace pe
