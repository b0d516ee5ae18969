// Local (sliding-window) instantiation of the CUDA-core packed attention
// backward passes (kernels in pe_bwd_simt.cuh): each pass visits only the
// blocks inside the window band and zeroes P and dS outside each row's window.
#include "pe_bwd_simt.cuh"

namespace pe {
namespace bwd_simt_impl {

pe_status passes_local(pe_dtype dtype, int D, const BwdArgs& a, TilePlan plan, int32_t B,
                       cudaStream_t stream) {
  if (dtype == PE_FP32) return dispatch_passes<float, true>(D, a, plan, B, stream);
  return dispatch_passes<__nv_bfloat16, true>(D, a, plan, B, stream);
}

}  // namespace bwd_simt_impl
}  // namespace pe
