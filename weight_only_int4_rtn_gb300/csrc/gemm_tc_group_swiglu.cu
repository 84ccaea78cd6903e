// Grouped W4A16 GEMM with the SwiGLU epilogue available per problem: the
// tcgen05 kernel template instantiated for up to eight independent problems
// (bf16 activations, INT4 weights) in which a problem whose flag is set
// stores silu(gate) * up of its interleaved up/gate rows and the others store
// the plain GEMM, so an MLP block's gate/up projection runs in the same
// launch as its other projections ("Piper Kernels", section "ConvRot INT8":
// the SwiGLU of a raw [up | gate] tensor).
#include "gemm_tc.cuh"

namespace w4a16 {

cudaError_t launch_gemm_tc_group_swiglu(const GemmKernelConfig& c, const GemmGroup& grp,
                                        bool use_pdl, cudaStream_t stream) {
  if (c.simt || c.weight_format != kFmtInt4) return cudaErrorInvalidValue;
  for (int i = 0; i < grp.count; ++i)
    if (grp.p[i].act_f16) return cudaErrorInvalidValue;
  return launch_gemm_tc_typed<false, kMaxGroup, true>(c, grp, use_pdl, stream);
}

}  // namespace w4a16
