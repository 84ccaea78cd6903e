// W4A16 GEMM with the SwiGLU epilogue: the instantiation of the tcgen05
// kernel template whose epilogue stores silu(gate) * up for interleaved up
// and gate weight rows (an MLP's SwiGLU of a raw [up | gate] tensor, "Piper
// Kernels", section "ConvRot INT8", fused into the GEMM that produces it).
// One problem, INT4 weights, bf16 activations; the same configurations as the
// plain GEMM.
#include "gemm_tc.cuh"

namespace w4a16 {

cudaError_t launch_gemm_tc_swiglu(const GemmKernelConfig& c, const GemmGroup& grp, bool use_pdl,
                                  cudaStream_t stream) {
  if (grp.count != 1 || c.simt || c.weight_format != kFmtInt4 || grp.p[0].act_f16)
    return cudaErrorInvalidValue;
  return launch_gemm_tc_typed<false, 1, true>(c, grp, use_pdl, stream);
}

}  // namespace w4a16
