// FP4 weight-only GEMM: the tcgen05 kernel template instantiated with
// MXFP4 weights (E2M1 codes, one E8M0 scale byte per 32 values; OCP MX v1.0), bf16 activations ("Kernel dispatch and
// Humming quantization in PhyAI", section "Choose precision by layer and
// hardware").  Dequant mode: the dequant warps build bf16 e2m1 * block scale
// operands in TMEM; the rest is the INT4 pipeline.
#include "gemm_tc.cuh"

namespace w4a16 {

cudaError_t launch_gemm_tc_mxfp4(const GemmKernelConfig& c, const GemmGroup& grp, bool use_pdl,
                                 cudaStream_t stream) {
  if (grp.count != 1 || grp.p[0].act_f16) return cudaErrorInvalidValue;
  return launch_gemm_tc_fp4_typed<kFmtMxfp4>(c, grp, use_pdl, stream);
}

}  // namespace w4a16
