// W8A16 GEMM: the tcgen05 kernel template instantiated with INT8 weights
// and bf16 activations ("Kernel dispatch and Humming quantization in PhyAI",
// section "Choose precision by layer and hardware": INT8 is one of the
// Humming weight schemes).  The weight operand is built from one byte per
// code (16 KiB per 128 x 128 tile, 128-byte rows with the 128-byte swizzle);
// everything else is the INT4 pipeline.
#include "gemm_tc.cuh"

namespace w4a16 {

cudaError_t launch_gemm_tc_w8(const GemmKernelConfig& c, const GemmGroup& grp, bool use_pdl,
                              cudaStream_t stream) {
  if (grp.count != 1 || grp.p[0].act_f16) return cudaErrorInvalidValue;
  return launch_gemm_tc_w8_typed<kFmtInt8>(c, grp, use_pdl, stream);
}

}  // namespace w4a16
