// W4A16 GEMM with fp16 activations: the fp16 instantiation of the tcgen05
// kernel template ("Kernel dispatch and Humming quantization in PhyAI",
// section "Humming makes the separation useful": activations stay BF16 or
// FP16).  Weights are the same INT4 codes and fp16 scales; the weight operand
// is built as fp16, A, bias and Y are fp16.
#include "gemm_tc.cuh"

namespace w4a16 {

cudaError_t launch_gemm_tc_f16(const GemmKernelConfig& c, const GemmGroup& grp, bool use_pdl,
                               cudaStream_t stream) {
  return launch_gemm_tc_typed<true, 1>(c, grp, use_pdl, stream);
}

}  // namespace w4a16
