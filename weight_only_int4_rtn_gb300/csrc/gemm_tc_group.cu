// Grouped W4A16 GEMM, bf16 activations: the tcgen05 kernel template
// instantiated with arguments for up to eight independent problems (each on
// its own sub-grid of CTAs).
#include "gemm_tc.cuh"

namespace w4a16 {

cudaError_t launch_gemm_tc_group_bf16(const GemmKernelConfig& c, const GemmGroup& grp,
                                      bool use_pdl, cudaStream_t stream) {
  return launch_gemm_tc_typed<false, kMaxGroup>(c, grp, use_pdl, stream);
}

#ifdef W4A16_TRACE
// profiling builds: this unit's copy of the CTA timestamp buffer
extern "C" int w4a16_debug_set_trace_group(unsigned long long* buf) {
  return cudaMemcpyToSymbol(g_trace, &buf, sizeof(buf)) == cudaSuccess ? 0 : 1;
}
#endif

}  // namespace w4a16
