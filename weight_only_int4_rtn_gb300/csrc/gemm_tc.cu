// W4A16 GEMM: the single-problem bf16-activation instantiation of the
// tcgen05 kernel template, the launch dispatcher, configuration queries and
// the wait self test.
#include "gemm_tc.cuh"

namespace w4a16 {
namespace {

// One-thread kernel whose wait can never complete: exercises the bounded
// wait and the error word without faulting or hanging the GPU.
__global__ void wait_timeout_selftest_kernel(uint32_t* err, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    ptx::fence_mbar_init();
    abort_flag = 0;
    const WaitCtx wc{err, timeout_ns, &abort_flag};
    (void)wait_one(&bar, 0, wc);   // nobody arrives: times out
  }
}

}  // namespace

size_t gemm_smem_bytes(const GemmKernelConfig& c) {
  if (c.rb) return c.simt && c.weight_format == kFmtInt4 ? gemv_rb_smem_bytes(c.act_tile) : 0;
  if (c.simt) return gemv_smem_bytes(c);
#define W4A16_SMEM_CASE(BA, L, GRP, ST, UG)                                          \
  if (c.act_tile == BA && c.lanes == L && c.group_scale == GRP && c.stages == ST && \
      c.unit_groups == UG && c.weight_format == kFmtInt4)                                    \
    return Cfg<BA, L, GRP, ST, UG, kFmtInt4>::kSmem;
  W4A16_GEMM_INSTANCES(W4A16_SMEM_CASE)
#undef W4A16_SMEM_CASE
#define W8A16_SMEM_CASE(BA, L, GRP, ST, UG)                                          \
  if (c.act_tile == BA && c.lanes == L && c.group_scale == GRP && c.stages == ST && \
      c.unit_groups == UG && c.weight_format == kFmtInt8)                                    \
    return Cfg<BA, L, GRP, ST, UG, kFmtInt8>::kSmem;
  W8A16_GEMM_INSTANCES(W8A16_SMEM_CASE)
#undef W8A16_SMEM_CASE
#define FP4A16_SMEM_CASE(BA, L, GRP, ST, UG)                                         \
  if (c.act_tile == BA && c.lanes == L && c.group_scale == GRP && c.stages == ST && \
      c.unit_groups == UG && c.weight_format == kFmtMxfp4)                          \
    return Cfg<BA, L, GRP, ST, UG, kFmtMxfp4>::kSmem;                                \
  if (c.act_tile == BA && c.lanes == L && c.group_scale == GRP && c.stages == ST && \
      c.unit_groups == UG && c.weight_format == kFmtNvfp4)                          \
    return Cfg<BA, L, GRP, ST, UG, kFmtNvfp4>::kSmem;
  FP4A16_GEMM_INSTANCES(FP4A16_SMEM_CASE)
#undef FP4A16_SMEM_CASE
  return 0;
}

bool gemm_config_available(const GemmKernelConfig& c) { return gemm_smem_bytes(c) != 0; }

size_t gemm_workspace_bytes(const GemmKernelConfig& c, const GemmSchedule& s, int64_t M,
                            int64_t N, int64_t K) {
  (void)M;
  (void)N;
  (void)K;
  if (s.sk_units == 0) return 0;
  return kCounterBytes + static_cast<size_t>(s.grid) * 2 * c.act_tile * kTileW * sizeof(float);
}

cudaError_t launch_gemm_tc_group(const GemmKernelConfig& c, const GemmGroup& grp, bool use_pdl,
                                 cudaStream_t stream) {
  static_assert(kMaxGemmGroup == kMaxGroup, "group size of the kernel arguments");
  if (grp.count < 1 || grp.count > kMaxGroup) return cudaErrorInvalidValue;
  if (c.rb) return launch_gemv_rb(c, grp, use_pdl, stream);
  if (c.simt) return launch_gemv(c, grp, use_pdl, stream);
  bool any_sw = false;
  for (int i = 0; i < grp.count; ++i) any_sw = any_sw || grp.p[i].swiglu;
  if (any_sw)
    return grp.count == 1 ? launch_gemm_tc_swiglu(c, grp, use_pdl, stream)
                          : launch_gemm_tc_group_swiglu(c, grp, use_pdl, stream);
  if (c.weight_format == kFmtInt8) return launch_gemm_tc_w8(c, grp, use_pdl, stream);
  if (c.weight_format == kFmtMxfp4) return launch_gemm_tc_mxfp4(c, grp, use_pdl, stream);
  if (c.weight_format == kFmtNvfp4) return launch_gemm_tc_nvfp4(c, grp, use_pdl, stream);
  const bool f16 = grp.p[0].act_f16;
  if (grp.count == 1)
    return f16 ? launch_gemm_tc_f16(c, grp, use_pdl, stream)
               : launch_gemm_tc_typed<false, 1>(c, grp, use_pdl, stream);
  return f16 ? launch_gemm_tc_group_f16(c, grp, use_pdl, stream)
             : launch_gemm_tc_group_bf16(c, grp, use_pdl, stream);
}

cudaError_t launch_gemm_tc(const GemmKernelConfig& c, const GemmSchedule& s,
                           const GemmProblem& p, bool use_pdl, cudaStream_t stream) {
  GemmGroup grp;
  grp.count = 1;
  grp.p[0] = p;
  grp.s[0] = s;
  return launch_gemm_tc_group(c, grp, use_pdl, stream);
}

#ifdef W4A16_TRACE
extern "C" int w4a16_debug_set_trace(unsigned long long* buf) {
  return cudaMemcpyToSymbol(g_trace, &buf, sizeof(buf)) == cudaSuccess ? 0 : 1;
}
extern "C" int w4a16_debug_set_trace_units(unsigned long long* buf) {
  return cudaMemcpyToSymbol(g_trace_units, &buf, sizeof(buf)) == cudaSuccess ? 0 : 1;
}
#endif

cudaError_t launch_wait_timeout_selftest(uint32_t* error_word, uint64_t timeout_ns,
                                         cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(32);
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, wait_timeout_selftest_kernel, error_word, timeout_ns);
}

}  // namespace w4a16
