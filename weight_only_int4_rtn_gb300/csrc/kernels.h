// Internal launch interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace w4a16 {

constexpr int kGroup = 128;     // quantization group along K
constexpr int kTileW = 128;     // weight rows per GEMM tile (tcgen05 M)

// Weight formats: INT4 and INT8 codes with fp16 group scales; E2M1 codes (in
// the INT4 tile layout) with E8M0 scales per 32 values (MXFP4) or E4M3 scales
// per 16 values and an fp32 tensor scale (NVFP4).
constexpr int kFmtInt4 = 4;
constexpr int kFmtInt8 = 8;
constexpr int kFmtMxfp4 = 41;
constexpr int kFmtNvfp4 = 42;

// RTN quantize/pack; one launch.  sr_seed non-null: INT4 stochastic rounding
// with that seed (same scales and storage).  int8: the INT8 scheme (8-bit
// codes, 16 KiB tiles).
cudaError_t launch_rtn_quantize(const void* W, int64_t N, int64_t K, void* packed, void* scales,
                                int num_sms, uint32_t* error_word, uint64_t timeout_ns,
                                cudaStream_t stream, const uint64_t* sr_seed = nullptr,
                                bool int8 = false);

// FP4 quantize (format kFmtMxfp4 or kFmtNvfp4): codes in the INT4 tile
// layout, scale bytes [K/32, N] or [K/16, N].  NVFP4 also writes
// tensor_scale[0] = g and tensor_scale[1] = the tensor absmax (a memset, an
// absmax kernel, then the quantize kernel).
cudaError_t launch_fp4_quantize(const void* W, int64_t N, int64_t K, void* packed, void* scales,
                                float* tensor_scale, int format, int num_sms,
                                uint32_t* error_word, uint64_t timeout_ns, cudaStream_t stream);

// Several weights quantized in one launch (independent problems).
constexpr int kMaxQuantizeGroup = 8;
struct QuantizeProblem {
  const void* W;   // [N, K] bf16
  int64_t N, K;
  void* packed;    // tiled codes
  void* scales;    // [K/128, N] fp16
};
cudaError_t launch_rtn_quantize_group(const QuantizeProblem* probs, int count, int num_sms,
                                      uint32_t* error_word, uint64_t timeout_ns,
                                      cudaStream_t stream, const uint64_t* sr_seed = nullptr,
                                      bool int8 = false);

// One configuration of the tcgen05 GEMM kernel.
struct GemmKernelConfig {
  int act_tile;      // activation rows per tile (tcgen05 N): 16..256
  int lanes;         // independent pipelines (1 or 2), each with its own MMA
                     // issuing thread; units alternate between them
  bool group_scale;  // true: per-group fp32 scaling of integer-code partial sums
                     // false: weights dequantized to bf16(q*s) before the MMA
  int stages;        // shared-memory pipeline depth (all lanes together)
  int unit_groups = 1;  // k-groups per pipeline unit (1 or 2): one copy of the
                        // codes, scales and activations per unit
  int weight_format = kFmtInt4;  // kFmtInt4 (W4A16), kFmtInt8 (W8A16), kFmtMxfp4,
                                 // kFmtNvfp4 (FP4 weights, dequant mode)
  bool simt = false;  // a streaming kernel without tcgen05 pipeline roles for M <=
                      // act_tile, INT4 weights: the CUDA-core stream-K workers
                      // (gemv.cu, act_tile 1, 2, 4 or 8), or with rb:
  bool rb = false;    // the row-block warp-MMA kernel (gemv_rb.cu, act_tile 1, 2,
                      // 4, 8 or 16)
};

// The CUDA-core streaming kernel: every warp is a stream-K worker with two
// shared-memory stages of its own (9.1, 9.9, 11.5 or 14.8 KiB for M <= 1, 2,
// 4, 8); warps per CTA and the workers resident per SM that its schedules
// count on.
constexpr int gemv_warps_per_cta(int act_tile) { return act_tile <= 4 ? 4 : 2; }
constexpr int gemv_workers_per_sm(int act_tile) {
  return act_tile <= 1 ? 12 : act_tile <= 4 ? 8 : 6;
}

// The schedule of one launch.
struct GemmSchedule {
  int grid;          // CTAs (one per SM at most)
  int dp_tiles;      // tiles 0..dp_tiles-1 run whole, tile t on CTA t % grid
  int64_t sk_units;  // the remaining tiles' (tile, k-block) units, split in
                     // contiguous balanced ranges over all CTAs
  int cluster = 0;   // > 1: cluster split-K instead (dp_tiles = sk_units = 0):
                     // grid = tiles * cluster, tile t's K range split over the
                     // cluster CTAs t * cluster .. + cluster - 1 of one
                     // thread-block cluster, summed through distributed
                     // shared memory (no workspace)
  int team = 8;      // row-block kernel: warps splitting one row block's K
                     // range (1, 2, 4, 8; 8 with a cluster split)
};

struct GemmProblem {
  const void* A;       // [M, K] bf16
  const void* packed;  // [N, K/2] u8
  const void* scales;  // [K/128, N] fp16, or FP4 block-scale bytes [K/32 | K/16, N]
  const void* bias;    // [N] bf16 or null
  void* Y;             // [M, N] bf16
  int64_t M, N, K;
  void* workspace;
  size_t workspace_bytes;
  uint32_t* counters = nullptr;   // arrival counters of this problem's split tiles
                                  // (kCountersPerProblem words of the workspace's
                                  // fixed counter region)
  float* partials = nullptr;      // this problem's partial-tile slots
  uint32_t* error_word;
  uint64_t timeout_ns;
  bool act_f16 = false;  // A, bias and Y are fp16 (else bf16)
  const float* tensor_scale = nullptr;   // NVFP4: the fp32 tensor scale g (device)
  bool swiglu = false;   // SwiGLU epilogue: rows 2f (up) and 2f + 1 (gate) give
                         // Y[M, N/2][f] = silu(gate) * up
  bool weights_static = false;   // no kernel that may run just before this launch
                                 // on its stream writes packed or scales: the GEMM
                                 // may read them before the dependency wait
};

// Number of tiles of a problem under a configuration.
inline int64_t gemm_tiles(const GemmKernelConfig& c, int64_t M, int64_t N) {
  return ((N + kTileW - 1) / kTileW) * ((M + c.act_tile - 1) / c.act_tile);
}

// Workspace layout: kCounterBytes of uint32 counters (problem i of a launch
// owns words i * kCountersPerProblem .. + kCountersPerProblem - 1: one
// arrival counter per split tile; the region has a fixed size so every
// variant finds them at the same place), then [grid][2][act_tile][128] fp32
// partial slots (slot 0: the first stream-K tile of a CTA's range, slot 1:
// its last; inside a slot, column m of the tile is 128 contiguous weight
// rows).
constexpr int kCountersPerProblem = 256;
constexpr int kMaxGemmGroupCounters = 8;
constexpr size_t kCounterBytes =
    static_cast<size_t>(kMaxGemmGroupCounters) * kCountersPerProblem * sizeof(uint32_t);
constexpr int kMaxGrid = 1024;
size_t gemm_workspace_bytes(const GemmKernelConfig& c, const GemmSchedule& s, int64_t M,
                            int64_t N, int64_t K);

// Shared memory bytes of a configuration (for eligibility checks).
size_t gemm_smem_bytes(const GemmKernelConfig& c);

// True if the kernel for `c` is compiled in.
bool gemm_config_available(const GemmKernelConfig& c);

// Independent problems launched together (one kernel; problem i runs on its
// own s[i].grid CTAs).  All problems use one configuration and one
// activation type; workspaces must not overlap.
constexpr int kMaxGemmGroup = 8;
static_assert(kMaxGemmGroup <= kMaxGemmGroupCounters, "a counter block per problem");
struct GemmGroup {
  int count = 0;
  GemmProblem p[kMaxGemmGroup];
  GemmSchedule s[kMaxGemmGroup];
};

cudaError_t launch_gemm_tc(const GemmKernelConfig& c, const GemmSchedule& s,
                           const GemmProblem& p, bool use_pdl, cudaStream_t stream);
cudaError_t launch_gemm_tc_group(const GemmKernelConfig& c, const GemmGroup& grp, bool use_pdl,
                                 cudaStream_t stream);
// Instantiations called by launch_gemm_tc_group: single-problem fp16
// (gemm_tc_f16.cu) and the multi-problem ones (gemm_tc_group*.cu).
cudaError_t launch_gemm_tc_f16(const GemmKernelConfig& c, const GemmGroup& grp, bool use_pdl,
                               cudaStream_t stream);
cudaError_t launch_gemm_tc_group_bf16(const GemmKernelConfig& c, const GemmGroup& grp,
                                      bool use_pdl, cudaStream_t stream);
cudaError_t launch_gemm_tc_group_f16(const GemmKernelConfig& c, const GemmGroup& grp,
                                     bool use_pdl, cudaStream_t stream);
// The SwiGLU epilogue (gemm_tc_swiglu.cu): one problem, INT4 weights, bf16
// activations.
cudaError_t launch_gemm_tc_swiglu(const GemmKernelConfig& c, const GemmGroup& grp, bool use_pdl,
                                  cudaStream_t stream);
// Grouped launches in which some problems take the SwiGLU epilogue
// (gemm_tc_group_swiglu.cu): INT4 weights, bf16 activations.
cudaError_t launch_gemm_tc_group_swiglu(const GemmKernelConfig& c, const GemmGroup& grp,
                                        bool use_pdl, cudaStream_t stream);
// INT8 weights (gemm_tc_w8.cu): one problem, bf16 activations.
cudaError_t launch_gemm_tc_w8(const GemmKernelConfig& c, const GemmGroup& grp, bool use_pdl,
                              cudaStream_t stream);
// FP4 weights (gemm_tc_mxfp4.cu, gemm_tc_nvfp4.cu): one problem, bf16
// activations.
cudaError_t launch_gemm_tc_mxfp4(const GemmKernelConfig& c, const GemmGroup& grp, bool use_pdl,
                                 cudaStream_t stream);
cudaError_t launch_gemm_tc_nvfp4(const GemmKernelConfig& c, const GemmGroup& grp, bool use_pdl,
                                 cudaStream_t stream);

// The CUDA-core streaming kernel for tiny M (gemv.cu): one problem, INT4
// weights, bf16 or fp16 activations; shared memory of a configuration (0:
// none).
cudaError_t launch_gemv(const GemmKernelConfig& c, const GemmGroup& grp, bool use_pdl,
                        cudaStream_t stream);
size_t gemv_smem_bytes(const GemmKernelConfig& c);

// Row-major packed codes [N, K/2] (16-byte aligned, K % 128 == 0) to the
// tiled storage (layout.cu); one launch.
cudaError_t launch_repack_rowmajor(const void* rowmajor, int64_t N, int64_t K, void* tiled,
                                   int num_sms, cudaStream_t stream);

// Self test of the quantizer's corrected quotient against the IEEE division
// (quantize.cu): mode 0 INT4 scales, 1 INT8 scales, 2 NVFP4 steps; zeroes
// counts[0..3] on `stream`, then adds the pairs checked, the codes that
// differ, the quotients that differ in the normal range and anywhere.
cudaError_t launch_quotient_selftest(int mode, unsigned long long* counts, cudaStream_t stream);

// The row-block warp-MMA kernel (gemv_rb.cu): INT4 weights, bf16 or fp16
// activations, M <= act_tile (1, 2, 4, 8, 16), one problem or a group.  Persistent (cluster <= 1):
// any grid, teams of `team` warps walk row blocks round-robin.  Cluster
// split (cluster > 1): grid = row blocks x cluster, team = 8.  Rows per block
// and resident CTAs per SM for an act_tile.
cudaError_t launch_gemv_rb(const GemmKernelConfig& c, const GemmGroup& grp, bool use_pdl,
                           cudaStream_t stream);
int gemv_rb_rows(int act_tile);
constexpr int kRbWarpsPerCta = 8;
int gemv_rb_ctas_per_sm(int act_tile);
size_t gemv_rb_smem_bytes(int act_tile);   // dynamic shared memory; 0: no such kernel

// Failure-detection self test: one thread waits on an mbarrier nobody
// arrives at, with a bounded wait; records a timeout in *error_word.
cudaError_t launch_wait_timeout_selftest(uint32_t* error_word, uint64_t timeout_ns,
                                         cudaStream_t stream);

// Encoders for the TMA descriptors (driver entry point, resolved once).
CUresult encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                        uint64_t inner, uint64_t outer, uint64_t outer_stride_bytes,
                        uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle);
CUresult encode_tmap_3d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                        uint64_t d0, uint64_t d1, uint64_t d2, uint64_t stride1_bytes,
                        uint64_t stride2_bytes, uint32_t box0, uint32_t box1, uint32_t box2,
                        CUtensorMapSwizzle swizzle);

}  // namespace w4a16
