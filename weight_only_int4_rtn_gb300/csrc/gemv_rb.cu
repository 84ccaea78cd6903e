// W4A16 GEMV for M <= 4: a row-block CUDA-core kernel (sm_103a), bf16 or fp16
// activations.
//
// "Kernel dispatch and Humming quantization in PhyAI", section "Humming makes
// the separation useful": INT4 round-to-nearest weights, group 128 along K,
// BF16 (or FP16) activations; the packed layout runs only through the kernels
// that understand it.  At M <= 4 the GEMM does at most 8 flops per 0.52
// bytes of codes and scales: it is bound by streaming the weight from HBM,
// and the tensor-core path's fixed costs per 128 x 128 unit (the converted
// operand's TMEM round trip, MMA issue, barrier hand-offs between roles)
// are what limits it.  This kernel has no pipeline roles at all: every
// thread loads its own codes with 16-byte loads straight from the tiled
// storage (no TMA, no shared-memory staging, no mbarrier), converts them in
// registers and runs fp32 FMAs.
//
// Work split.  A CTA owns a block of RB = 16 consecutive weight rows (inside
// one 128-row storage tile) and a K range; its warps split that K range into
// equal runs of groups.  A lane owns a chunk of CH = 16 codes (an 8-byte
// piece of a 64-byte tile row) of RPL = 4 rows, r = lane / 8 + 4 j, so a
// warp's load instruction covers 4 consecutive rows, i.e. one contiguous
// 256-byte run of the tile (for M <= 1 two CTAs of 8 warps fit an SM at
// 128 registers; 32-code chunks spill at that size).  The activations of the lane's chunk (CH
// values per activation row) are loaded once per group and serve its RPL
// rows.  When there are too few row blocks to occupy the GPU, the K range is
// also split over the S CTAs of a thread-block cluster and summed through
// distributed shared memory.
//
// Codes to floats.  One shift of a code word puts two neighbouring nibbles
// at bits 12..15 and 16..19; one AND-XOR each places them under the exponent
// of 2048 (bits 12..15) or 128 (bits 16..19) with the nibble's sign bit
// flipped (n ^ 8 = q + 8), so a code of even k reads 2056 + q and one of odd
// k reads 136 + q, exactly: twelve operations per eight codes.  Products
// with a bf16 or fp16 activation are exact in fp32 (at most 12 + 11
// significant bits), and per chunk
//   sum_k q_k a_k = sum_k x_k a_k - 2056 sum_even a - 136 sum_odd a,
// the two activation sums formed once per group and shared by the lane's
// rows.  The group's partial times the fp32 scale goes to the row's total.
//
// Reduction.  Lanes of one row sum their totals by shuffles (fixed order);
// each warp writes its rows' totals to shared memory; after a CTA barrier
// the totals of the warps are summed in warp order (k order), then (with a
// cluster) the CTAs' sums in rank order; the bias is added in fp32 and Y
// rounded once.  The result does not depend on timing.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"

namespace w4a16 {
namespace {

constexpr int kRbWarps = 8;   // warps per CTA (a K split of the block)

struct RbArgs {
  const uint16_t* A;       // [M, K] activation type
  const uint8_t* packed;   // tiled codes
  const __half* scales;    // [K/128, N]
  const uint16_t* bias;    // [N] or null
  uint16_t* Y;             // [M, N]
  int M, N, K, KB;         // KB: groups along K
  int cluster;             // CTAs of a cluster splitting K (1: none)
};

template <bool F16>
__device__ __forceinline__ float rb_act(uint16_t b) {
  if constexpr (F16) {
    return __half2float(__ushort_as_half(b));
  } else {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
  }
}

// Activations of one chunk: CH values (as CH / 2 words of two 16-bit values)
// to floats, and the chunk's even-k and odd-k sums.
template <int CH, bool F16>
__device__ __forceinline__ void rb_acts(const uint32_t (&w)[CH / 2], float (&a)[CH], float& se,
                                        float& so) {
  se = 0.0f;
  so = 0.0f;
#pragma unroll
  for (int i = 0; i < CH / 2; ++i) {
    if constexpr (F16) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
      a[2 * i] = f.x;
      a[2 * i + 1] = f.y;
    } else {
      a[2 * i] = __uint_as_float(w[i] << 16);
      a[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
    se += a[2 * i];
    so += a[2 * i + 1];
  }
}

// sum_k x_k a_k over the 8 codes of one word (x: 2056 + q for even k, 136 +
// q for odd k).
__device__ __forceinline__ float rb_dot8(uint32_t w, const float* a, float acc) {
  constexpr uint32_t kLo = 0x45008000u;   // 2048 with bit 15 flipped: 2056 + q at bits 12..15
  constexpr uint32_t kHi = 0x43080000u;   // 128 with bit 19 flipped: 136 + q at bits 16..19
  const uint32_t s0 = w << 12, s1 = w << 4, s2 = w >> 4, s3 = w >> 12;
  acc = fmaf(__uint_as_float(ptx::and_xor(s0, 0x0000F000u, kLo)), a[0], acc);
  acc = fmaf(__uint_as_float(ptx::and_xor(s0, 0x000F0000u, kHi)), a[1], acc);
  acc = fmaf(__uint_as_float(ptx::and_xor(s1, 0x0000F000u, kLo)), a[2], acc);
  acc = fmaf(__uint_as_float(ptx::and_xor(s1, 0x000F0000u, kHi)), a[3], acc);
  acc = fmaf(__uint_as_float(ptx::and_xor(s2, 0x0000F000u, kLo)), a[4], acc);
  acc = fmaf(__uint_as_float(ptx::and_xor(s2, 0x000F0000u, kHi)), a[5], acc);
  acc = fmaf(__uint_as_float(ptx::and_xor(s3, 0x0000F000u, kLo)), a[6], acc);
  acc = fmaf(__uint_as_float(ptx::and_xor(s3, 0x000F0000u, kHi)), a[7], acc);
  return acc;
}

// MT: activation rows (M <= MT); CH: codes per lane chunk (32 or 16); RPL:
// rows per lane.
template <int MT, int CH, int RPL>
struct RbCfg {
  static constexpr int kLPR = kGroup / CH;           // lanes per row
  static constexpr int kRowsPerPass = 32 / kLPR;     // rows one warp instruction covers
  static constexpr int kRB = kRowsPerPass * RPL;     // rows per CTA
  static constexpr int kWords = CH / 8;              // code words per lane-chunk
  static_assert(kGroup % kRB == 0, "a row block sits inside one 128-row tile");
};

// CTAs per SM the registers allow without spills: two for M <= 1, one above
template <int MT>
constexpr int rb_min_blocks() { return MT <= 1 ? 2 : 1; }

template <int MT, int CH, int RPL, bool F16>
__global__ void __launch_bounds__(kRbWarps * 32, rb_min_blocks<MT>())
    gemv_rb_kernel(const __grid_constant__ RbArgs g) {
  using C = RbCfg<MT, CH, RPL>;
  constexpr int W = C::kWords;
  __shared__ float red[kRbWarps][C::kRB][MT];   // per warp: its rows' totals
  __shared__ float csum[C::kRB][MT];            // the CTA's totals (read by its cluster)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = g.cluster;
  const int blk = static_cast<int>(blockIdx.x) / S;
  const int rank = static_cast<int>(blockIdx.x) - blk * S;
  const int r0 = blk * C::kRB;                    // first row of the block
  const int tn = r0 / kTileW;
  const int rin0 = r0 - tn * kTileW;              // its row inside the tile
  const int c = lane % C::kLPR;                   // the lane's chunk
  const int rl = lane / C::kLPR;                  // the lane's first row in the block

  // this warp's groups: the CTA's rank-th share of K, then the warp's share
  const int cg0 = (rank * g.KB) / S, cg1 = ((rank + 1) * g.KB) / S;
  const int g0 = cg0 + (warp * (cg1 - cg0)) / kRbWarps;
  const int g1 = cg0 + ((warp + 1) * (cg1 - cg0)) / kRbWarps;

  // the weights are constant for the launch; the activations may be the
  // previous kernel's output
  ptx::grid_dependency_wait();
  ptx::grid_launch_dependents();

  float acc[RPL][MT];
#pragma unroll
  for (int j = 0; j < RPL; ++j)
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[j][m] = 0.0f;

  // code words of row j of group gg for this lane
  auto code_ptr = [&](int gg, int j) -> const uint8_t* {
    return g.packed + ((static_cast<int64_t>(tn) * g.KB + gg) * kTileW + rin0 + rl + C::kRowsPerPass * j) * 64 +
           c * (CH / 2);
  };
  auto load_codes = [&](int gg, uint32_t (&cw)[RPL][W]) {
#pragma unroll
    for (int j = 0; j < RPL; ++j) {
      if constexpr (W == 4) {
        const uint4 v = __ldcs(reinterpret_cast<const uint4*>(code_ptr(gg, j)));
        cw[j][0] = v.x;
        cw[j][1] = v.y;
        cw[j][2] = v.z;
        cw[j][3] = v.w;
      } else {
        const uint2 v = __ldcs(reinterpret_cast<const uint2*>(code_ptr(gg, j)));
        cw[j][0] = v.x;
        cw[j][1] = v.y;
      }
    }
  };
  auto load_acts = [&](int gg, uint32_t (&aw)[MT][CH / 2]) {
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      if (m < g.M) {
        const uint4* p = reinterpret_cast<const uint4*>(g.A + static_cast<int64_t>(m) * g.K +
                                                        gg * kGroup + c * CH);
#pragma unroll
        for (int q = 0; q < CH / 8; ++q) {
          const uint4 v = __ldg(p + q);
          aw[m][4 * q] = v.x;
          aw[m][4 * q + 1] = v.y;
          aw[m][4 * q + 2] = v.z;
          aw[m][4 * q + 3] = v.w;
        }
      } else {
#pragma unroll
        for (int i = 0; i < CH / 2; ++i) aw[m][i] = 0u;
      }
    }
  };
  auto load_scales = [&](int gg, float (&sc)[RPL]) {
#pragma unroll
    for (int j = 0; j < RPL; ++j) {
      const int n = r0 + rl + C::kRowsPerPass * j;
      sc[j] = n < g.N ? __half2float(g.scales[static_cast<int64_t>(gg) * g.N + n]) : 0.0f;
    }
  };

  // two groups in flight: the next group's codes, activations and scales
  // are requested before the current group's arithmetic (the loop runs two
  // groups per trip so that both buffers have fixed registers)
  auto compute = [&](const uint32_t (&cw)[RPL][W], const uint32_t (&aw)[MT][CH / 2],
                     const float (&sc)[RPL]) {
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      float a[CH], se, so;
      rb_acts<CH, F16>(aw[m], a, se, so);
      const float corr = fmaf(2056.0f, se, 136.0f * so);
#pragma unroll
      for (int j = 0; j < RPL; ++j) {
        float p = 0.0f;
#pragma unroll
        for (int wi = 0; wi < W; ++wi) p = rb_dot8(cw[j][wi], a + 8 * wi, p);
        acc[j][m] = fmaf(sc[j], p - corr, acc[j][m]);
      }
    }
  };
  uint32_t cw0[RPL][W], cw1[RPL][W];
  uint32_t aw0[MT][CH / 2], aw1[MT][CH / 2];
  float sc0[RPL], sc1[RPL];
  if (g0 < g1) {
    load_codes(g0, cw0);
    load_acts(g0, aw0);
    load_scales(g0, sc0);
  }
#pragma unroll 1
  for (int gg = g0; gg < g1; gg += 2) {
    const bool second = gg + 1 < g1;
    if (second) {
      load_codes(gg + 1, cw1);
      load_acts(gg + 1, aw1);
      load_scales(gg + 1, sc1);
    }
    compute(cw0, aw0, sc0);
    if (second) {
      if (gg + 2 < g1) {
        load_codes(gg + 2, cw0);
        load_acts(gg + 2, aw0);
        load_scales(gg + 2, sc0);
      }
      compute(cw1, aw1, sc1);
    }
  }

  // lanes of a row: chunks summed in a fixed order (butterfly over the
  // lane's low bits)
#pragma unroll
  for (int j = 0; j < RPL; ++j)
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int o = 1; o < C::kLPR; o <<= 1) acc[j][m] += __shfl_xor_sync(0xFFFFFFFFu, acc[j][m], o);
  if (c == 0) {
#pragma unroll
    for (int j = 0; j < RPL; ++j)
#pragma unroll
      for (int m = 0; m < MT; ++m) red[warp][rl + C::kRowsPerPass * j][m] = acc[j][m];
  }
  __syncthreads();
  // warps in k order
  for (int e = threadIdx.x; e < C::kRB * MT; e += blockDim.x) {
    const int row = e / MT, m = e - row * MT;
    float t = 0.0f;
#pragma unroll
    for (int w = 0; w < kRbWarps; ++w) t += red[w][row][m];
    csum[row][m] = t;
  }
  if (S > 1) {
    // CTAs of the cluster in rank (k) order; rank q stores rows q, q + S, ...
    ptx::cluster_sync();
    const uint32_t base = ptx::smem_u32(&csum[0][0]);
    for (int e = threadIdx.x; e < C::kRB * MT; e += blockDim.x) {
      const int row = e / MT, m = e - row * MT;
      if (row % S != rank) continue;
      const int n = r0 + row;
      if (n >= g.N || m >= g.M) continue;
      float t = 0.0f;
      for (int q = 0; q < S; ++q) t += ptx::ld_dsmem_f32(base + 4u * static_cast<uint32_t>(e), q);
      if (g.bias != nullptr) t += rb_act<F16>(g.bias[n]);
      g.Y[static_cast<int64_t>(m) * g.N + n] =
          F16 ? __half_as_ushort(__float2half_rn(t)) : __bfloat16_as_ushort(__float2bfloat16_rn(t));
    }
    ptx::cluster_sync();   // every CTA's sums stay alive until read
  } else {
    __syncthreads();
    for (int e = threadIdx.x; e < C::kRB * MT; e += blockDim.x) {
      const int row = e / MT, m = e - row * MT;
      const int n = r0 + row;
      if (n >= g.N || m >= g.M) continue;
      float t = csum[row][m];
      if (g.bias != nullptr) t += rb_act<F16>(g.bias[n]);
      g.Y[static_cast<int64_t>(m) * g.N + n] =
          F16 ? __half_as_ushort(__float2half_rn(t)) : __bfloat16_as_ushort(__float2bfloat16_rn(t));
    }
  }
}

template <int MT, int CH, int RPL, bool F16>
cudaError_t launch_rb(const GemmProblem& p, const GemmSchedule& s, bool use_pdl, cudaStream_t stream) {
  using C = RbCfg<MT, CH, RPL>;
  const int64_t blocks = (p.N + C::kRB - 1) / C::kRB;
  const int S = s.cluster > 1 ? s.cluster : 1;
  if (p.M > MT || blocks * S != s.grid || S > 8 || p.K / kGroup < S) return cudaErrorInvalidValue;
  RbArgs g{};
  g.A = static_cast<const uint16_t*>(p.A);
  g.packed = static_cast<const uint8_t*>(p.packed);
  g.scales = static_cast<const __half*>(p.scales);
  g.bias = static_cast<const uint16_t*>(p.bias);
  g.Y = static_cast<uint16_t*>(p.Y);
  g.M = static_cast<int>(p.M);
  g.N = static_cast<int>(p.N);
  g.K = static_cast<int>(p.K);
  g.KB = static_cast<int>(p.K / kGroup);
  g.cluster = S;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(s.grid));
  cfg.blockDim = dim3(kRbWarps * 32);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (use_pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (S > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = static_cast<unsigned>(S);
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, gemv_rb_kernel<MT, CH, RPL, F16>, g);
}

}  // namespace

int gemv_rb_rows(int act_tile) {
  (void)act_tile;
  return RbCfg<1, 16, 4>::kRB;
}

cudaError_t launch_gemv_rb(const GemmKernelConfig& c, const GemmGroup& grp, bool use_pdl,
                           cudaStream_t stream) {
  if (grp.count != 1) return cudaErrorInvalidValue;
  const GemmProblem& p = grp.p[0];
  const GemmSchedule& s = grp.s[0];
  if (p.swiglu) return cudaErrorInvalidValue;   // the fused epilogue is the tcgen05 path's
  const bool f16 = p.act_f16;
  switch (c.act_tile) {
    case 1: return f16 ? launch_rb<1, 16, 4, true>(p, s, use_pdl, stream)
                       : launch_rb<1, 16, 4, false>(p, s, use_pdl, stream);
    case 2: return f16 ? launch_rb<2, 16, 4, true>(p, s, use_pdl, stream)
                       : launch_rb<2, 16, 4, false>(p, s, use_pdl, stream);
    case 4: return f16 ? launch_rb<4, 16, 4, true>(p, s, use_pdl, stream)
                       : launch_rb<4, 16, 4, false>(p, s, use_pdl, stream);
    default: return cudaErrorInvalidConfiguration;
  }
}

}  // namespace w4a16
