// W4A16 GEMV for tiny M (M <= 8): a CUDA-core streaming kernel (sm_103a),
// bf16 or fp16 activations.
//
// "Kernel dispatch and Humming quantization in PhyAI", section "Humming makes
// the separation useful": INT4 round-to-nearest weights, group 128 along K,
// BF16 activations, and the packed layout runs only through the kernels that
// understand it.  At M <= 8 the GEMM does 2 M flops per 0.52 bytes of codes
// and scales, far below the tensor cores' ridge: it is bound by streaming the
// weight from HBM.  This variant therefore feeds no tensor cores; it streams
// the same tiled codes and scales as the tcgen05 kernel and reduces on the
// CUDA cores, with none of the tcgen05 pipeline's fixed costs (TMEM, MMA
// issue, operand stores).
//
// Workers.  Every warp is an independent worker of the stream-K schedule the
// tcgen05 kernel uses (units = (128-row tile, group of 128 k); contiguous
// balanced unit ranges; a tile split between workers is finished by the last
// contributor to arrive, which sums the fp32 partials in k order, adds the
// bias and rounds once).  A warp owns R shared-memory stages: one TMA copy
// brings a unit's 8 KiB of codes (one contiguous block of the tiled storage,
// rows of 64 bytes with the 64-byte swizzle: chunk c of row r lands at
// c ^ ((r >> 1) & 3), so that lanes reading the same chunk of consecutive
// rows hit different banks), one 1-D bulk copy its fp16 scales and one each
// activation row's 256-byte slice; when the warp is done with a stage it
// issues the copy of its unit R ahead into it.  Warps never wait for one
// another.
//
// Per unit, lane l:
//   1. converts activations k = 4 l .. 4 l + 3 of each row to fp32 into the
//      stage and reduces the group's even-k and odd-k activation sums over
//      the warp;
//   2. for each 32-k quarter, turns the 32 codes of weight rows l, l + 32,
//      l + 64, l + 96 into floats and runs fp32 FMAs against the quarter's
//      activations, which every lane reads from the same address (broadcast)
//      and keeps in registers for its four rows; four independent chains.
// Codes to floats: a code c (a two's-complement nibble) placed under a fixed
// exponent by one AND-XOR reads 128 + n at bits 16..19 of the float with
// exponent 2^7 and 2048 + n at bits 12..15 of the float with exponent 2^11,
// n = c ^ 8 = q + 8.  Shifting each code word four ways puts every even
// nibble at bit 16 and every odd one at bit 12, so x = 136 + q (even k) or
// 2056 + q (odd k), twelve operations per eight codes, and
//   sum_k q_k a_k = sum_k x_k a_k - 136 sum_even a - 2056 sum_odd a.
// |sum x a| is at most about 2056 times the odd-k activation sum, so fp32
// rounding leaves a relative error of order 1e-4 of a group's partial: far
// inside the GEMM tolerance.  The partial times the group's fp32 scale is
// added to the row's total.
#include "gemm_tc.cuh"

namespace w4a16 {
namespace {

constexpr int kGvStagesPerWarp = 2;

template <int MT>
struct GvCfg {
  static constexpr int kWarps = gemv_warps_per_cta(MT);
  static constexpr int kR = kGvStagesPerWarp;
  static constexpr int kCodeOff = 0;                       // 128 rows x 64 B
  static constexpr int kScaleOff = kCodeOff + 8192;        // 128 fp16
  static constexpr int kActOff = kScaleOff + 256;          // [MT][128] bf16 / fp16
  static constexpr int kActF32Off = kActOff + MT * 256;    // [MT][128] fp32
  static constexpr int kActF32Row = 512;
  static constexpr int kStageRaw = kActF32Off + MT * kActF32Row;
  static constexpr int kStage = (kStageRaw + 1023) / 1024 * 1024;   // swizzled TMA destination
  static constexpr int kBarOff = kWarps * kR * kStage;     // full barriers [warp][stage]
  static constexpr int kFlagOff = kBarOff + kWarps * kR * 8;   // the CTA's abort flag
  static constexpr size_t kSmem = static_cast<size_t>(kFlagOff) + 16 + 1024;   // + alignment
  static_assert(kActOff % 16 == 0 && kActF32Off % 16 == 0, "alignment");
};

struct GvArgs {
  CUtensorMap tm_w;        // tiled codes as rows of 64 B, 64-byte swizzle, box 64 x 128
  Args a;
  const uint16_t* A;       // [M, K] activations
  int workers;             // stream-K workers (warps) of the schedule
};

// Codes of one word (code j in nibble j) as floats 136 + q (even j) or
// 2056 + q (odd j).
__device__ __forceinline__ void nibbles_to_magic(uint32_t w, float* x) {
  constexpr uint32_t kM16 = 0x000F0000u, kE16 = 0x43080000u;   // 128 + (c ^ 8)
  constexpr uint32_t kM12 = 0x0000F000u, kE12 = 0x45008000u;   // 2048 + (c ^ 8)
  const uint32_t l8 = w << 8, l16 = w << 16, r8 = w >> 8, r16 = w >> 16;
  x[0] = __uint_as_float(ptx::and_xor(l16, kM16, kE16));
  x[1] = __uint_as_float(ptx::and_xor(l8, kM12, kE12));
  x[2] = __uint_as_float(ptx::and_xor(l8, kM16, kE16));
  x[3] = __uint_as_float(ptx::and_xor(w, kM12, kE12));
  x[4] = __uint_as_float(ptx::and_xor(w, kM16, kE16));
  x[5] = __uint_as_float(ptx::and_xor(r8, kM12, kE12));
  x[6] = __uint_as_float(ptx::and_xor(r8, kM16, kE16));
  x[7] = __uint_as_float(ptx::and_xor(r16, kM12, kE12));
}

__device__ __forceinline__ uint32_t lds_u16(uint32_t saddr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(saddr));
  return v;
}

__device__ __forceinline__ void sts128(uint32_t saddr, float a, float b, float c, float d) {
  asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(saddr), "f"(a), "f"(b), "f"(c),
               "f"(d)
               : "memory");
}

template <int MT, bool F16>
__global__ void __launch_bounds__(32 * gemv_warps_per_cta(MT),
                                  gemv_workers_per_sm(MT) / gemv_warps_per_cta(MT))
    w4a16_gemv_kernel(const __grid_constant__ GvArgs g) {
  using C = GvCfg<MT>;
  constexpr int R = C::kR;
  const Args& a = g.a;
  extern __shared__ __align__(1024) uint8_t gv_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(gv_smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kBarOff) + warp * R;
  int& abort_flag = *reinterpret_cast<int*>(smem + C::kFlagOff);
  if (threadIdx.x == 0) abort_flag = 0;
  if (lane == 0) {
    for (int s = 0; s < R; ++s) ptx::mbar_init(&full[s], 1);
    ptx::fence_mbar_init();
    if (warp == 0) ptx::prefetch_tmap(&g.tm_w);
  }
  __syncthreads();
  const WaitCtx wc{a.err, a.timeout_ns, &abort_flag};
  const int worker = static_cast<int>(blockIdx.x) * C::kWarps + warp;
  Sched sched;
  sched.init(a, worker, g.workers);
  const int total = worker < g.workers ? sched.total : 0;
  const int M = a.M;
  const uint32_t stage0 = ptx::smem_u32(smem + warp * R * C::kStage);
  // inputs may be the previous kernel's outputs: nothing is read before this
  ptx::grid_dependency_wait();
  ptx::grid_launch_dependents();

  UnitIter issue_it;
  issue_it.init(sched);
  // copies of this warp's n-th unit into its stage n % R (lane 0)
  auto issue = [&](int n) {
    const Unit u = issue_it.next();
    const int st = n % R;
    uint8_t* stg = smem + (warp * R + st) * C::kStage;
    const int tn = u.tile % a.n_tiles;
    const int gi = u.kb;
    const uint32_t sbytes = static_cast<uint32_t>(min(kTileW, a.N - tn * kTileW)) * 2u;
    ptx::mbar_arrive_expect_tx(&full[st], 8192u + sbytes + static_cast<uint32_t>(M) * 256u);
    ptx::tma_load_2d(stg + C::kCodeOff, &g.tm_w, &full[st], 0,
                     (tn * a.KB + gi) * kTileW);
    ptx::bulk_g2s(stg + C::kScaleOff, a.scales + static_cast<int64_t>(gi) * a.N + tn * kTileW,
                  sbytes, &full[st]);
    for (int m = 0; m < M; ++m)
      ptx::bulk_g2s(stg + C::kActOff + m * 256, g.A + static_cast<int64_t>(m) * a.K + gi * kUnitK,
                    256u, &full[st]);
  };
  if (lane == 0)
    for (int n = 0; n < R && n < total; ++n) issue(n);

  UnitIter it;
  it.init(sched);
  float tot[4][MT];
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int m = 0; m < MT; ++m) tot[j][m] = 0.0f;
  const int swz = (lane >> 1) & 3;   // the swizzle of rows lane + 32 j
  int n = 0;
  for (; n < total; ++n) {
    const Unit u = it.next();
    if (u.seg_first) {
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int m = 0; m < MT; ++m) tot[j][m] = 0.0f;
    }
    const int st = n % R;
    if (!wait_warp(&full[st], (n / R) & 1, wc)) break;
    const uint32_t stg = stage0 + st * C::kStage;

    // 1. activations to fp32, and the group's even- and odd-k sums
    float corr[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      float f0 = 0.0f, f1 = 0.0f, f2 = 0.0f, f3 = 0.0f;
      if (m < M) {
        const uint2 v = ptx::lds64(stg + C::kActOff + m * 256 + 8 * lane);
        f0 = act_to_float<F16>(static_cast<uint16_t>(v.x));
        f1 = act_to_float<F16>(static_cast<uint16_t>(v.x >> 16));
        f2 = act_to_float<F16>(static_cast<uint16_t>(v.y));
        f3 = act_to_float<F16>(static_cast<uint16_t>(v.y >> 16));
      }
      sts128(stg + C::kActF32Off + m * C::kActF32Row + 16 * lane, f0, f1, f2, f3);
      float se = f0 + f2, so = f1 + f3;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        se += __shfl_xor_sync(0xFFFFFFFFu, se, d);
        so += __shfl_xor_sync(0xFFFFFFFFu, so, d);
      }
      corr[m] = fmaf(-136.0f, se, -2056.0f * so);
    }
    __syncwarp();

    // 2. the four rows' dot products over the group
    float s[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      s[j] = __half2float(__ushort_as_half(static_cast<unsigned short>(
          lds_u16(stg + C::kScaleOff + 2 * (lane + 32 * j)))));
    float part[4][MT];
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int m = 0; m < MT; ++m) part[j][m] = 0.0f;
    // one 32-k quarter at a time (rolled for more than two activation rows:
    // the quarter's operands of the four rows stay in registers)
    constexpr int kUnrollQ = MT <= 2 ? 4 : 1;
#pragma unroll kUnrollQ
    for (int c = 0; c < 4; ++c) {
      float x[4][32];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 cw = ptx::lds128(stg + C::kCodeOff + (lane + 32 * j) * 64 + 16 * (c ^ swz));
        nibbles_to_magic(cw.x, x[j]);
        nibbles_to_magic(cw.y, x[j] + 8);
        nibbles_to_magic(cw.z, x[j] + 16);
        nibbles_to_magic(cw.w, x[j] + 24);
      }
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        const uint32_t ab = stg + C::kActF32Off + m * C::kActF32Row + 128 * c;
        float p[4][2];
#pragma unroll
        for (int j = 0; j < 4; ++j) p[j][0] = p[j][1] = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint4 av = ptx::lds128(ab + 16 * i);   // the same address in every lane
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            p[j][i & 1] = fmaf(x[j][4 * i + 0], __uint_as_float(av.x), p[j][i & 1]);
            p[j][i & 1] = fmaf(x[j][4 * i + 1], __uint_as_float(av.y), p[j][i & 1]);
            p[j][i & 1] = fmaf(x[j][4 * i + 2], __uint_as_float(av.z), p[j][i & 1]);
            p[j][i & 1] = fmaf(x[j][4 * i + 3], __uint_as_float(av.w), p[j][i & 1]);
          }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) part[j][m] += p[j][0] + p[j][1];
      }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int m = 0; m < MT; ++m) tot[j][m] = fmaf(s[j], part[j][m] + corr[m], tot[j][m]);

    // the stage is free: its next copy (generic reads before async writes)
    __syncwarp();
    if (lane == 0 && n + R < total) {
      ptx::fence_proxy_async_smem();
      issue(n + R);
    }
    if (!u.seg_last) continue;

    const int tn = u.tile % a.n_tiles;
    if (u.whole) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int nrow = tn * kTileW + lane + 32 * j;
        if (nrow >= a.N) continue;
        const float bias_f = a.bias != nullptr ? act_to_float<F16>(a.bias[nrow]) : 0.0f;
#pragma unroll
        for (int m = 0; m < MT; ++m)
          if (m < M) a.Y[static_cast<int64_t>(m) * a.N + nrow] = act_from_float<F16>(tot[j][m] + bias_f);
      }
      continue;
    }
    // split tile: this worker's partial, then the arrival count; the last
    // contributor sums every partial in k order
    constexpr int64_t kSlot = static_cast<int64_t>(MT) * kTileW;
    float* slot = a.ws + (static_cast<int64_t>(worker) * 2 + u.slot) * kSlot;
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int m = 0; m < MT; ++m) slot[m * kTileW + lane + 32 * j] = tot[j][m];
    __threadfence();
    __syncwarp();
    const SplitInfo si = split_info(a, u.sk_tile, g.workers);
    int last = 0;
    if (lane == 0) {
      uint32_t* cnt = a.counters + u.sk_tile;
      const uint32_t old = ptx::atom_add_acq_rel_gpu(cnt, 1u);
      last = old == static_cast<uint32_t>(si.c_hi - si.c_lo) ? 1 : 0;
      if (last) atomicExch(cnt, 0u);
    }
    last = __shfl_sync(0xFFFFFFFFu, last, 0);
    if (!last) continue;
    __threadfence();
    // lane l sums rows 4 l .. 4 l + 3 over the contributors in k order; the
    // loads of a batch of contributors are issued together (a tile may have
    // tens of contributors)
    constexpr int kBatch = MT <= 2 ? 8 : MT <= 4 ? 2 : 1;
    float4 acc[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m)
      acc[m] = __ldcg(reinterpret_cast<const float4*>(
          a.ws + (static_cast<int64_t>(si.c_lo) * 2 + si.slot_lo) * kSlot + m * kTileW) + lane);
    for (int c0 = si.c_lo + 1; c0 <= si.c_hi; c0 += kBatch) {
      float4 v[kBatch][MT];
#pragma unroll
      for (int b = 0; b < kBatch; ++b)
#pragma unroll
        for (int m = 0; m < MT; ++m)
          if (c0 + b <= si.c_hi)
            v[b][m] = __ldcg(reinterpret_cast<const float4*>(
                a.ws + static_cast<int64_t>(c0 + b) * 2 * kSlot + m * kTileW) + lane);
#pragma unroll
      for (int b = 0; b < kBatch; ++b)
#pragma unroll
        for (int m = 0; m < MT; ++m)
          if (c0 + b <= si.c_hi) {
            acc[m].x += v[b][m].x;
            acc[m].y += v[b][m].y;
            acc[m].z += v[b][m].z;
            acc[m].w += v[b][m].w;
          }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int nrow = tn * kTileW + 4 * lane + e;
      if (nrow >= a.N) continue;
      const float bias_f = a.bias != nullptr ? act_to_float<F16>(a.bias[nrow]) : 0.0f;
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        if (m >= M) continue;
        const float vv = e == 0 ? acc[m].x : e == 1 ? acc[m].y : e == 2 ? acc[m].z : acc[m].w;
        a.Y[static_cast<int64_t>(m) * a.N + nrow] = act_from_float<F16>(vv + bias_f);
      }
    }
  }
  if (n < total && lane == 0) {
    // gave up: this warp's copies in flight land before the CTA exits
    const int last_issued = min(total, n + R);
    for (int j = n; j < last_issued; ++j) {
      const uint64_t t0 = ptx::globaltimer_ns();
      while (!ptx::mbar_try_wait(&full[j % R], (j / R) & 1))
        if (ptx::globaltimer_ns() - t0 > a.timeout_ns) break;
    }
  }
}

template <int MT, bool F16>
cudaError_t launch_gemv_typed(const GemmProblem& p, const GemmSchedule& s, bool use_pdl,
                              cudaStream_t stream) {
  using C = GvCfg<MT>;
  auto kernel = w4a16_gemv_kernel<MT, F16>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static bool attr_set[64] = {};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(C::kSmem));
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  if (p.M > MT || p.K % kUnitK != 0 || s.grid < 1) return cudaErrorInvalidValue;
  if (p.swiglu) return cudaErrorInvalidValue;   // the fused epilogue is the tcgen05 path's
  GvArgs g{};
  Args& a = g.a;
  a.M = static_cast<int>(p.M);
  a.N = static_cast<int>(p.N);
  a.K = static_cast<int>(p.K);
  a.KB = static_cast<int>(p.K / kUnitK);
  a.n_tiles = static_cast<int>((p.N + kTileW - 1) / kTileW);
  a.dp_tiles = s.dp_tiles;
  a.sk_units = static_cast<int>(s.sk_units);
  a.act_3d = 0;
  a.scales = static_cast<const __half*>(p.scales);
  a.out_scale = nullptr;
  a.bias = static_cast<const uint16_t*>(p.bias);
  a.Y = static_cast<uint16_t*>(p.Y);
  a.counters = p.counters != nullptr ? p.counters : static_cast<uint32_t*>(p.workspace);
  a.ws = p.partials != nullptr
             ? p.partials
             : reinterpret_cast<float*>(static_cast<uint8_t*>(p.workspace) + kCounterBytes);
  a.err = p.error_word;
  a.timeout_ns = p.timeout_ns;
  const uint64_t w_rows = static_cast<uint64_t>(a.n_tiles) * a.KB * kTileW;
  if (encode_tmap_2d(&g.tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.packed, 64, w_rows, 64, 64, kTileW,
                     CU_TENSOR_MAP_SWIZZLE_64B) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  g.A = static_cast<const uint16_t*>(p.A);
  g.workers = s.grid;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((s.grid + C::kWarps - 1) / C::kWarps));
  cfg.blockDim = dim3(32 * C::kWarps);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = use_pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, g);
}

}  // namespace

size_t gemv_smem_bytes(const GemmKernelConfig& c) {
  if (!c.simt || c.weight_format != kFmtInt4 || c.unit_groups != 1 || c.stages != kGvStagesPerWarp)
    return 0;
  switch (c.act_tile) {
    case 1: return GvCfg<1>::kSmem;
    case 2: return GvCfg<2>::kSmem;
    case 4: return GvCfg<4>::kSmem;
    case 8: return GvCfg<8>::kSmem;
    default: return 0;
  }
}

cudaError_t launch_gemv(const GemmKernelConfig& c, const GemmGroup& grp, bool use_pdl,
                        cudaStream_t stream) {
  if (grp.count != 1 || gemv_smem_bytes(c) == 0) return cudaErrorInvalidValue;
  const GemmProblem& p = grp.p[0];
  const GemmSchedule& s = grp.s[0];
  const bool f16 = p.act_f16;
  switch (c.act_tile) {
    case 1: return f16 ? launch_gemv_typed<1, true>(p, s, use_pdl, stream)
                       : launch_gemv_typed<1, false>(p, s, use_pdl, stream);
    case 2: return f16 ? launch_gemv_typed<2, true>(p, s, use_pdl, stream)
                       : launch_gemv_typed<2, false>(p, s, use_pdl, stream);
    case 4: return f16 ? launch_gemv_typed<4, true>(p, s, use_pdl, stream)
                       : launch_gemv_typed<4, false>(p, s, use_pdl, stream);
    case 8: return f16 ? launch_gemv_typed<8, true>(p, s, use_pdl, stream)
                       : launch_gemv_typed<8, false>(p, s, use_pdl, stream);
    default: return cudaErrorInvalidConfiguration;
  }
}

}  // namespace w4a16
