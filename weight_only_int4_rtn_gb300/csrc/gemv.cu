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
// Work.  The units are (128-row tile, group of 128 k), scheduled exactly as
// the tcgen05 kernel does (whole tiles, then balanced stream-K ranges; a
// split tile's contributors write fp32 partials and the last to arrive sums
// them in k order, adds the bias and rounds once).  Per unit, one 1-D bulk
// copy brings the tile's 8 KiB of codes (one contiguous block of the tiled
// storage), one its fp16 scales and one each activation row's 256-byte slice
// into a ring of shared-memory stages.
//
// Staging warp.  Lane 0 issues the copies, up to (stages - 2) units ahead.
// The warp then converts each landed activation slice to fp32 in a layout
// whose four k-quarters sit 144 bytes apart (so that the compute threads'
// broadcast reads of different quarters hit different banks), and writes the
// sums of its even-k and odd-k values per quarter.
//
// Compute warps.  Thread t owns weight rows t/4 and t/4 + 64 and the k
// quarter t%4 (32 codes per row).  A code c (a two's-complement nibble) is
// turned into a float by one AND-XOR that places it under a fixed exponent:
// at bits 16..19 of the float with exponent 2^7 it reads 128 + n, at bits
// 12..15 of the float with exponent 2^11 it reads 2048 + n, with n = c ^ 8 =
// q + 8.  Shifting each code word four ways puts every even nibble at bit 16
// and every odd one at bit 12, so x = 136 + q (even k) or 2056 + q (odd k),
// twelve operations per eight codes, and
//   sum_k q_k a_k = sum_k x_k a_k - 136 sum_even a - 2056 sum_odd a,
// with the two sums from the staging warp.  The dot products run as fp32
// FMAs in four independent chains per row; a group's partial times its fp32
// scale is added to the row's total.  |sum x a| is at most about 2056 times
// the odd-k activation sum, so fp32 rounding leaves a relative error of order
// 1e-4 of a group's partial: far inside the GEMM tolerance.
#include "gemm_tc.cuh"

namespace w4a16 {
namespace {

constexpr int kGvComputeWarps = 8;
constexpr int kGvThreads = 32 * (kGvComputeWarps + 1);
constexpr int kGvStagingWarp = kGvComputeWarps;
constexpr int kGvMaxStages = 8;
constexpr int kGvChunk = 144;   // one k-quarter of an fp32 activation row: 32 floats + 16 B

struct GvShared {
  uint64_t full[kGvMaxStages];    // the unit's copies landed
  uint64_t ready[kGvMaxStages];   // its activations converted
  uint64_t empty[kGvMaxStages];   // the compute warps are done with the stage
  uint64_t sync;                  // barrier of the compute warps (split-tile fixup)
  int abort_flag;
  int fixup_last;
};

template <int MT>
struct GvCfg {
  static constexpr int kStages = MT <= 2 ? 8 : 6;
  static constexpr int kCodeOff = 0;                       // 128 rows x 64 B
  static constexpr int kScaleOff = kCodeOff + 8192;        // 128 fp16
  static constexpr int kActOff = kScaleOff + 256;          // [MT][128] bf16
  static constexpr int kActF32Off = kActOff + MT * 256;    // [MT][4 quarters][144 B]
  static constexpr int kActF32Row = 4 * kGvChunk;
  static constexpr int kSumOff = kActF32Off + MT * kActF32Row;   // [MT][4][even, odd]
  static constexpr int kStageRaw = kSumOff + MT * 32;
  static constexpr int kStage = (kStageRaw + 127) / 128 * 128;
  static constexpr size_t kSmem = static_cast<size_t>(kStages) * kStage + sizeof(GvShared) + 128;
  static_assert(kStages <= kGvMaxStages, "barrier arrays");
  static_assert(kActOff % 16 == 0 && kActF32Off % 16 == 0 && kSumOff % 16 == 0, "alignment");
};

struct GvArgs {
  Args a;
  const uint8_t* packed;   // tiled codes
  const uint16_t* A;       // [M, K] bf16
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

// Barrier of the compute warps on an mbarrier (bounded: a warp that gave up
// cannot leave the others blocked).
__device__ __forceinline__ bool gv_sync(GvShared* sh, uint32_t& n, const WaitCtx& wc) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) ptx::mbar_arrive(&sh->sync);
  const bool ok = wait_warp(&sh->sync, n & 1, wc);
  ++n;
  return ok;
}

template <int MT, bool F16>
__global__ void __launch_bounds__(kGvThreads, gemv_ctas_per_sm(MT))
    w4a16_gemv_kernel(const __grid_constant__ GvArgs g) {
  using C = GvCfg<MT>;
  constexpr int S = C::kStages;
  const Args& a = g.a;
  const int cta = static_cast<int>(blockIdx.x);
  const int ctas = static_cast<int>(gridDim.x);
  extern __shared__ __align__(128) uint8_t gv_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(gv_smem_raw) + 127) &
                                             ~static_cast<uintptr_t>(127));
  GvShared* sh = reinterpret_cast<GvShared*>(smem + S * C::kStage);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(&sh->full[s], 1);
      ptx::mbar_init(&sh->ready[s], 1);
      ptx::mbar_init(&sh->empty[s], kGvComputeWarps);
    }
    ptx::mbar_init(&sh->sync, kGvComputeWarps);
    sh->abort_flag = 0;
    sh->fixup_last = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  const WaitCtx wc{a.err, a.timeout_ns, &sh->abort_flag};
  Sched sched;
  sched.init(a, cta, ctas);
  const int total = sched.total;
  const int M = a.M;
  // inputs may be the previous kernel's outputs: nothing is read before this
  ptx::grid_dependency_wait();
  ptx::grid_launch_dependents();

  if (warp == kGvStagingWarp) {
    // ------------------------------------------------------------ staging
    UnitIter it;
    it.init(sched);
    int issued = 0;
    for (int i = 0; i < total; ++i) {
      if (lane == 0) {
        // copies up to S - 2 units ahead: the stage of unit i + S - 2 was
        // last used by unit i - 2, whose activations are already staged
        while (issued < total && issued <= i + S - 2) {
          const Unit u = it.next();
          const int st = issued % S;
          if (issued >= S && !wait_one(&sh->empty[st], ((issued / S) - 1) & 1, wc)) break;
          const int tn = u.tile % a.n_tiles;
          const int gi = u.kb;
          uint8_t* stg = smem + st * C::kStage;
          const uint32_t sbytes = static_cast<uint32_t>(min(kTileW, a.N - tn * kTileW)) * 2u;
          ptx::mbar_arrive_expect_tx(&sh->full[st], 8192u + sbytes + static_cast<uint32_t>(M) * 256u);
          ptx::bulk_g2s(stg + C::kCodeOff,
                        g.packed + (static_cast<int64_t>(tn) * a.KB + gi) * 8192, 8192u,
                        &sh->full[st]);
          ptx::bulk_g2s(stg + C::kScaleOff,
                        a.scales + static_cast<int64_t>(gi) * a.N + tn * kTileW, sbytes,
                        &sh->full[st]);
          for (int m = 0; m < M; ++m)
            ptx::bulk_g2s(stg + C::kActOff + m * 256,
                          g.A + static_cast<int64_t>(m) * a.K + gi * kUnitK, 256u, &sh->full[st]);
          ++issued;
        }
      }
      __syncwarp();
      const int st = i % S;
      if (!wait_warp(&sh->full[st], (i / S) & 1, wc)) break;
      uint8_t* stg = smem + st * C::kStage;
      // lane l: k = 4 l .. 4 l + 3 of each activation row (quarter l / 8)
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        float f0 = 0.0f, f1 = 0.0f, f2 = 0.0f, f3 = 0.0f;
        if (m < M) {
          const uint2 v = ptx::lds64(ptx::smem_u32(stg + C::kActOff + m * 256 + 8 * lane));
          f0 = act_to_float<F16>(static_cast<uint16_t>(v.x));
          f1 = act_to_float<F16>(static_cast<uint16_t>(v.x >> 16));
          f2 = act_to_float<F16>(static_cast<uint16_t>(v.y));
          f3 = act_to_float<F16>(static_cast<uint16_t>(v.y >> 16));
        }
        *reinterpret_cast<float4*>(stg + C::kActF32Off + m * C::kActF32Row + (lane >> 3) * kGvChunk +
                                   (lane & 7) * 16) = make_float4(f0, f1, f2, f3);
        float se = f0 + f2, so = f1 + f3;
#pragma unroll
        for (int d = 1; d < 8; d <<= 1) {
          se += __shfl_xor_sync(0xFFFFFFFFu, se, d);
          so += __shfl_xor_sync(0xFFFFFFFFu, so, d);
        }
        if ((lane & 7) == 0)
          *reinterpret_cast<float2*>(stg + C::kSumOff + m * 32 + (lane >> 3) * 8) = make_float2(se, so);
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&sh->ready[st]);
    }
    if (lane == 0 && *reinterpret_cast<volatile int*>(&sh->abort_flag)) {
      // copies still in flight land before the CTA exits
      const int first = issued > S ? issued - S : 0;
      for (int j = first; j < issued; ++j) {
        const uint64_t t0 = ptx::globaltimer_ns();
        while (!ptx::mbar_try_wait(&sh->full[j % S], (j / S) & 1))
          if (ptx::globaltimer_ns() - t0 > a.timeout_ns) break;
      }
    }
    return;
  }

  // -------------------------------------------------------------- compute
  const int t = threadIdx.x;
  const int rp = t >> 2;   // rows rp and rp + 64
  const int qk = t & 3;    // codes 32 qk .. 32 qk + 31 of each row
  UnitIter it;
  it.init(sched);
  float tot[2][MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) tot[0][m] = tot[1][m] = 0.0f;
  uint32_t nsync = 0;
  for (int i = 0; i < total; ++i) {
    const Unit u = it.next();
    if (u.seg_first) {
#pragma unroll
      for (int m = 0; m < MT; ++m) tot[0][m] = tot[1][m] = 0.0f;
    }
    const int st = i % S;
    if (!wait_warp(&sh->ready[st], (i / S) & 1, wc)) break;
    const uint32_t stg = ptx::smem_u32(smem + st * C::kStage);
    const uint4 c0 = ptx::lds128(stg + C::kCodeOff + rp * 64 + 16 * qk);
    const uint4 c1 = ptx::lds128(stg + C::kCodeOff + (rp + 64) * 64 + 16 * qk);
    const __half* sc = reinterpret_cast<const __half*>(smem + st * C::kStage + C::kScaleOff);
    const float s0 = __half2float(sc[rp]);
    const float s1 = __half2float(sc[rp + 64]);
    float x0[32], x1[32];
    nibbles_to_magic(c0.x, x0);
    nibbles_to_magic(c0.y, x0 + 8);
    nibbles_to_magic(c0.z, x0 + 16);
    nibbles_to_magic(c0.w, x0 + 24);
    nibbles_to_magic(c1.x, x1);
    nibbles_to_magic(c1.y, x1 + 8);
    nibbles_to_magic(c1.z, x1 + 16);
    nibbles_to_magic(c1.w, x1 + 24);
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      const uint32_t abase = stg + C::kActF32Off + m * C::kActF32Row + qk * kGvChunk;
      float p0[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      float p1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint4 av = ptx::lds128(abase + 16 * j);
        const float av4[4] = {__uint_as_float(av.x), __uint_as_float(av.y), __uint_as_float(av.z),
                              __uint_as_float(av.w)};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          p0[j >> 1] = fmaf(x0[4 * j + e], av4[e], p0[j >> 1]);
          p1[j >> 1] = fmaf(x1[4 * j + e], av4[e], p1[j >> 1]);
        }
      }
      const uint2 sv = ptx::lds64(stg + C::kSumOff + m * 32 + qk * 8);
      const float corr = fmaf(-136.0f, __uint_as_float(sv.x), -2056.0f * __uint_as_float(sv.y));
      tot[0][m] = fmaf(s0, ((p0[0] + p0[1]) + (p0[2] + p0[3])) + corr, tot[0][m]);
      tot[1][m] = fmaf(s1, ((p1[0] + p1[1]) + (p1[2] + p1[3])) + corr, tot[1][m]);
    }
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(&sh->empty[st]);
    if (!u.seg_last) continue;

    // the row totals: sum over the four k-quarters
#pragma unroll
    for (int m = 0; m < MT; ++m) {
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        float v = tot[r][m];
        v += __shfl_xor_sync(0xFFFFFFFFu, v, 1);
        v += __shfl_xor_sync(0xFFFFFFFFu, v, 2);
        tot[r][m] = v;
      }
    }
    const int tn = u.tile % a.n_tiles;
    if (u.whole) {
      if (qk == 0) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int n = tn * kTileW + rp + 64 * r;
          if (n >= a.N) continue;
          const float bias_f = a.bias != nullptr ? act_to_float<F16>(a.bias[n]) : 0.0f;
#pragma unroll
          for (int m = 0; m < MT; ++m)
            if (m < M) a.Y[static_cast<int64_t>(m) * a.N + n] = act_from_float<F16>(tot[r][m] + bias_f);
        }
      }
      continue;
    }
    // split tile: this CTA's partial, then the arrival count; the last
    // contributor sums every partial in k order
    constexpr int64_t kSlot = static_cast<int64_t>(MT) * kTileW;
    if (qk == 0) {
      float* slot = a.ws + (static_cast<int64_t>(cta) * 2 + u.slot) * kSlot;
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        slot[m * kTileW + rp] = tot[0][m];
        slot[m * kTileW + rp + 64] = tot[1][m];
      }
    }
    __threadfence();
    if (!gv_sync(sh, nsync, wc)) break;
    const SplitInfo si = split_info(a, u.sk_tile, ctas);
    if (t == 0) {
      uint32_t* cnt = a.counters + u.sk_tile;
      const uint32_t old = ptx::atom_add_acq_rel_gpu(cnt, 1u);
      const bool last = old == static_cast<uint32_t>(si.c_hi - si.c_lo);
      if (last) atomicExch(cnt, 0u);
      sh->fixup_last = last ? 1 : 0;
    }
    if (!gv_sync(sh, nsync, wc)) break;
    if (!sh->fixup_last) continue;
    __threadfence();
    if (qk == 0) {
      const float* lo = a.ws + (static_cast<int64_t>(si.c_lo) * 2 + si.slot_lo) * kSlot;
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int row = rp + 64 * r;
        const int n = tn * kTileW + row;
        if (n >= a.N) continue;
        const float bias_f = a.bias != nullptr ? act_to_float<F16>(a.bias[n]) : 0.0f;
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          if (m >= M) continue;
          float acc = __ldcg(lo + m * kTileW + row);
          for (int c = si.c_lo + 1; c <= si.c_hi; ++c)
            acc += __ldcg(a.ws + static_cast<int64_t>(c) * 2 * kSlot + m * kTileW + row);
          a.Y[static_cast<int64_t>(m) * a.N + n] = act_from_float<F16>(acc + bias_f);
        }
      }
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
  if (p.M > MT || p.K % kUnitK != 0) return cudaErrorInvalidValue;
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
  g.packed = static_cast<const uint8_t*>(p.packed);
  g.A = static_cast<const uint16_t*>(p.A);

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(s.grid));
  cfg.blockDim = dim3(kGvThreads);
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
  if (!c.simt || c.weight_format != kFmtInt4 || c.unit_groups != 1) return 0;
  switch (c.act_tile) {
    case 1: return c.stages == GvCfg<1>::kStages ? GvCfg<1>::kSmem : 0;
    case 2: return c.stages == GvCfg<2>::kStages ? GvCfg<2>::kSmem : 0;
    case 4: return c.stages == GvCfg<4>::kStages ? GvCfg<4>::kSmem : 0;
    case 8: return c.stages == GvCfg<8>::kStages ? GvCfg<8>::kSmem : 0;
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
