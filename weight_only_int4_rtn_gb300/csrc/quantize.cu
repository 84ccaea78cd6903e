// RTN INT4 quantize/pack kernel, group 128 along K (sm_103a).
//
// "Kernel dispatch and Humming quantization in PhyAI", section "Humming makes
// the separation useful": round-to-nearest post-training quantization at
// load, INT4, group size 128.  Per row n and group g the kernel computes
//   amax = max |w|;  s = fp16_rn(amax / 7.0f) (1 if that is 0);
//   q = clamp(rint_even(fl32(w / s)), -8, 7)
// and stores two's-complement nibbles (low nibble = even k) and s.  The codes
// go to the tiled storage layout of the GEMM: 128 rows x 128 K values per
// 8 KiB tile, tile (tn, g) at (tn * K/128 + g) * 8192, row-major inside; rows
// past N (up to the next multiple of 128) get zero codes.
//
// Work split.  A work tile is exactly one storage tile: 128 consecutive rows
// x one group (32 KiB of bf16 in, 8 KiB of codes and 256 B of scales out).
// A producer thread streams tiles with TMA into a ring of shared-memory
// stages, as two boxes of 128 rows x 64 values with the 128-byte swizzle (so
// that the per-row reads below hit 32 different banks).  Two teams of eight
// consumer warps take alternate tiles; in a team a pair of threads owns one
// row of the tile, i.e. one (row, group), each thread 64 of its values:
//   pass 1: absmax (packed bf16x2 max of |w|), combined across the pair,
//           then the scale, once per group;
//   pass 2: the codes, 8 packed 32-bit words per thread, stored as two
//           16-byte stores (the tile's 8 KiB are written by its 256 threads).
// Tiles are numbered group fastest within a 128-row block, so neighbouring
// CTAs read neighbouring 256-byte pieces of the same rows and write
// neighbouring 8 KiB blocks.
//
// Division.  The codes must equal rint_even(fl32(w / s)) bit for bit.  All
// 128 values of a group share s, so r = fl32(1/s) is computed once, and per
// value the quotient is q1 = fl32(w r), the remainder e = w - q1 s (exact:
// one fused multiply-add) and q2 = fl32(q1 + e r).  With r the correctly
// rounded reciprocal this one correction gives the correctly rounded quotient
// q2 = fl32(w / s) (Markstein's theorem), which a fused add of 1.5 * 2^23
// rounds half to even; the low four bits of that float are the code's
// two's-complement nibble.  For a normal scale |w / s| <= 7 (1 + 2^-11) < 7.5,
// so no clamp can be active.  A subnormal or infinite scale (rare) takes the IEEE
// division __fdiv_rn and the clamp value by value.
//
// Stochastic-rounding mode ("Piper Kernels", section "Stochastic
// quantization"; the scales stay the round-to-nearest ones, section "ConvRot
// INT8").  The same kernel with the last step replaced: with r = fl32(w / s)
// (the same correctly rounded quotient), a value interior to the code range
// (-8 <= r <= 7) takes floor(r) + 1 when u < r - floor(r), else floor(r);
// others take the round-to-nearest code.  u is drawn from Philox4x32-10
// (Salmon et al., "Parallel random numbers: as easy as 1, 2, 3") by logical
// element offset e = n * K + k: key (seed mod 2^32, seed div 2^32), counter
// (e div 4 as two 32-bit words, 0, 0), word e mod 4, u = (word >> 8) * 2^-24.
// Exact hits (r integral) and values outside the range are never perturbed,
// and the draws do not depend on the launch geometry.
//
// INT8 mode (the W8A16 scheme: "Kernel dispatch and Humming quantization in
// PhyAI", section "Choose precision by layer and hardware").  The same
// kernel with 8-bit codes: s = fp16_rn(amax / 127.0f) (1 if that is 0), q =
// clamp(rint_even(fl32(w / s)), -128, 127), one two's-complement byte per
// code, tiles of 128 rows x 128 K values (16 KiB, 128 B per row).  For a
// normal scale |w / s| <= 127 (1 + 2^-11) < 127.5, so again no clamp is
// active and the low byte of the rounded float is the code.
//
// FP4 modes (MXFP4 and NVFP4 weights: "Kernel dispatch and Humming
// quantization in PhyAI", section "Choose precision by layer and hardware";
// NVFP4's blocks of 16 and per-tensor scale: "Piper Kernels", section "NVFP4
// construction").  E2M1 codes (sign in the nibble's top bit) in the INT4 tile
// layout; the rounding is the conversion instruction cvt.rn.satfinite.e2m1x2
// (nearest, ties to the even mantissa, saturating at 6), with the sign of a
// code whose magnitude rounds to 0 cleared afterwards.
//   MXFP4 (OCP MX v1.0): blocks of 32 values; E = floor(log2 amax) - 2 + 127
//   read off amax's exponent field (127 for an all-zero block), one scale
//   byte per block; the elements are w * 2^(127 - E), an exact product.
//   NVFP4: a first kernel takes the tensor's absmax (atomic max of the bit
//   patterns, non-negative floats order like integers) into the second word
//   of the caller's tensor-scale pair; here g = fl32(amax / 2688) (1 for a
//   zero tensor) is written to the first word; per block of 16, the scale
//   code is E4M3_rn_sat(fl32(fl32(amax_b / 6) / g)) (cvt.rn.satfinite.e4m3x2)
//   and the elements are fl32(w / fl32(s_b g)) by IEEE division (the step
//   is a full fp32 value, for which the one-step correction of the other
//   modes is not always correctly rounded).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"
#include "waits.cuh"

namespace w4a16 {

namespace {

constexpr float kRoundMagic = 12582912.0f;        // 1.5 * 2^23

constexpr int kQRows = 128;                       // rows per tile (one storage tile)
constexpr int kQBoxBytes = kQRows * 128;          // one box: 128 rows x 64 bf16
constexpr int kQTileBytes = 2 * kQBoxBytes;       // 32 KiB
constexpr int kQStages = 6;                       // even: each stage feeds one tile team
constexpr int kQTeamWarps = 8;                    // a team: 256 threads, two per row
constexpr int kQConsumerWarps = 2 * kQTeamWarps;  // two teams, alternate tiles
constexpr int kQThreads = 32 * (kQConsumerWarps + 1);

// A launch quantizes up to kQMaxGroup independent weights: weight p owns the
// CTAs cta_start[p] .. cta_start[p+1]-1.  A single weight is a group of one.
constexpr int kQMaxGroup = 8;
struct QGroupArgs {
  CUtensorMap tm[kQMaxGroup];
  uint32_t* packed[kQMaxGroup];
  void* scales[kQMaxGroup];   // fp16 (INT4, INT8) or bytes (FP4 block scales)
  int N[kQMaxGroup];
  int G[kQMaxGroup];
  int tiles[kQMaxGroup];
  int cta_start[kQMaxGroup + 1];
  int count;
  uint64_t seed;   // stochastic-rounding mode: the generator's key
  float* tscale;   // NVFP4 mode: {g (written here), tensor absmax (read)}
};

struct QShared {
  uint64_t full[kQStages];
  uint64_t empty[kQStages];
  int abort_flag;
};

// 16-byte chunk c (0..7) of row r of a 128-byte-swizzled box.
__device__ __forceinline__ uint32_t chunk_addr(uint32_t box, int r, int c) {
  return box + r * 128 + ((c ^ (r & 7)) << 4);
}

// Nibbles of 8 rounded values (float bit patterns, code in the low 4 bits)
// into one word, code i in nibble i.
__device__ __forceinline__ uint32_t pack8(const uint32_t (&y)[8]) {
  uint32_t p[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) p[i] = (y[2 * i] & 0xFu) | ((y[2 * i + 1] << 4) & ~0xFu);
  const uint32_t lo = ptx::prmt(p[0], p[1], 0x0040);
  const uint32_t hi = ptx::prmt(p[2], p[3], 0x0040);
  return ptx::prmt(lo, hi, 0x5410);
}

// The quotient fl32(w / s) from r = fl32(1 / s): q1 = fl32(w r), the
// remainder e = w - q1 s (exact: one fused multiply-add, while it is a
// normal float) and one correction q2 = fl32(q1 + e r) (Markstein's
// refinement).  The INT4 and INT8 modes use it for normal, finite fp16
// scales (11 significant bits), and w4a16_selftest_quotient checks it
// against the IEEE division over every such scale and every bf16 weight
// those modes can meet: no code differs, and no quotient differs where
// |w| >= 2^-100.  For general fp32 divisors (the NVFP4 steps) the same
// check finds codes that differ, so that mode divides with __fdiv_rn.
__device__ __forceinline__ float quotient_corrected(float w, float s, float r) {
  const float q1 = __fmul_rn(w, r);
  const float e = fmaf(-q1, s, w);
  return fmaf(e, r, q1);
}

// True for an fp16 scale that takes the corrected quotient: normal and
// finite.  A subnormal scale, and an infinite one (amax / 7 above fp16's
// range: outside the method's preconditions, but then the IEEE division
// gives the oracle's code 0 where the remainder step would give NaN), take
// the IEEE division value by value.
__device__ __forceinline__ bool scale_fast(__half s16) {
  const uint32_t e = __half_as_ushort(s16) & 0x7C00u;
  return e != 0u && e != 0x7C00u;
}

// Codes of 8 values for a normal scale: the corrected quotient, rounded half
// to even.  |w / s| < 7.5, so no clamp is active.
__device__ __forceinline__ uint32_t codes_corrected(const float (&f)[8], float s, float r) {
  uint32_t y[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    y[i] = __float_as_uint(__fadd_rn(quotient_corrected(f[i], s, r), kRoundMagic));
  return pack8(y);
}

// Codes of 8 values for a subnormal scale: IEEE quotient, clamp (|w / s|
// may exceed the code range), round half to even.
__device__ __forceinline__ uint32_t codes_exact(const float (&f)[8], float s) {
  uint32_t y[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float tc = fminf(fmaxf(__fdiv_rn(f[i], s), -8.0f), 7.0f);
    y[i] = __float_as_uint(__fadd_rn(tc, kRoundMagic));
  }
  return pack8(y);
}

// ------------------------------------------------- stochastic-rounding mode
constexpr uint32_t kPhiloxM0 = 0xD2511F53u;
constexpr uint32_t kPhiloxM1 = 0xCD9E8D57u;
constexpr uint32_t kPhiloxW0 = 0x9E3779B9u;
constexpr uint32_t kPhiloxW1 = 0xBB67AE85u;

// Philox4x32-10: ten rounds; one round maps (c0, c1, c2, c3) under (k0, k1)
// to (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2), hi(M0 c0) ^ c3 ^ k1, lo(M0 c0)), the
// key advancing by the Weyl constants before every round but the first.
__device__ __forceinline__ void philox4x32_10(uint32_t (&c)[4], uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    // one 32 x 32 -> 64-bit product gives both halves
    const uint64_t p0 = static_cast<uint64_t>(kPhiloxM0) * c[0];
    const uint64_t p1 = static_cast<uint64_t>(kPhiloxM1) * c[2];
    const uint32_t n0 = static_cast<uint32_t>(p1 >> 32) ^ c[1] ^ (k0 + static_cast<uint32_t>(r) * kPhiloxW0);
    const uint32_t n2 = static_cast<uint32_t>(p0 >> 32) ^ c[3] ^ (k1 + static_cast<uint32_t>(r) * kPhiloxW1);
    c[0] = n0;
    c[1] = static_cast<uint32_t>(p1);
    c[2] = n2;
    c[3] = static_cast<uint32_t>(p0);
  }
}

// Codes of 8 values at logical offsets e0 .. e0 + 7 (e0 a multiple of 4)
// from their correctly rounded quotients x[i] = fl32(w / s): stochastic
// between the adjacent integers where -8 <= x <= 7, nearest (clamped)
// elsewhere.
__device__ __forceinline__ uint32_t codes_stochastic(const float (&x)[8], uint64_t e0, uint32_t k0,
                                                     uint32_t k1) {
  uint32_t y[8];
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const uint64_t ctr = (e0 >> 2) + static_cast<uint64_t>(half);
    uint32_t c[4] = {static_cast<uint32_t>(ctr), static_cast<uint32_t>(ctr >> 32), 0u, 0u};
    philox4x32_10(c, k0, k1);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float r = x[4 * half + w];
      const float u = __uint2float_rn(c[w] >> 8) * 5.9604644775390625e-08f;   // * 2^-24, exact
      const float lo = floorf(r);
      const float up = (u < r - lo) ? 1.0f : 0.0f;                          // r - lo exact
      const bool interior = (r >= -8.0f) && (r <= 7.0f);
      const float code = interior ? lo + up : fminf(fmaxf(r, -8.0f), 7.0f);
      y[4 * half + w] = __float_as_uint(__fadd_rn(code, kRoundMagic));     // rint for the clamp
    }
  }
  return pack8(y);
}

// Low bytes of 4 rounded values (float bit patterns) into one word, code i
// in byte i.
__device__ __forceinline__ uint32_t pack4_bytes(uint32_t y0, uint32_t y1, uint32_t y2, uint32_t y3) {
  return ptx::prmt(ptx::prmt(y0, y1, 0x0040), ptx::prmt(y2, y3, 0x0040), 0x5410);
}

// INT8 codes of 8 values (two words), normal scale: the corrected quotient
// rounded half to even (|w / s| < 127.5: no clamp is active).
__device__ __forceinline__ void codes8_corrected(const float (&f)[8], float s, float r,
                                                 uint32_t& w0, uint32_t& w1) {
  uint32_t y[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    y[i] = __float_as_uint(__fadd_rn(quotient_corrected(f[i], s, r), kRoundMagic));
  w0 = pack4_bytes(y[0], y[1], y[2], y[3]);
  w1 = pack4_bytes(y[4], y[5], y[6], y[7]);
}

// INT8 codes of 8 values, subnormal scale: IEEE quotient, clamp, round.
__device__ __forceinline__ void codes8_exact(const float (&f)[8], float s, uint32_t& w0,
                                             uint32_t& w1) {
  uint32_t y[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float tc = fminf(fmaxf(__fdiv_rn(f[i], s), -128.0f), 127.0f);
    y[i] = __float_as_uint(__fadd_rn(tc, kRoundMagic));
  }
  w0 = pack4_bytes(y[0], y[1], y[2], y[3]);
  w1 = pack4_bytes(y[4], y[5], y[6], y[7]);
}

// ------------------------------------------------------------- FP4 modes
// E2M1 codes of two values in one byte: b in the low nibble, a in the high
// nibble (round to nearest even, saturating at +-6).
__device__ __forceinline__ uint32_t e2m1x2(float a, float b) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
      : "=r"(r)
      : "f"(a), "f"(b));
  return r;
}

// Eight E2M1 codes (x[i] in nibble i) with the sign of zero magnitudes
// cleared: a nibble keeps its sign bit only if its low three bits are not 0.
__device__ __forceinline__ uint32_t e2m1_word(const float (&x)[8]) {
  const uint32_t w = ptx::prmt(ptx::prmt(e2m1x2(x[1], x[0]), e2m1x2(x[3], x[2]), 0x0040),
                               ptx::prmt(e2m1x2(x[5], x[4]), e2m1x2(x[7], x[6]), 0x0040), 0x5410);
  const uint32_t mag = w & 0x77777777u;
  return mag | (w & ((mag + 0x77777777u) & 0x88888888u));
}

// E4M3 code (round to nearest even, saturating at 448) of a non-negative
// float.
__device__ __forceinline__ uint32_t e4m3_code(float v) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));
  return static_cast<uint32_t>(r) & 0xFFu;
}

// Value of an E4M3 code (bias 7): its 7 bits placed under the fp32 exponent
// field's low bits give the value * 2^-120 (normal or subnormal alike), and
// one exact product restores the scale.
__device__ __forceinline__ float e4m3_value(uint32_t code) {
  return __uint_as_float((code & 0x7Fu) << 20) * 0x1p120f;
}

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint32_t bf16x2_absmax(uint32_t acc, uint32_t w) {
  const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&acc);
  const __nv_bfloat162 b = __habs2(*reinterpret_cast<const __nv_bfloat162*>(&w));
  const __nv_bfloat162 m = __hmax2(a, b);
  return *reinterpret_cast<const uint32_t*>(&m);
}

// |bf16| maximum of 16 values (two 16-byte chunks) as a float.
__device__ __forceinline__ float absmax16(const uint4& a, const uint4& b) {
  uint32_t m = bf16x2_absmax(bf16x2_absmax(bf16x2_absmax(0u, a.x), a.y),
                             bf16x2_absmax(bf16x2_absmax(0u, a.z), a.w));
  m = bf16x2_absmax(m, bf16x2_absmax(bf16x2_absmax(bf16x2_absmax(0u, b.x), b.y),
                                     bf16x2_absmax(bf16x2_absmax(0u, b.z), b.w)));
  return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xFFFF0000u));
}

// Tensor absmax of an NVFP4 weight: every thread takes 16-byte pieces of
// the [N, K] bf16 weight (N K a multiple of 128), reduces them, a warp
// reduces its lanes and lane 0 takes an atomic max into *amax_bits (zeroed
// before the launch).
__global__ void __launch_bounds__(256) tensor_absmax_kernel(const uint4* __restrict__ w,
                                                            int64_t n16, uint32_t* amax_bits) {
  uint32_t m = 0;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16;
       i += stride) {
    const uint4 v = __ldg(w + i);
    m = bf16x2_absmax(m, v.x);
    m = bf16x2_absmax(m, v.y);
    m = bf16x2_absmax(m, v.z);
    m = bf16x2_absmax(m, v.w);
  }
  uint32_t a = __float_as_uint(fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xFFFF0000u)));
  a = __reduce_max_sync(0xFFFFFFFFu, a);
  if ((threadIdx.x & 31) == 0 && a != 0) atomicMax(amax_bits, a);
}

// MODE: kModeRtn4 (INT4, round to nearest), kModeSr4 (INT4, stochastic
// rounding), kModeRtn8 (INT8, round to nearest).
constexpr int kModeRtn4 = 0;
constexpr int kModeSr4 = 1;
constexpr int kModeRtn8 = 2;
constexpr int kModeMx4 = 3;   // MXFP4
constexpr int kModeNv4 = 4;   // NVFP4
constexpr int kModes = 5;

template <int MODE>
__global__ void __launch_bounds__(kQThreads, 1)
    rtn_quantize_kernel(const __grid_constant__ QGroupArgs q, uint32_t* err, uint64_t timeout_ns) {
  constexpr bool SR = MODE == kModeSr4;
  constexpr bool W8 = MODE == kModeRtn8;
  constexpr bool FP4 = MODE == kModeMx4 || MODE == kModeNv4;
  // this CTA's weight and its index in that weight's sub-grid
  int prob = 0;
  while (prob + 1 < q.count && static_cast<int>(blockIdx.x) >= q.cta_start[prob + 1]) ++prob;
  const CUtensorMap* const tm_w = &q.tm[prob];
  const int N = q.N[prob];
  const int G = q.G[prob];
  const int tiles = q.tiles[prob];
  uint32_t* const packed = q.packed[prob];
  const int cta = static_cast<int>(blockIdx.x) - q.cta_start[prob];
  const int ctas = q.cta_start[prob + 1] - q.cta_start[prob];
  extern __shared__ __align__(1024) uint8_t q_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(q_smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  QShared* sh = reinterpret_cast<QShared*>(smem + kQStages * kQTileBytes);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kQStages; ++s) {
      ptx::mbar_init(&sh->full[s], 1);
      ptx::mbar_init(&sh->empty[s], kQTeamWarps);
    }
    sh->abort_flag = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tmap(tm_w);
  }
  __syncthreads();
  const WaitCtx wc{err, timeout_ns, &sh->abort_flag};
  // The weight may be written by the previous kernel on the stream; the next
  // kernel may start its own set-up now (it waits for this grid to complete
  // before it reads anything this kernel writes).
  ptx::grid_dependency_wait();
  ptx::grid_launch_dependents();

  // NVFP4: the tensor scale from the absmax the previous kernel reduced
  float g_t = 1.0f;
  if constexpr (MODE == kModeNv4) {
    const float amax_t = __ldcg(q.tscale + 1);
    g_t = amax_t == 0.0f ? 1.0f : __fdiv_rn(amax_t, 2688.0f);
    if (blockIdx.x == 0 && threadIdx.x == 0) q.tscale[0] = g_t;
  }

  const int n_local = (tiles - cta + ctas - 1) / ctas;

  if (warp == kQConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int issued = 0;
      for (int i = 0; i < n_local; ++i) {
        const int stage = i % kQStages;
        if (!wait_one(&sh->empty[stage], ((i / kQStages) & 1) ^ 1, wc)) break;
        const int t = cta + i * ctas;
        const int tn = t / G;
        const int g = t - tn * G;
        uint8_t* dst = smem + stage * kQTileBytes;
        ptx::mbar_arrive_expect_tx(&sh->full[stage], kQTileBytes);
        ptx::tma_load_2d(dst, tm_w, &sh->full[stage], g * kGroup, tn * kQRows);
        ptx::tma_load_2d(dst + kQBoxBytes, tm_w, &sh->full[stage], g * kGroup + 64, tn * kQRows);
        issued = i + 1;
      }
      if (*reinterpret_cast<volatile int*>(&sh->abort_flag)) {
        // let the copies in flight land before the CTA exits
        const int first = issued > kQStages ? issued - kQStages : 0;
        for (int i = first; i < issued; ++i) {
          const uint64_t t0 = ptx::globaltimer_ns();
          while (!ptx::mbar_try_wait(&sh->full[i % kQStages], (i / kQStages) & 1))
            if (ptx::globaltimer_ns() - t0 > timeout_ns) break;
        }
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  // Team `team` takes tiles team, team + 2, ...  Thread pair (2 row, 2 row + 1)
  // owns row `row`: half h = box h = values 64 h .. 64 h + 63 (the two halves
  // read their chunks in different orders, so one instruction never hits the
  // same bank in both boxes).
  const int team = warp / kQTeamWarps;
  const int tt = (warp % kQTeamWarps) * 32 + lane;   // 0..255
  const int row = tt >> 1;
  const int h = tt & 1;
  for (int i = team; i < n_local; i += 2) {
    const int stage = i % kQStages;
    if (!wait_warp(&sh->full[stage], (i / kQStages) & 1, wc)) break;
    const int t = cta + i * ctas;
    const int tn = t / G;
    const int g = t - tn * G;
    const uint32_t box = ptx::smem_u32(smem + stage * kQTileBytes) + h * kQBoxBytes;
    const int n = tn * kQRows + row;

    if constexpr (FP4) {
      // this thread's half row: values 64 h .. 64 h + 63 of the group, 32
      // code bytes at word 8 h of the row's 16 words.  Blocks are taken in
      // the rotated order (the two threads of a pair read chunks four apart,
      // so one instruction never hits one bank twice).
      uint32_t* const dst = packed + ((static_cast<int64_t>(tn) * G + g) * kQRows + row) * 16 + 8 * h;
      uint8_t* const sc = static_cast<uint8_t*>(q.scales[prob]);
      if constexpr (MODE == kModeMx4) {
#pragma unroll
        for (int bb = 0; bb < 2; ++bb) {
          const int b = bb ^ h;   // block of 32 values: chunks 4 b .. 4 b + 3
          uint4 v[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) v[j] = ptx::lds128(chunk_addr(box, row, 4 * b + j));
          const float amax = fmaxf(absmax16(v[0], v[1]), absmax16(v[2], v[3]));
          const uint32_t ef = __float_as_uint(amax) >> 23;   // amax >= 0: the exponent field
          const uint32_t E = amax == 0.0f ? 127u : (ef > 2u ? ef - 2u : 0u);
          // 2^(127 - E): E <= 252 for bf16 input, so the factor is normal
          const float inv = __uint_as_float((254u - E) << 23);
          uint32_t words[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            float f[8];
            unpack8(v[j], f);
#pragma unroll
            for (int i = 0; i < 8; ++i) f[i] = __fmul_rn(f[i], inv);
            words[j] = e2m1_word(f);
          }
          reinterpret_cast<uint4*>(dst)[b] = make_uint4(words[0], words[1], words[2], words[3]);
          if (n < N) sc[static_cast<int64_t>(4 * g + 2 * h + b) * N + n] = static_cast<uint8_t>(E);
        }
      } else {
#pragma unroll
        for (int bb = 0; bb < 4; ++bb) {
          const int b = (bb + 2 * h) & 3;   // block of 16 values: chunks 2 b, 2 b + 1
          const uint4 v0 = ptx::lds128(chunk_addr(box, row, 2 * b));
          const uint4 v1 = ptx::lds128(chunk_addr(box, row, 2 * b + 1));
          const float amax = absmax16(v0, v1);
          const uint32_t code = e4m3_code(__fdiv_rn(__fdiv_rn(amax, 6.0f), g_t));
          const float step = __fmul_rn(e4m3_value(code), g_t);
          float f[16];
          unpack8(v0, *reinterpret_cast<float(*)[8]>(&f[0]));
          unpack8(v1, *reinterpret_cast<float(*)[8]>(&f[8]));
          // IEEE division: the step is a full fp32 value (fl32(e4m3 * g)),
          // for which the one-step reciprocal correction is not always the
          // correctly rounded quotient (w4a16_selftest_quotient finds E2M1
          // codes that differ), unlike the fp16 scales of the other modes
          if (step == 0.0f) {
#pragma unroll
            for (int i = 0; i < 16; ++i) f[i] = 0.0f;
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) f[i] = __fdiv_rn(f[i], step);
          }
          const uint32_t w0 = e2m1_word(*reinterpret_cast<const float(*)[8]>(&f[0]));
          const uint32_t w1 = e2m1_word(*reinterpret_cast<const float(*)[8]>(&f[8]));
          reinterpret_cast<uint2*>(dst)[b] = make_uint2(w0, w1);
          if (n < N) sc[static_cast<int64_t>(8 * g + 4 * h + b) * N + n] = static_cast<uint8_t>(code);
        }
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&sh->empty[stage]);
      continue;
    }

    // pass 1: absmax of the row's 128 values (two independent chains per
    // thread, then across the pair), and the scale
    uint32_t ma = 0, mb = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint4 v = ptx::lds128(chunk_addr(box, row, (j + 4 * h) & 7));
      ma = bf16x2_absmax(ma, v.x);
      mb = bf16x2_absmax(mb, v.y);
      ma = bf16x2_absmax(ma, v.z);
      mb = bf16x2_absmax(mb, v.w);
    }
    ma = bf16x2_absmax(ma, mb);
    float amax = fmaxf(__uint_as_float(ma << 16), __uint_as_float(ma & 0xFFFF0000u));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
    __half s16 = __float2half_rn(__fdiv_rn(amax, W8 ? 127.0f : 7.0f));
    if (__half_as_ushort(s16) == 0) s16 = __ushort_as_half(0x3C00);   // zero rule: 1.0
    const float s = __half2float(s16);
    const float r = __frcp_rn(s);

    // pass 2: the codes.  The quotient is corrected to fl32(w / s) for every
    // normal scale (no divergence between rows); a subnormal scale takes the
    // IEEE division and the clamp.
    // this thread's half row of codes: 8 words (INT4) or 16 words (INT8)
    constexpr int kRowWords = W8 ? 32 : 16;
    uint32_t* const dst =
        packed + ((static_cast<int64_t>(tn) * G + g) * kQRows + row) * kRowWords + (kRowWords / 2) * h;
    if constexpr (W8) {
      if (scale_fast(s16)) {
        // chunks in the rotated order (j + 4 h) mod 8, as in the INT4 path;
        // chunk c's two words are words 2c, 2c + 1 of the half row, so the
        // j-th pair of chunks goes to 16-byte store (j + 2 h) mod 4
        uint32_t words[16];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          float f[8];
          unpack8(ptx::lds128(chunk_addr(box, row, (j + 4 * h) & 7)), f);
          codes8_corrected(f, s, r, words[2 * j], words[2 * j + 1]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
          reinterpret_cast<uint4*>(dst)[(i + 2 * h) & 3] =
              make_uint4(words[4 * i], words[4 * i + 1], words[4 * i + 2], words[4 * i + 3]);
      } else {
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          float f[8];
          unpack8(ptx::lds128(chunk_addr(box, row, c)), f);
          codes8_exact(f, s, dst[2 * c], dst[2 * c + 1]);
        }
      }
    } else if constexpr (SR) {
      // logical offset of this thread's first value: row n, k = 128 g + 64 h
      const uint64_t e_row = static_cast<uint64_t>(tn * kQRows + row) * static_cast<uint64_t>(G) *
                                 kGroup + static_cast<uint64_t>(g * kGroup + 64 * h);
      const uint32_t k0 = static_cast<uint32_t>(q.seed);
      const uint32_t k1 = static_cast<uint32_t>(q.seed >> 32);
      const bool normal = scale_fast(s16);
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        float f[8];
        unpack8(ptx::lds128(chunk_addr(box, row, c)), f);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (normal) {
            f[i] = quotient_corrected(f[i], s, r);   // fl32(w / s), as in the RTN mode
          } else {
            f[i] = __fdiv_rn(f[i], s);
          }
        }
        dst[c] = codes_stochastic(f, e_row + 8 * c, k0, k1);
      }
    } else if (scale_fast(s16)) {
      uint32_t words[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        float f[8];
        unpack8(ptx::lds128(chunk_addr(box, row, (j + 4 * h) & 7)), f);
        words[j] = codes_corrected(f, s, r);   // chunk (j + 4 h) mod 8
      }
      const uint4 w0 = make_uint4(words[0], words[1], words[2], words[3]);
      const uint4 w1 = make_uint4(words[4], words[5], words[6], words[7]);
      reinterpret_cast<uint4*>(dst)[0] = h ? w1 : w0;
      reinterpret_cast<uint4*>(dst)[1] = h ? w0 : w1;
    } else {
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        float f[8];
        unpack8(ptx::lds128(chunk_addr(box, row, c)), f);
        dst[c] = codes_exact(f, s);
      }
    }
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(&sh->empty[stage]);
    if (h == 0 && n < N) static_cast<__half*>(q.scales[prob])[static_cast<int64_t>(g) * N + n] = s16;
  }
}

}  // namespace

namespace {

cudaError_t launch_quantize_mode(const QuantizeProblem* probs, int count, int num_sms,
                                 uint32_t* error_word, uint64_t timeout_ns, cudaStream_t stream,
                                 int mode, uint64_t seed, float* tscale) {
  static_assert(kQMaxGroup == kMaxQuantizeGroup, "group size of the kernel arguments");
  if (count < 1 || count > kQMaxGroup) return cudaErrorInvalidValue;
  QGroupArgs q{};
  int64_t total_tiles = 0;
  for (int i = 0; i < count; ++i) {
    const QuantizeProblem& p = probs[i];
    // the weight as [N][K] bf16; boxes of 128 rows x 64 values, 128-byte
    // swizzle; rows past N read as zeros
    if (encode_tmap_2d(&q.tm[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.W, static_cast<uint64_t>(p.K),
                       static_cast<uint64_t>(p.N), static_cast<uint64_t>(p.K) * 2, 64, kQRows,
                       CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    q.packed[i] = static_cast<uint32_t*>(p.packed);
    q.scales[i] = p.scales;
    q.N[i] = static_cast<int>(p.N);
    q.G[i] = static_cast<int>(p.K / kGroup);
    q.tiles[i] = static_cast<int>((p.N + kQRows - 1) / kQRows) * q.G[i];
    total_tiles += q.tiles[i];
  }
  // CTAs in proportion to each weight's tiles, at least one each, at most
  // one per tile, no more than the SMs in total
  int ctas[kQMaxGroup];
  int used = 0;
  for (int i = 0; i < count; ++i) {
    int64_t c = (static_cast<int64_t>(num_sms) * q.tiles[i]) / total_tiles;
    if (c < 1) c = 1;
    if (c > q.tiles[i]) c = q.tiles[i];
    ctas[i] = static_cast<int>(c);
    used += ctas[i];
  }
  while (used < num_sms) {   // hand spare SMs to the weights with most tiles per CTA
    int best = -1;
    for (int i = 0; i < count; ++i)
      if (ctas[i] < q.tiles[i] &&
          (best < 0 || static_cast<int64_t>(q.tiles[i]) * ctas[best] > static_cast<int64_t>(q.tiles[best]) * ctas[i]))
        best = i;
    if (best < 0) break;
    ++ctas[best];
    ++used;
  }
  int start = 0;
  for (int i = 0; i < count; ++i) {
    q.cta_start[i] = start;
    start += ctas[i];
  }
  q.cta_start[count] = start;
  q.count = count;
  q.seed = seed;
  q.tscale = tscale;
  auto kernel = mode == kModeRtn8 ? rtn_quantize_kernel<kModeRtn8>
                : mode == kModeSr4 ? rtn_quantize_kernel<kModeSr4>
                : mode == kModeMx4 ? rtn_quantize_kernel<kModeMx4>
                : mode == kModeNv4 ? rtn_quantize_kernel<kModeNv4>
                                   : rtn_quantize_kernel<kModeRtn4>;

  constexpr size_t smem = static_cast<size_t>(kQStages) * kQTileBytes + sizeof(QShared) + 1024;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static bool attr_set[kModes][64] = {};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[mode][dev]) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    attr_set[mode][dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(start));
  cfg.blockDim = dim3(kQThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  // programmatic dependent launch: set-up overlaps the previous kernel's tail
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, q, error_word, timeout_ns);
}

// Self test of quotient_corrected against the IEEE division __fdiv_rn.
// Block b takes one divisor d and every finite bf16 value w (both signs)
// with |w| <= bound * d.  For each pair it compares what the quantizer
// stores, the code (rint, ties to even, of the quotient for INT4 and INT8;
// the E2M1 conversion for NVFP4), and the quotient itself; one atomic per
// warp adds the counts to counts[0] (pairs checked), counts[1] (codes that
// differ), counts[2] (quotients that differ where |w| >= 2^-100: then the
// remainder w - q1 d, about 2^-24 |w|, is a normal float and the fused
// multiply-add gives it exactly) and counts[3] (quotients that differ
// anywhere; for |w| < 2^-100 and a normal fp16 scale the quotient is below
// 2^-86, so its code is 0 either way).  Floats compare as values, so +0 and
// -0 are equal.
//   mode 0 (INT4): d = every normal finite fp16 scale, bound 7.5 (a normal
//     scale s = fp16(amax / 7) keeps |w| <= amax <= 7.0035 s);
//   mode 1 (INT8): the same scales, bound 127.5;
//   mode 2 (fp32 divisors of the NVFP4 form): d = fl32(e4m3(c) * g) for the
//     E4M3 codes c = 1 .. 126 and 512 tensor scales g = 2^e (1 + f), e in
//     [-40, 40] and f from a fixed integer hash; bound 8 (E2M1 codes
//     saturate at 6); normal d only.  No kernel uses the corrected quotient
//     for such divisors: this mode is the check that shows why (it finds
//     codes that differ), so the NVFP4 quantize divides with __fdiv_rn.
__global__ void __launch_bounds__(256) quotient_selftest_kernel(int mode,
                                                                unsigned long long* counts) {
  float d, bound;
  if (mode == 2) {
    const uint32_t c = 1u + blockIdx.x % 126u;
    uint32_t h = blockIdx.x / 126u;
    h = (h ^ 61u) ^ (h >> 16);
    h *= 9u;
    h ^= h >> 4;
    h *= 0x27D4EB2Du;
    h ^= h >> 15;
    const int ex = static_cast<int>(h % 81u) - 40;
    const float g = __uint_as_float(static_cast<uint32_t>(127 + ex) << 23 | (h >> 9));
    d = __fmul_rn(e4m3_value(c), g);
    bound = 8.0f;
    if ((__float_as_uint(d) & 0x7F800000u) == 0u || (__float_as_uint(d) & 0x7F800000u) == 0x7F800000u)
      return;
  } else {
    d = __half2float(__ushort_as_half(static_cast<unsigned short>(0x0400u + blockIdx.x)));
    bound = mode == 0 ? 7.5f : 127.5f;
  }
  const float r = __frcp_rn(d);
  const float lim = bound * d;
  unsigned long long cnt[4] = {0, 0, 0, 0};
  for (uint32_t b = threadIdx.x; b < 0x7F80u; b += blockDim.x) {
    const float w = __uint_as_float(b << 16);
    if (w > lim) continue;
#pragma unroll
    for (int sgn = 0; sgn < 2; ++sgn) {
      const float x = sgn ? -w : w;
      const float q = quotient_corrected(x, d, r);
      const float ref = __fdiv_rn(x, d);
      bool code_differs;
      if (mode == 2) {
        code_differs = e2m1x2(q, q) != e2m1x2(ref, ref);
      } else {
        code_differs = __fadd_rn(q, kRoundMagic) != __fadd_rn(ref, kRoundMagic);
      }
      cnt[0] += 1;
      cnt[1] += code_differs ? 1 : 0;
      cnt[2] += (q != ref && w >= 0x1p-100f) ? 1 : 0;
      cnt[3] += q != ref ? 1 : 0;
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cnt[i] += __shfl_xor_sync(0xFFFFFFFFu, cnt[i], o);
  }
  if ((threadIdx.x & 31) == 0) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (cnt[i] != 0) atomicAdd(counts + i, cnt[i]);
  }
}

}  // namespace

cudaError_t launch_rtn_quantize_group(const QuantizeProblem* probs, int count, int num_sms,
                                      uint32_t* error_word, uint64_t timeout_ns,
                                      cudaStream_t stream, const uint64_t* sr_seed, bool int8) {
  if (int8 && sr_seed != nullptr) return cudaErrorInvalidValue;
  const int mode = int8 ? kModeRtn8 : sr_seed != nullptr ? kModeSr4 : kModeRtn4;
  return launch_quantize_mode(probs, count, num_sms, error_word, timeout_ns, stream, mode,
                              sr_seed != nullptr ? *sr_seed : 0, nullptr);
}

cudaError_t launch_rtn_quantize(const void* W, int64_t N, int64_t K, void* packed, void* scales,
                                int num_sms, uint32_t* error_word, uint64_t timeout_ns,
                                cudaStream_t stream, const uint64_t* sr_seed, bool int8) {
  QuantizeProblem p{W, N, K, packed, scales};
  return launch_rtn_quantize_group(&p, 1, num_sms, error_word, timeout_ns, stream, sr_seed, int8);
}

cudaError_t launch_fp4_quantize(const void* W, int64_t N, int64_t K, void* packed, void* scales,
                                float* tensor_scale, int format, int num_sms,
                                uint32_t* error_word, uint64_t timeout_ns, cudaStream_t stream) {
  QuantizeProblem p{W, N, K, packed, scales};
  if (format == kFmtMxfp4)
    return launch_quantize_mode(&p, 1, num_sms, error_word, timeout_ns, stream, kModeMx4, 0,
                                nullptr);
  if (format != kFmtNvfp4 || tensor_scale == nullptr) return cudaErrorInvalidValue;
  // the tensor absmax into tensor_scale[1] (zeroed first), then the codes
  cudaError_t e = cudaMemsetAsync(tensor_scale, 0, 2 * sizeof(float), stream);
  if (e != cudaSuccess) return e;
  const int64_t n16 = N * K / 8;
  int blocks = 4 * num_sms;
  if (static_cast<int64_t>(blocks) * 256 > n16) blocks = static_cast<int>((n16 + 255) / 256);
  tensor_absmax_kernel<<<blocks, 256, 0, stream>>>(static_cast<const uint4*>(W), n16,
                                                     reinterpret_cast<uint32_t*>(tensor_scale + 1));
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_quantize_mode(&p, 1, num_sms, error_word, timeout_ns, stream, kModeNv4, 0,
                              tensor_scale);
}

cudaError_t launch_quotient_selftest(int mode, unsigned long long* counts, cudaStream_t stream) {
  if (mode < 0 || mode > 2 || counts == nullptr) return cudaErrorInvalidValue;
  cudaError_t e = cudaMemsetAsync(counts, 0, 4 * sizeof(unsigned long long), stream);
  if (e != cudaSuccess) return e;
  // mode 0, 1: the fp16 scales 0x0400 .. 0x7BFF; mode 2: 126 codes x 512 g
  const unsigned blocks = mode == 2 ? 126u * 512u : 0x7C00u - 0x0400u;
  quotient_selftest_kernel<<<blocks, 256, 0, stream>>>(mode, counts);
  return cudaGetLastError();
}

}  // namespace w4a16
