// RTN INT4 quantize/pack kernel, group 128 along K (sm_103a).
//
// "Kernel dispatch and Humming quantization in PhyAI", section "Humming makes
// the separation useful": round-to-nearest post-training quantization at
// load, INT4, group size 128.  Per row n and group g the kernel computes
//   amax = max |w|;  s = fp16_rn(amax / 7.0f) (1 if that is 0);
//   q = clamp(rint_even(fl32(w / s)), -8, 7)
// and stores two's-complement nibbles (low nibble = even k) and s.
//
// Work split: one half-warp per (n, g).  Each lane loads 16 bytes (8 bf16),
// so a half-warp reads the group's 256 contiguous bytes; the group absmax
// is a 4-step xor-shuffle max inside the half-warp.  Each lane writes one
// 32-bit word of codes (64 contiguous bytes per group).  Consecutive
// half-warps take consecutive rows of one group, so their scale stores are
// contiguous.
//
// Division.  The codes must equal rint(fl32(w / s)) bit for bit.  All 128
// elements of a group share s, so the kernel multiplies by r = fl32(1/s)
// (__frcp_rn) instead of dividing.  Error bound: with e = w/s exact,
// |fl(w*r) - e| <= |e| * 2^-23 (1 + 2^-24) and |fl32(e) - e| <= |e| * 2^-24;
// |e| < 16 for every element of every group (e <= 7 * (1 + 2^-11) for a
// normal scale, < 10.5 for a subnormal one, < 2^-22 when the zero rule
// applies), so fl(w*r) and fl32(e) differ by less than 2^-18.  Unless
// fl(w*r) lies within 2^-17 of a half-integer, both therefore round to the
// same integer.  A lane that sees such a near-tie redoes its 8 elements with
// the IEEE division __fdiv_rn, so the result is the one of the plain
// division for every input.  Rounding to an integer uses the exact
// round-to-nearest-even of fp32 addition: tc + 1.5 * 2^23 lands in
// [2^23, 2^24), where the fp32 spacing is 1; its low 4 bits are then the
// two's-complement nibble of the code.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"

namespace w4a16 {

namespace {

constexpr float kRoundMagic = 12582912.0f;        // 1.5 * 2^23
constexpr float kTieGuard = 0.5f - 7.62939453125e-06f;  // 0.5 - 2^-17

__device__ __forceinline__ uint4 load_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void unpack_bf16x8(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// Codes of 8 elements as packed nibbles, given the quotients t ~ w / s.
// Returns the largest |t_clamped - rint(t_clamped)| seen, for the tie check.
__device__ __forceinline__ uint32_t codes_from_quotients(const float (&t)[8], float& worst) {
  uint32_t word = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float tc = fminf(fmaxf(t[i], -8.0f), 7.0f);
    const float tm = tc + kRoundMagic;            // exact RNE to an integer
    const float d = (tm - kRoundMagic) - tc;      // exact
    worst = fmaxf(worst, fabsf(d));
    word |= (__float_as_uint(tm) & 0xFu) << (4 * i);
  }
  return word;
}

template <int ITEMS>
__global__ void __launch_bounds__(256) rtn_quantize_kernel(const uint4* __restrict__ W,
                                                           int64_t N, int64_t K,
                                                           uint32_t* __restrict__ packed,
                                                           __half* __restrict__ scales,
                                                           int64_t n_items) {
  const int lane16 = threadIdx.x & 15;
  const uint32_t half_mask = (threadIdx.x & 16) ? 0xFFFF0000u : 0x0000FFFFu;
  const int64_t hw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 4;
  const int64_t n_hw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 4;
  const int64_t row_u4 = K >> 3;     // uint4 per row of W
  const int64_t row_u32 = K >> 3;    // 32-bit words per row of packed (K/2 bytes)

  for (int64_t base = hw; base < n_items; base += n_hw * ITEMS) {
    uint4 v[ITEMS];
#pragma unroll
    for (int j = 0; j < ITEMS; ++j) {
      const int64_t item = base + j * n_hw;
      if (item < n_items) {
        const int64_t g = item / N;
        const int64_t n = item - g * N;
        v[j] = load_stream(W + n * row_u4 + g * 16 + lane16);
      }
    }
#pragma unroll
    for (int j = 0; j < ITEMS; ++j) {
      const int64_t item = base + j * n_hw;
      if (item >= n_items) break;   // uniform within the half-warp
      const int64_t g = item / N;
      const int64_t n = item - g * N;

      float f[8];
      unpack_bf16x8(v[j], f);
      float amax = 0.0f;
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
#pragma unroll
      for (int off = 8; off >= 1; off >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(half_mask, amax, off, 16));

      __half sh = __float2half_rn(__fdiv_rn(amax, 7.0f));
      if (__half_as_ushort(sh) == 0) sh = __ushort_as_half(0x3C00);   // zero rule: 1.0
      const float s = __half2float(sh);
      const float r = __frcp_rn(s);

      float t[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) t[i] = f[i] * r;
      float worst = 0.0f;
      uint32_t word = codes_from_quotients(t, worst);
      if (worst >= kTieGuard) {
        // near a half-integer: take the IEEE quotient itself
#pragma unroll
        for (int i = 0; i < 8; ++i) t[i] = __fdiv_rn(f[i], s);
        float unused = 0.0f;
        word = codes_from_quotients(t, unused);
      }
      packed[n * row_u32 + g * 16 + lane16] = word;
      if (lane16 == 0) scales[g * N + n] = sh;
    }
  }
}

}  // namespace

cudaError_t launch_rtn_quantize(const void* W, int64_t N, int64_t K, void* packed, void* scales,
                                int num_sms, cudaStream_t stream) {
  const int64_t n_items = N * (K / 128);
  constexpr int kItems = 2;
  constexpr int kThreads = 256;
  const int64_t half_warps_needed = (n_items + kItems - 1) / kItems;
  int64_t blocks = (half_warps_needed * 16 + kThreads - 1) / kThreads;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  rtn_quantize_kernel<kItems><<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(
      static_cast<const uint4*>(W), N, K, static_cast<uint32_t*>(packed),
      static_cast<__half*>(scales), n_items);
  return cudaGetLastError();
}

}  // namespace w4a16
