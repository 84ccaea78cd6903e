// Arithmetic of the warp-MMA GEMM kernel for small M (gemv_rb.cu): the
// synchronous m16n8k16 MMA, the conversion of INT4 code words into MMA
// operands and the activation-type conversions.
//
// "Kernel dispatch and Humming quantization in PhyAI", section "Humming
// makes the separation useful": INT4 round-to-nearest codes, group 128 along
// K, BF16 or FP16 activations.  A stored nibble n is the 4-bit two's
// complement of the code q, so n ^ 8 = q + 8.  One shift and one AND-XOR
// turn nibbles s and s + 4 of a 32-bit code word into two 16-bit values
// x + q under the exponent whose unit is bit 0: 0x4300 | (n ^ 8) is
// 128 + q + 8, x = 136 for bf16, and x = 1032 for fp16 (0x6400 = 1024), both
// exact.  Products of these values (at most 11 significant bits) with an
// activation are exact in fp32; the kernels take x times the activation sum
// off each group's partial before its scale multiplies it, which leaves the
// sum of q times the activations.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "ptx.cuh"

namespace w4a16 {
namespace wmma16 {

// Activation value (bf16 or fp16 bits) as fp32.
template <bool F16>
__device__ __forceinline__ float act_to_f32(uint16_t b) {
  if constexpr (F16) {
    return __half2float(__ushort_as_half(b));
  } else {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
  }
}

// fp32 to the output type, rounded to nearest even once.
template <bool F16>
__device__ __forceinline__ uint16_t f32_to_out(float x) {
  if constexpr (F16) {
    return __half_as_ushort(__float2half_rn(x));
  } else {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
  }
}

__device__ __forceinline__ uint32_t lds_u16(uint32_t saddr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(saddr));
  return v;
}

// fp16 scale at a shared-memory address, as fp32.
__device__ __forceinline__ float lds_scale(uint32_t saddr) {
  return __half2float(__ushort_as_half(static_cast<uint16_t>(lds_u16(saddr))));
}

// D += A B for one m16n8k16 tile (A row-major 16 x 16, B column-major 16 x
// 8, fp32 accumulators), bf16 or fp16 operands.
template <bool F16>
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  if constexpr (F16) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

// Nibbles s and s + 4 of a code word as two 16-bit values x + q (low half:
// nibble s).
template <bool F16>
__device__ __forceinline__ uint32_t code_pair16(uint32_t w, int s) {
  return ptx::and_xor(w >> (4 * s), 0x000F000Fu, F16 ? 0x64086408u : 0x43084308u);
}

// The offset x the code values carry, and the all-ones operand.
template <bool F16>
struct CodeOffset {
  static constexpr float kOff = F16 ? 1032.0f : 136.0f;
  static constexpr uint32_t kOnes = F16 ? 0x3C003C00u : 0x3F803F80u;
};

}  // namespace wmma16
}  // namespace w4a16
