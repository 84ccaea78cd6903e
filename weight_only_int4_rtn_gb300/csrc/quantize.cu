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
// Work split.  A tile is 64 consecutive rows x one group (64 x 256 B).  A
// producer thread streams tiles with 2-D TMA loads into a ring of shared-
// memory stages (up to 96 KiB in flight per CTA, two CTAs per SM); eight
// consumer warps quantize from shared memory.  One half-warp handles one
// (row, group): each lane reads 16 bytes (8 bf16) of the row's 256, the
// group absmax is a 4-step xor-shuffle max inside the half-warp, and each
// lane writes one 32-bit word of codes (64 contiguous bytes per group).
// Tiles are numbered row-block fastest, so a CTA's 64 scale stores of one
// group are contiguous, and its 64 rows of codes are one contiguous 4 KiB
// run of the tiled layout.  Rows past N arrive zero-filled; their (zero)
// codes are stored, their scales are not.
//
// Division.  The codes must equal rint(fl32(w / s)) bit for bit.  All 128
// elements of a group share s, so the kernel multiplies by r = fl32(1/s)
// (__frcp_rn) where that provably gives the same integer:
//  * Let w = X * 2^a (|X| < 2^8: w is bf16) and s = S * 2^b with a normal
//    fp16 significand 2^10 <= S < 2^11.  If w/s is not itself a half-integer
//    h, then |w/s - h| = |X 2^(a+1) - (2k+1) S 2^b| / (2 s) is either at
//    least 2^-12 (when a + 1 >= b) or |w/s| < 1/8 (when a + 1 < b).
//  * w/s = h exactly needs (2k+1) * (odd part of S) < 2^8, i.e. the odd
//    part of S below 2^8, i.e. S divisible by 8.
//  * |w/s| <= amax/s <= 7 / (1 - 2^-11) < 7.5 for a normal scale, so no
//    clamp is ever active, and |w*r - w/s| <= |w/s| 2^-24 < 2^-21.
// So for a normal scale whose significand is not a multiple of 8, w*r and
// fl32(w/s) lie strictly on the same side of every half-integer and round to
// the same integer; w*r + 1.5 * 2^23 (one fused multiply-add) rounds it, and
// the low 4 bits of that float are the two's-complement nibble.  Every
// other group (significand a multiple of 8, subnormal scale, or the zero
// rule) takes the IEEE division __fdiv_rn and the clamp element by element.
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

__device__ __forceinline__ void unpack_bf16x8(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// Codes of 8 elements from their exact fp32 quotients w / s: clamp, round to
// nearest even (fp32 addition of 1.5 * 2^23 rounds to an integer), keep the
// low nibble.
__device__ __forceinline__ uint32_t codes_exact(const float (&f)[8], float s) {
  uint32_t word = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float tc = fminf(fmaxf(__fdiv_rn(f[i], s), -8.0f), 7.0f);
    const float tm = tc + kRoundMagic;
    word |= (__float_as_uint(tm) & 0xFu) << (4 * i);
  }
  return word;
}

// Same codes through the reciprocal (valid when no tie and no clamp can occur;
// see the derivation at the top of this file).
__device__ __forceinline__ uint32_t codes_fast(const float (&f)[8], float r) {
  uint32_t word = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float tm = fmaf(f[i], r, kRoundMagic);
    word |= (__float_as_uint(tm) & 0xFu) << (4 * i);
  }
  return word;
}

constexpr int kQRows = 64;                  // rows per tile
constexpr int kQStages = 6;                 // shared-memory ring depth
constexpr int kQTileBytes = kQRows * 256;   // 64 rows x 128 bf16
constexpr int kQConsumerWarps = 8;
constexpr int kQThreads = 32 * (kQConsumerWarps + 1);

struct QShared {
  uint64_t full[kQStages];
  uint64_t empty[kQStages];
  int abort_flag;
};

__global__ void __launch_bounds__(kQThreads, 2)
    rtn_quantize_kernel(const __grid_constant__ CUtensorMap tm_w, int N, int K,
                        uint32_t* __restrict__ packed, __half* __restrict__ scales, int tiles,
                        int row_blocks, uint32_t* err, uint64_t timeout_ns) {
  extern __shared__ __align__(128) uint8_t q_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(q_smem_raw) + 127) &
                                             ~static_cast<uintptr_t>(127));
  QShared* sh = reinterpret_cast<QShared*>(smem + kQStages * kQTileBytes);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kQStages; ++s) {
      ptx::mbar_init(&sh->full[s], 1);
      ptx::mbar_init(&sh->empty[s], kQConsumerWarps);
    }
    sh->abort_flag = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tmap(&tm_w);
  }
  __syncthreads();
  const WaitCtx wc{err, timeout_ns, &sh->abort_flag};
  ptx::grid_dependency_wait();

  const int n_local = (tiles - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                      static_cast<int>(gridDim.x);

  if (warp == kQConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int issued = 0;
      for (int i = 0; i < n_local; ++i) {
        const int stage = i % kQStages;
        if (!wait_one(&sh->empty[stage], ((i / kQStages) & 1) ^ 1, wc)) break;
        const int t = static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x);
        const int g = t / row_blocks;
        const int rb = t - g * row_blocks;
        ptx::mbar_arrive_expect_tx(&sh->full[stage], kQTileBytes);
        ptx::tma_load_2d(smem + stage * kQTileBytes, &tm_w, &sh->full[stage], g * kGroup,
                         rb * kQRows);
        issued = i + 1;
      }
      if (*reinterpret_cast<volatile int*>(&sh->abort_flag)) {
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
  const int hw = warp * 2 + (lane >> 4);          // half-warp 0..15
  const int lane16 = lane & 15;
  const uint32_t half_mask = (lane & 16) ? 0xFFFF0000u : 0x0000FFFFu;
  const int n_groups = K / kGroup;
  for (int i = 0; i < n_local; ++i) {
    const int stage = i % kQStages;
    if (!wait_warp(&sh->full[stage], (i / kQStages) & 1, wc)) break;
    const int t = static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x);
    const int g = t / row_blocks;
    const int rb = t - g * row_blocks;
    const uint32_t tile = ptx::smem_u32(smem + stage * kQTileBytes);
#pragma unroll
    for (int j = 0; j < kQRows / 16; ++j) {
      const int r = hw + 16 * j;
      const uint4 v = ptx::lds128(tile + r * 256 + lane16 * 16);
      float f[8];
      unpack_bf16x8(v, f);
      float amax = 0.0f;
#pragma unroll
      for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(f[e]));
#pragma unroll
      for (int off = 8; off >= 1; off >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(half_mask, amax, off, 16));

      __half sh16 = __float2half_rn(__fdiv_rn(amax, 7.0f));
      if (__half_as_ushort(sh16) == 0) sh16 = __ushort_as_half(0x3C00);   // zero rule: 1.0
      const float s = __half2float(sh16);
      const uint32_t sbits = __half_as_ushort(sh16);
      const bool normal = (sbits & 0x7C00u) != 0;
      uint32_t word;
      if (normal && (sbits & 7u) != 0) {
        word = codes_fast(f, __frcp_rn(s));     // significand not a multiple of 8
      } else {
        word = codes_exact(f, s);
      }
      const int n = rb * kQRows + r;
      // tiled storage: ((tn * G + g) * 128 + n % 128) rows of 16 words
      packed[((static_cast<int64_t>(n >> 7) * n_groups + g) * 128 + (n & 127)) * 16 + lane16] = word;
      if (lane16 == 0 && n < N) scales[static_cast<int64_t>(g) * N + n] = sh16;
    }
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(&sh->empty[stage]);
  }
}

}  // namespace

cudaError_t launch_rtn_quantize(const void* W, int64_t N, int64_t K, void* packed, void* scales,
                                int num_sms, uint32_t* error_word, uint64_t timeout_ns,
                                cudaStream_t stream) {
  CUtensorMap tm_w;
  if (encode_tmap_2d(&tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, W, static_cast<uint64_t>(K),
                     static_cast<uint64_t>(N), static_cast<uint64_t>(K) * 2, kGroup, kQRows,
                     CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  // row blocks cover the rows padded to a multiple of 128 (tile height)
  const int row_blocks = static_cast<int>((N + 127) / 128) * (128 / kQRows);
  const int tiles = row_blocks * static_cast<int>(K / kGroup);
  constexpr size_t smem = static_cast<size_t>(kQStages) * kQTileBytes + sizeof(QShared) + 128;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static bool attr_set[64] = {};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(rtn_quantize_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  int grid = 2 * num_sms;
  if (grid > tiles) grid = tiles;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kQThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, rtn_quantize_kernel, tm_w, static_cast<int>(N),
                            static_cast<int>(K), static_cast<uint32_t*>(packed),
                            static_cast<__half*>(scales), tiles, row_blocks, error_word,
                            timeout_ns);
}

}  // namespace w4a16
