// Row-major packed INT4 codes -> the GEMM's tiled code storage (sm_103a).
//
// "Kernel dispatch and Humming quantization in PhyAI", section "Humming makes
// the separation useful": a packed INT4 layout is executed only by the kernel
// that understands it.  The plain interchange form of the codes is the
// row-major [N, K/2] byte array (byte j of row n: code of k = 2j in the low
// nibble, k = 2j + 1 in the high nibble, two's complement); this kernel
// moves those bytes into the library's 128 x 128 tiles (tile (n / 128,
// j / 64) at ((n / 128) * K/128 + j / 64) * 8192, row-major inside, 64 B per
// row), with zero rows past N.  A pure byte permutation: nothing is decoded.
//
// Work split: one thread per 16-byte chunk of the output, chunks in output
// order, so a warp writes 512 contiguous bytes and reads 64-byte runs of
// eight consecutive rows.  A grid-stride loop over a grid of a few waves.
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"

namespace w4a16 {

namespace {

__global__ void __launch_bounds__(256) repack_rowmajor_kernel(const uint4* __restrict__ src,
                                                              uint4* __restrict__ dst, int64_t N,
                                                              int64_t row_chunks, int64_t G,
                                                              int64_t total) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t o = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; o < total;
       o += stride) {
    // o = ((tn * G + g) * 128 + r) * 4 + c
    const int64_t c = o & 3;
    const int64_t r = (o >> 2) & 127;
    const int64_t tile = o >> 9;
    const int64_t tn = tile / G;
    const int64_t g = tile - tn * G;
    const int64_t n = tn * 128 + r;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (n < N) v = __ldg(src + n * row_chunks + g * 4 + c);
    dst[o] = v;
  }
}

}  // namespace

cudaError_t launch_repack_rowmajor(const void* rowmajor, int64_t N, int64_t K, void* tiled,
                                   int num_sms, cudaStream_t stream) {
  const int64_t G = K / kGroup;
  const int64_t tiles_n = (N + kTileW - 1) / kTileW;
  const int64_t total = tiles_n * G * kTileW * 4;   // 16-byte chunks of the output
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;   // 8 resident blocks of 256 per SM
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  repack_rowmajor_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      static_cast<const uint4*>(rowmajor), static_cast<uint4*>(tiled), N, K / 32, G, total);
  return cudaGetLastError();
}

}  // namespace w4a16
