// W4A16 GEMM on the sm_103a tensor cores (tcgen05 + TMEM + TMA): the kernel
// template, instantiated for bf16 activations (gemm_tc.cu) and fp16
// activations (gemm_tc_f16.cu).
//
//   Y[M, N] = bf16( A[M, K] . dequant(W)[N, K]^T + bias[N] ),
//   dequant(W)[n, k] = q[n, k] * s[k / 128, n]
//
// "Kernel dispatch and Humming quantization in PhyAI", section "Humming
// makes the separation useful": INT4 group-128 weights execute through a
// kernel that understands their packed layout, with BF16 activations.
//
// Orientation ("swap AB").  One tile is 128 weight rows x act_tile activation
// rows.  The tcgen05 MMA computes D[128, act_tile] = Wt[128, 128k] .
// At[act_tile, 128k]^T per K block, so the accumulator D holds a tile of
// Y^T: TMEM lane i = weight row n0 + i, column j = activation row m0 + j.
//   * The weight operand is produced by the dequant warps and written into
//     TMEM with tcgen05.st (the MMA's A operand may live in TMEM): no shared
//     memory round trip for the converted weights.
//   * The activation operand is TMA-loaded into shared memory in the
//     128-byte-swizzled K-major layout and described by a shared-memory
//     descriptor (the MMA's B operand).
//   * Each K block (128 values = one quantization group) is one pipeline
//     unit: TMA brings the packed codes (one contiguous 8 KiB tile of the
//     tiled storage: 128 rows x 64 B), the 128 scales of that group and the
//     activation slice; the dequant warps convert; one thread issues 8 MMAs
//     of K = 16.  (Row-major codes would make every unit 128 separate 64-byte
//     pieces K/2 bytes apart, which TMA streams several times slower.)
//
// Two scaling modes:
//   group_scale = true:  the weight operand holds the integer codes (exact in
//     bf16); each unit's MMA result D_g is the integer-code partial sum of one
//     group, which the readout warps accumulate as acc += s[g, n] * D_g in
//     fp32 registers.  Cheapest conversion; used for small act_tile.
//   group_scale = false: the weight operand is bf16_rn(q * s), computed
//     exactly as fma(q, s_hi, q * s_lo) with s = s_hi + s_lo split into two
//     bf16 values; D accumulates the whole K range in TMEM.
//
// Schedule.  Units are (tile, k-block) pairs, tiles ordered weight-row-tile
// fastest.  Tiles 0 .. dp_tiles-1 run whole on CTA t % grid.  The units of
// the remaining tiles are split into contiguous, balanced ranges over all
// CTAs (stream-K).  A range that covers only part of a tile writes an fp32
// partial tile to the workspace.  When every CTA is done, one grid-wide
// barrier; then all CTAs together sum each split tile's partials in k order
// (deterministic), add the bias and store Y.  The grid is at most one CTA
// per SM and a CTA needs more than half an SM's shared memory, so all CTAs
// are resident at once and the barrier cannot wait on an unscheduled CTA.
//
// Lanes.  One thread issuing tcgen05.mma with a small N (16..64) is limited
// by its own issue rate (about 47 cycles per MMA), well below the tensor
// pipe; two issuing threads reach the pipe's rate.  So the group-scale
// variants run two lanes: even units and odd units each have their own
// producer, dequant warpgroup and MMA issuer, their own shared-memory stages,
// TMEM weight stages, accumulators and barrier rings; only the readout
// visits all units, in order.
//
// Warp roles (16 warps):
//   warps 0, 2  TMA producers (one lane each; even and odd units, because one
//               thread can only complete a few mbarrier phases per
//               microsecond, fewer than the weight stream needs)
//   warp 1      TMEM allocator; MMA issuer of lane 0 (of all units with one lane)
//   warp 15     MMA issuer of lane 1
//   warps 3-6   readout: accumulator -> registers -> Y or partial tile
//   warps 7-14  dequant, two warpgroups (even / odd units): packed codes
//               (shared memory) -> weight operand (TMEM)
// A warp may only touch TMEM lanes 32 * (warp % 4) .. + 31, so each readout
// and dequant thread owns weight row 32 * (warp % 4) + lane.  The dequant
// warps never wait on accumulators: they run up to the TMEM weight-stage
// count ahead of the MMA, which runs up to the accumulator count ahead of the
// readout.
//
// Every wait on an mbarrier is bounded by a time limit; on expiry the kernel
// records an error word, lets every role leave its loop, waits (bounded) for
// its own copies and MMAs in flight, frees TMEM and returns.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"
#include "waits.cuh"

namespace w4a16 {

#ifdef W4A16_TRACE
// Timestamp probes for profiling builds only (never in the default build).
static __device__ unsigned long long* g_trace = nullptr;
static __device__ unsigned long long* g_trace_units = nullptr;
#define W4A16_TRACE_POINT(id)                                                           \
  do {                                                                                  \
    if (trace_cta != nullptr) trace_cta[blockIdx.x * 16 + (id)] = ptx::globaltimer_ns(); \
  } while (0)
#define W4A16_TRACE_UNIT(role, i)                                                       \
  do {                                                                                  \
    if (trace_unit != nullptr && (i) < 64 && (role) < 32)                               \
      trace_unit[(role) * 64 + (i)] = static_cast<unsigned long long>(clock64());     \
  } while (0)
#else
#define W4A16_TRACE_POINT(id) \
  do {                        \
  } while (0)
#define W4A16_TRACE_UNIT(role, i) \
  do {                            \
  } while (0)
#endif

namespace {

constexpr int kUnitK = 128;                    // K values per unit (one group)
// Weight formats (kernels.h): INT4 or INT8 codes with one fp16 scale per
// row and group; E2M1 codes (INT4 layout) with one E8M0 byte per 32 values
// (MXFP4) or one E4M3 byte per 16 values (NVFP4).
constexpr int wf_bits(int wf) { return wf == kFmtInt8 ? 8 : 4; }
constexpr bool wf_fp4(int wf) { return wf == kFmtMxfp4 || wf == kFmtNvfp4; }
constexpr int wf_blocks(int wf) { return wf == kFmtMxfp4 ? 4 : wf == kFmtNvfp4 ? 8 : 1; }
// code bytes of one group of a tile: 8 KiB (4-bit codes) or 16 KiB (INT8)
constexpr int w_group_bytes(int wf) { return kTileW * kUnitK * wf_bits(wf) / 8; }
// scale bytes of one group of a tile: 256 B of fp16, or the block-scale bytes
constexpr int w_scale_bytes(int wf) { return wf_fp4(wf) ? kTileW * wf_blocks(wf) : kTileW * 2; }
constexpr int kMaxAStages = 6;                 // weight-operand stages in TMEM (at most)
constexpr int kAStageCols = kUnitK / 2;        // 64 TMEM columns per stage
constexpr uint32_t kTmemCols = 512;
constexpr int kWarps = 16;
constexpr int kReadoutWarp0 = 3;
constexpr int kDequantWarp0 = 7;
constexpr int kMmaWarp2 = 15;                  // second MMA issuer (two lanes)
constexpr int kScaleRing = 8;                  // group mode: units of scales in shared memory
constexpr int kScaleAhead = 2;                 // ... copied this many unit pairs ahead
constexpr int kPairRing = 8;                   // group mode: pair_done barriers

struct Args {
  int M, N, K, KB;
  int n_tiles;
  int dp_tiles;
  int sk_units;
  int act_3d;                  // activation map is 3-D: both 64-k halves in one copy
  int csk;                     // cluster split-K: each tile's K range split over the
                               // csk CTAs of one thread-block cluster (0: off)
  int sw;                      // this problem takes the SwiGLU epilogue (read by the
                               // instances compiled with it only)
  int prefetch_w;              // weights are not written by the previous kernel on
                               // the stream: the codes and scales of this many
                               // first units go out before the dependency wait
  int tail_tile0;              // dequant mode: tiles from this one on are the last
                               // activation tile, whose MMAs run tail_n columns
                               // (M rounded up to 16 there) instead of BA
  int tail_n;
  const __half* scales;        // [K/128, N]; the group-mode readout reads its scales here
  const float* out_scale;      // NVFP4: the tensor scale g, applied to the fp32 sums
  const uint16_t* bias;        // [N] activation type (bf16 or fp16 bits)
  uint16_t* Y;                 // [M, N] activation type
  float* ws;
  uint32_t* counters;
  uint32_t* err;
  uint64_t timeout_ns;
};

// A launch runs up to kMaxGroup independent problems: problem p owns the
// CTAs cta_start[p] .. cta_start[p+1]-1 (its "sub-grid") and runs the
// single-problem schedule on them, with its own TMA descriptors, arguments
// and workspace.  A single GEMM is a group of one.
// The arguments are sized for G problems (kernel parameters are copied at
// every launch, so a single GEMM uses G = 1).
constexpr int kMaxGroup = 8;
template <int G>
struct GroupArgs {
  CUtensorMap tm[G][3];   // per problem: activations, codes, scales
  Args a[G];
  int cta_start[G + 1];
  int count;
};

struct Unit {
  int tile, kb;
  bool seg_first, seg_last;   // first / last unit of this CTA's run on the tile
  bool whole;                 // the run covers the whole tile
  int slot;                   // partial slot (0: first stream-K tile of the CTA, 1: last)
  int sk_tile;                // index among stream-K tiles, -1 for whole tiles
};

struct Sched {
  int c, C, KB, dp_tiles, dp_iters;
  int u0, u1;                 // this CTA's stream-K unit range [u0, u1)
  int total;

  __device__ void init(const Args& a, int cta, int ctas) {
    c = cta;
    C = ctas;
    KB = a.KB;
    dp_tiles = a.dp_tiles;
    if (a.csk > 1) {
      // cluster split-K: cluster cta / csk owns tile cta / csk; its CTA of
      // rank r runs that tile's units [r KB / csk, (r + 1) KB / csk)
      const int t = cta / a.csk, r = cta - t * a.csk;
      dp_tiles = 0;
      dp_iters = 0;
      u0 = t * KB + (r * KB) / a.csk;
      u1 = t * KB + ((r + 1) * KB) / a.csk;
      total = u1 - u0;
      return;
    }
    dp_iters = (dp_tiles > c) ? (dp_tiles - c + C - 1) / C : 0;
    u0 = static_cast<int>((static_cast<int64_t>(c) * a.sk_units) / C);
    u1 = static_cast<int>((static_cast<int64_t>(c + 1) * a.sk_units) / C);
    total = dp_iters * KB + (u1 - u0);
  }
};

// Walks this CTA's units in order, one at a time, with no division per unit
// (the issuing threads are on the critical path of the pipeline).
struct UnitIter {
  int C, KB, ndp, u0, u1, dp_tiles;
  int i, tile, kb, u, tl, first_tl;

  __device__ void init(const Sched& s) {
    C = s.C;
    KB = s.KB;
    ndp = s.dp_iters * s.KB;
    u0 = s.u0;
    u1 = s.u1;
    dp_tiles = s.dp_tiles;
    i = 0;
    tile = s.c;
    kb = 0;
    if (ndp == 0) start_sk();
  }
  __device__ void start_sk() {
    u = u0;
    tl = u0 / KB;
    first_tl = tl;
    kb = u0 - tl * KB;
    tile = dp_tiles + tl;
  }
  __device__ Unit next() {
    Unit r;
    r.tile = tile;
    r.kb = kb;
    if (i < ndp) {
      r.seg_first = (kb == 0);
      r.seg_last = (kb == KB - 1);
      r.whole = true;
      r.slot = 0;
      r.sk_tile = -1;
      ++i;
      if (++kb == KB) {
        kb = 0;
        tile += C;
      }
      if (i == ndp) start_sk();
    } else {
      r.seg_first = (kb == 0) || (u == u0);
      r.seg_last = (kb == KB - 1) || (u == u1 - 1);
      r.whole = (tl * KB >= u0) && ((tl + 1) * KB <= u1);
      r.slot = (tl == first_tl) ? 0 : 1;
      r.sk_tile = tl;
      ++i;
      ++u;
      if (++kb == KB) {
        kb = 0;
        ++tl;
        ++tile;
      }
    }
    return r;
  }
};

// Walks this CTA's runs ("segments": consecutive units on one tile) in
// order.  For the readout, which needs tile-level facts only at the ends of
// runs.
struct SegCursor {
  int C, KB, dp_left, tile, u, u1, first_sk;
  __device__ void init(const Sched& s) {
    C = s.C;
    KB = s.KB;
    dp_left = s.dp_iters;
    tile = s.c;
    u = s.u0;
    u1 = s.u1;
    first_sk = 1;
  }
  // Next run: its tile, first k-block, length, and whether it is the whole
  // tile (else: the partial slot it writes).
  __device__ void next(Unit& r, int& kb0, int& len, int dp_tiles) {
    if (dp_left > 0) {
      --dp_left;
      r.tile = tile;
      tile += C;
      kb0 = 0;
      len = KB;
      r.whole = true;
      r.slot = 0;
      r.sk_tile = -1;
    } else {
      const int tl = u / KB;
      kb0 = u - tl * KB;
      const int end = min(u1, (tl + 1) * KB);
      len = end - u;
      r.tile = dp_tiles + tl;
      r.whole = (kb0 == 0) && (len == KB);
      r.slot = first_sk ? 0 : 1;
      r.sk_tile = tl;
      first_sk = 0;
      u = end;
    }
    r.kb = kb0;
    r.seg_first = true;
    r.seg_last = true;
  }
};

// CTA that owns stream-K unit u under the balanced split.
__device__ __forceinline__ int sk_owner(int u, int C, int sk_units) {
  return static_cast<int>(((static_cast<int64_t>(u) + 1) * C - 1) / sk_units);
}

struct Shared {
  uint64_t full[16];          // a shared-memory stage's copies landed (split
                              // rings: the activation stage's)
  uint64_t wfull[16];         // split rings: a code stage's copies landed
  uint64_t wempty[16];        // split rings: the dequant read a code stage
  uint64_t afull[kMaxAStages];   // a TMEM weight stage is written (it is free
                                 // again when its unit's MMAs completed)
  uint64_t unit_done[32];     // per lane a ring: a unit's MMAs completed
  uint64_t dfull[8];          // dequant mode: a run on a tile is accumulated
  uint64_t dempty[8];         // the readout drained an accumulator buffer
                              // (group mode: buffer dl of lane p at p * DL + dl)
  uint64_t pair_done[8];       // group mode: both lanes' units of a pair completed
  uint64_t mma_done[2];
  uint64_t rsync;             // readout warps' barrier (split-tile fixup)
  uint32_t tmem_base;
  int abort_flag;
  int fixup_last;             // this CTA completed a split tile's count
  int fixup_defer;            // ... on its last run: the whole CTA sums it at exit
  int fix_tile, fix_clo, fix_chi, fix_slot;   // that tile and its contributors
};

// ------------------------------------------------ activation-type helpers
// The activations (and Y, bias) are bf16 or fp16; the weight operand takes
// the same type (one tcgen05.mma kind::f16 reads both operands in one type).
template <bool F16>
__device__ __forceinline__ float act_to_float(uint16_t b) {
  if constexpr (F16) {
    return __half2float(__ushort_as_half(b));
  } else {
    return __bfloat162float(__ushort_as_bfloat16(b));
  }
}
template <bool F16>
__device__ __forceinline__ uint16_t act_from_float(float x) {
  if constexpr (F16) {
    return __half_as_ushort(__float2half_rn(x));
  } else {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
  }
}

// Packed fused multiply-add of two 16-bit values per word.
template <bool F16>
__device__ __forceinline__ uint32_t x2_fma(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  if constexpr (F16) {
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  } else {
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  }
  return d;
}

// ------------------------------------------------- codes -> operand pairs
// Eight 4-bit codes (one 32-bit word, code k in nibble k) to four words of
// two 16-bit values holding the code pairs (k0,k1), (k2,k3), (k4,k5), (k6,k7)
// as exact integers.  bf16: 0x4300 | (nibble ^ 8) is the value 136 + q;
// fp16: 0x6400 | (nibble ^ 8) is 1032 + q; one fused multiply-add removes
// the offset.
template <bool F16>
__device__ __forceinline__ void codes_to_operand(uint32_t w, uint32_t* out) {
  const uint32_t v = w >> 4;
  constexpr uint32_t one = F16 ? 0x3C003C00u : 0x3F803F80u;     // (1, 1)
  constexpr uint32_t off = F16 ? 0xE408E408u : 0xC308C308u;     // (-1032, -1032) / (-136, -136)
  constexpr uint32_t magic = F16 ? 0x64086408u : 0x43084308u;
  out[0] = x2_fma<F16>(ptx::and_xor(ptx::prmt(w, v, 0x0400), 0x000F000Fu, magic), one, off);
  out[1] = x2_fma<F16>(ptx::and_xor(ptx::prmt(w, v, 0x0501), 0x000F000Fu, magic), one, off);
  out[2] = x2_fma<F16>(ptx::and_xor(ptx::prmt(w, v, 0x0602), 0x000F000Fu, magic), one, off);
  out[3] = x2_fma<F16>(ptx::and_xor(ptx::prmt(w, v, 0x0703), 0x000F000Fu, magic), one, off);
}

// Four 8-bit codes (one word, code k in byte k, two's complement) to two
// words of bf16 pairs (k0, k1), (k2, k3), exact: with q = 16 hi + lo (hi the
// signed high nibble, lo the unsigned low nibble), one byte permute puts each
// nibble under the exponent byte 0x43 (bf16 128 + nibble; the high nibble in
// offset binary: 136 + hi), then t = 16 X_hi - 2304 = 16 hi - 128 and q =
// X_lo + t, both exact (every value is a small integer).
__device__ __forceinline__ void bytes_to_operand_bf16(uint32_t w, uint32_t* out) {
  const uint32_t lo = w & 0x0F0F0F0Fu;
  const uint32_t hi = ((w >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u;
  constexpr uint32_t kExp = 0x43434343u;
  constexpr uint32_t k16 = 0x41804180u;        // (16, 16)
  constexpr uint32_t kOff = 0xC510C510u;       // (-2304, -2304)
  constexpr uint32_t kOne = 0x3F803F80u;       // (1, 1)
  const uint32_t xl0 = ptx::prmt(lo, kExp, 0x4140), xl1 = ptx::prmt(lo, kExp, 0x4342);
  const uint32_t xh0 = ptx::prmt(hi, kExp, 0x4140), xh1 = ptx::prmt(hi, kExp, 0x4342);
  out[0] = x2_fma<false>(xl0, kOne, x2_fma<false>(xh0, k16, kOff));
  out[1] = x2_fma<false>(xl1, kOne, x2_fma<false>(xh1, k16, kOff));
}

// bf16_rn(q * s) for an exact pair of codes (INT8): q * s is exact in fp32
// (8- and 11-bit significands), then one rounding to bf16.
__device__ __forceinline__ uint32_t scale_pair_bf16_f32(uint32_t q2, float s) {
  const float a = __uint_as_float(q2 << 16) * s;
  const float b = __uint_as_float(q2 & 0xFFFF0000u) * s;
  const __nv_bfloat162 r = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&r);
}

// bf16_rn(q * s) for both halves: q * s_lo is exact (<= 7 significant bits),
// so fma(q, s_hi, q * s_lo) rounds the exact product once.
__device__ __forceinline__ uint32_t scale_pair_bf16(uint32_t q, uint32_t s_hi2, uint32_t s_lo2) {
  const uint32_t lo = x2_fma<false>(q, s_lo2, 0x80008000u);   // q * s_lo + (-0)
  return x2_fma<false>(q, s_hi2, lo);
}

// FP4 (E2M1) codes to bf16 operand pairs, scaled: eight codes (one word,
// code k in nibble k; sign bit 3, magnitude index bits 0..2) to four words
// (k0,k1) .. (k6,k7) of bf16 e2m1(c) * s.  One byte permute looks up
// m = 2 |e2m1| (0, 1, 2, 3, 4, 6, 8, 12) for four magnitude indices; with the
// exponent byte 0x43 above it a bf16 holds 128 + m, and one fused
// multiply-add with h = s / 2 and off = -128 h leaves m h = |e2m1| s,
// rounded once (exact whenever the product fits bf16).  The sign bits are
// replicated into place by a sign-extending byte permute: nibble 2 i's sign
// is the top bit of byte i of w << 4, nibble 2 i + 1's of byte i of w.
__device__ __forceinline__ void e2m1_to_operand(uint32_t w, uint32_t h2, uint32_t off2,
                                                uint32_t* out) {
  constexpr uint32_t kLo = 0x03020100u;     // m for indices 0..3
  constexpr uint32_t kHi = 0x0C080604u;     // m for indices 4..7
  constexpr uint32_t kExp = 0x43434343u;
  const uint32_t sel = w & 0x77777777u;
  const uint32_t m0 = ptx::prmt(kLo, kHi, sel);          // m of codes 0..3
  const uint32_t m1 = ptx::prmt(kLo, kHi, sel >> 16);    // m of codes 4..7
  const uint32_t w4 = w << 4;
  out[0] = x2_fma<false>(ptx::prmt(m0, kExp, 0x4140), h2, off2) |
           (ptx::prmt(w4, w, 0xC080) & 0x80008000u);
  out[1] = x2_fma<false>(ptx::prmt(m0, kExp, 0x4342), h2, off2) |
           (ptx::prmt(w4, w, 0xD090) & 0x80008000u);
  out[2] = x2_fma<false>(ptx::prmt(m1, kExp, 0x4140), h2, off2) |
           (ptx::prmt(w4, w, 0xE0A0) & 0x80008000u);
  out[3] = x2_fma<false>(ptx::prmt(m1, kExp, 0x4342), h2, off2) |
           (ptx::prmt(w4, w, 0xF0B0) & 0x80008000u);
}

// MXFP4 block scale (E8M0 code E: 2^(E - 127)) as the pair h = 2^(E - 128),
// off = -128 h = -2^(E - 121) in bf16 (both halves).  h is subnormal for
// E <= 1; off overflows for E > 248 (blocks with |w| >= 2^123, outside the
// GEMM's range).
__device__ __forceinline__ void mx_half_scale(uint32_t e, uint32_t& h2, uint32_t& off2) {
  const uint32_t h = e >= 2u ? (e - 1u) << 7 : 0x40u >> (1u - e);
  const uint32_t off = 0x8000u | ((e + 6u) << 7);
  h2 = h | (h << 16);
  off2 = off | (off << 16);
}

// NVFP4 block scale (E4M3 code: bias 7, three mantissa bits) as h = s / 2,
// off = -64 s in bf16; both exact (s has 4 significant bits, 2^-9 <= s <=
// 448 or s = 0).
__device__ __forceinline__ void nv_half_scale(uint32_t code, uint32_t& h2, uint32_t& off2) {
  const float s = __uint_as_float((code & 0x7Fu) << 20) * 0x1p120f;   // exact E4M3 value
  const __nv_bfloat162 hv = __float2bfloat162_rn(s * 0.5f);
  const __nv_bfloat162 ov = __float2bfloat162_rn(s * -64.0f);
  h2 = *reinterpret_cast<const uint32_t*>(&hv);
  off2 = *reinterpret_cast<const uint32_t*>(&ov);
}

template <int BA, int L, bool GRP, int STAGES, int UG, int WF = kFmtInt4>
struct Cfg {
  static constexpr int kWB = w_group_bytes(WF);                 // code bytes per group
  static constexpr int kSB = w_scale_bytes(WF);                 // scale bytes per group
  // A shared-memory stage holds one unit of UG groups: 2 * UG activation
  // boxes (64 k each), then UG code tiles (8 KiB each), then UG scale rows.
  static constexpr int kActBox = BA * 128;                        // bytes per 64-k box
  static constexpr int kWOff = 2 * UG * kActBox;
  static constexpr int kSOff = kWOff + UG * kWB;
  static constexpr int kStageRaw = UG * (2 * kActBox + kWB + kSB);
  static constexpr int kStage = (kStageRaw + 1023) / 1024 * 1024;
  // STAGES >= 32 (dequant mode, one lane, INT8): split rings.  The codes and
  // scales take a ring of their own, STAGES / 32 stages deep, released as
  // soon as the dequant has read a unit's codes, and the activations one of
  // STAGES % 32 stages, released by the unit's MMAs: where the combined
  // stages are few (8-bit codes beside a 256-wide activation tile), the
  // dequant runs further ahead of the MMAs.
  static constexpr int kCodeStages = STAGES / 32;
  static constexpr bool kSplit = kCodeStages > 0;
  static constexpr int kActStages = STAGES % 32;
  static constexpr int kActStage = (2 * UG * kActBox + 1023) / 1024 * 1024;
  static constexpr int kCodeStage = (UG * (kWB + kSB) + 1023) / 1024 * 1024;
  static constexpr int kActStride = kSplit ? kActStage : kStage;  // act stage to stage
  static constexpr int kWStride = kSplit ? kCodeStage : kStage;   // code stage to stage
  static constexpr int kWBase = kSplit ? kActStages * kActStage : kWOff;   // code stage 0
  static constexpr int kSRel = kSplit ? UG * kWB : kSOff - kWOff;  // scales after the codes
  static constexpr int kRing = kSplit ? kActStages * kActStage + kCodeStages * kCodeStage
                                      : STAGES * kStage;
  static constexpr uint32_t kTxAct = 2 * UG * kActBox;
  static constexpr uint32_t kTxCode = UG * (kWB + kSB);
  static constexpr int kThreads = 32 * kWarps;                    // 16 warps: <= 128 registers
  static constexpr int kSL = kActStages / L;                      // shared-memory stages per lane
  // TMEM: kAS weight stages of 64 columns, then the accumulators.  The
  // narrowest group-mode tile needs few accumulator columns, so it takes
  // three weight stages per lane (the dequant runs further ahead).
  static constexpr int kAS = (BA == 16 && (GRP || UG == 2)) ? 6 : 4;
  static constexpr int kDCol = kAS * kAStageCols;
  static constexpr int kDCols = 512 - kDCol;
  static constexpr int kAL = kAS / L;                             // TMEM weight stages per lane
  // Group mode: kDB accumulators of BA columns, split over the lanes (kDL
  // per lane).  Dequant mode: kDB run buffers of L * BA columns (one BA-wide
  // half per lane; the readout adds the halves).
  static constexpr int kBufCols = GRP ? UG * BA : L * BA;
  static constexpr int kDBfit = kDCols / kBufCols;                // buffers that fit
  static constexpr int kDB = kDBfit < (GRP ? 8 : 4) ? kDBfit : (GRP ? 8 : 4);
  static constexpr int kDL = GRP ? kDB / L : kDB;                 // buffers a lane cycles through
  static constexpr int kRL = kSL > kAL ? kSL : kAL;               // unit_done ring per lane
  static constexpr int kChunk = BA < (GRP ? 16 : 32) ? BA : (GRP ? 16 : 32);
  static constexpr size_t kSmem = static_cast<size_t>(kRing) + 1024 + sizeof(Shared) +
                                  (GRP ? kScaleRing * UG * kTileW * 2 : 0);
  static constexpr uint32_t kTx = kStageRaw;
  static_assert(BA % 16 == 0 && BA >= 16 && BA <= 256, "tcgen05 N for M=128");
  static_assert(L == 1 || L == 2, "lanes");
  static_assert(UG == 1 || UG == 2, "groups per unit (TMA boxes of up to 256 rows)");
  static_assert(WF == kFmtInt4 || WF == kFmtInt8 || wf_fp4(WF), "weight format");
  static_assert(!wf_fp4(WF) || !GRP, "FP4 weights run in dequant mode (block scales inside a group)");
  static_assert(kAS % L == 0 && kAS <= kMaxAStages, "TMEM weight stages split over the lanes");
  static_assert(kActStages % L == 0 && kActStages >= 1 && kActStages <= 16, "stages split over the lanes");
  static_assert(!kSplit || (!GRP && L == 1 && WF == kFmtInt8 && kCodeStages % 2 == 0 &&
                            kCodeStages <= 16),
                "split rings: dequant mode, one lane, INT8, an even code ring (the two dequant "
                "warpgroups alternate units)");
  static_assert(kDB >= 1 && kDL >= 1 && (!GRP || kDB % L == 0), "accumulators split over the lanes");
  static_assert(kDB <= 8, "barrier arrays");
  static_assert(L * kRL <= 32, "barrier arrays");
  static_assert(!GRP || BA <= 64, "group mode keeps BA fp32 accumulators per thread");
  static_assert(BA * kTileW * 4 <= kRing, "cluster split-K partial fits the stages");
  static_assert(!GRP || L == 2, "group mode runs two lanes (the readout takes units in pairs)");
  // group mode: the pair ring replaces the unit ring for every waiter, so
  // it must be as deep as the stage rings and the accumulator buffers
  static_assert(!GRP || (kDL <= kPairRing && kSL <= kPairRing && kAL <= kPairRing),
                "pair ring covers the stage rings and the accumulator buffers");
};

// Lane of unit i and its index within the lane.
template <int L>
__device__ __forceinline__ void lane_split(int i, int& p, int& j) {
  if constexpr (L == 1) {
    p = 0;
    j = i;
  } else {
    p = i & 1;
    j = i >> 1;
  }
}

template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t* r) {
  if constexpr (N == 8) {
    ptx::tmem_ld_x8_sync(taddr, r);
  } else if constexpr (N == 16) {
    ptx::tmem_ld_x16_sync(taddr, r);
  } else {
    static_assert(N == 32, "chunk");
    ptx::tmem_ld_x32_sync(taddr, r);
  }
}

template <int CNT>
__device__ __forceinline__ void load_cols(uint32_t taddr, float (&v)[CNT]) {
  uint32_t r[CNT];
  tmem_ld_cols<CNT>(taddr, r);
#pragma unroll
  for (int j = 0; j < CNT; ++j) v[j] = __uint_as_float(r[j]);
}

// SwiGLU epilogue.  Weight rows 2f (up) and 2f + 1 (gate) are held by
// adjacent lanes (a thread's weight row is its lane plus a multiple of 32).
// swiglu_vals turns K final fp32 values y (bias added) of this lane's row into
// silu(gate) * up = gate / (1 + e^-gate) * up with the neighbouring lane's
// values as gate (meaningful on the lanes of even rows, which store them at
// Y[m, f] of the [M, N/2] output), in fp32: the exponential and quotient by
// the fast intrinsics, whose relative error, near 2^-21, is far below the
// output's rounding.  All shuffles of a batch come before its arithmetic and
// its stores, so the K chains overlap.  Every lane of the warp calls it.  The
// epilogue is a template parameter (SW) of the kernel: the plain instances
// compile none of it, so their code (and its instruction-cache footprint) is
// unchanged.
template <int K>
__device__ __forceinline__ void swiglu_vals(float (&h)[K]) {
  float g[K];
#pragma unroll
  for (int i = 0; i < K; ++i) g[i] = __shfl_xor_sync(0xFFFFFFFFu, h[i], 1);
#pragma unroll
  for (int i = 0; i < K; ++i) h[i] = __fdividef(g[i], 1.0f + __expf(-g[i])) * h[i];
}

// Write accumulator columns [col0, col0 + CNT) of this thread's weight row
// either to Y (whole tile: bias added, one rounding to the output type; or
// the SwiGLU epilogue, swiglu_vals) or to this CTA's partial slot (fp32, no
// bias; column m of the slot holds 128 rows).  Called by whole warps.
// Cluster split-K: the CTA's partial tile, [BA][128] fp32 at the start of
// the (by then drained) shared-memory stages.
__device__ __forceinline__ float* csk_partial(uint8_t* smem) { return reinterpret_cast<float*>(smem); }

template <int BA, int CNT, bool F16, bool SW>
__device__ __forceinline__ void emit_cols(const Args& a, const Unit& u, int row, int col0,
                                          const float (&v)[CNT], float bias_n, int cta,
                                          float* sp) {
  const int n0 = (u.tile % a.n_tiles) * kTileW;
  const int m0 = (u.tile / a.n_tiles) * BA;
  if (u.whole) {
    const int n = n0 + row;
    if (SW && a.sw) {
      constexpr int kB = CNT < 8 ? CNT : 8;
#pragma unroll
      for (int j0 = 0; j0 < CNT; j0 += kB) {
        float h[kB];
#pragma unroll
        for (int i = 0; i < kB; ++i) h[i] = v[j0 + i] + bias_n;
        swiglu_vals(h);
        if (n < a.N && (n & 1) == 0) {
#pragma unroll
          for (int i = 0; i < kB; ++i) {
            const int m = m0 + col0 + j0 + i;
            if (m < a.M) a.Y[static_cast<int64_t>(m) * (a.N >> 1) + (n >> 1)] = act_from_float<F16>(h[i]);
          }
        }
      }
    } else if (n < a.N) {
#pragma unroll
      for (int j = 0; j < CNT; ++j) {
        const int m = m0 + col0 + j;
        if (m < a.M) a.Y[static_cast<int64_t>(m) * a.N + n] = act_from_float<F16>(v[j] + bias_n);
      }
    }
  } else if (a.csk > 1) {
    // the run's partial stays in this CTA's shared memory; the cluster sums
    // the partials of the tile at exit
#pragma unroll
    for (int j = 0; j < CNT; ++j) sp[(col0 + j) * kTileW + row] = v[j];
  } else {
    float* slot = a.ws + (static_cast<int64_t>(cta) * 2 + u.slot) * (BA * kTileW) + row;
#pragma unroll
    for (int j = 0; j < CNT; ++j) {
      if (m0 + col0 + j < a.M) slot[(col0 + j) * kTileW] = v[j];
    }
  }
}

// A split tile's contributors: CTAs c_lo .. c_hi (in k order) of the
// balanced stream-K split; CTA c_lo keeps the tile in slot 0 only if its
// range starts exactly at the tile's first k-block, every later contributor's
// range starts inside the tile (slot 0).
struct SplitInfo {
  int c_lo, c_hi, slot_lo;
};

__device__ __forceinline__ SplitInfo split_info(const Args& a, int tl, int ctas) {
  SplitInfo r;
  const int S = a.sk_units;
  const int KB = a.KB;
  r.c_lo = sk_owner(tl * KB, ctas, S);
  r.c_hi = sk_owner(tl * KB + KB - 1, ctas, S);
  const int u0_lo = static_cast<int>((static_cast<int64_t>(r.c_lo) * S) / ctas);
  r.slot_lo = (u0_lo == tl * KB) ? 0 : 1;
  return r;
}

// Barrier of the four readout warps on an mbarrier, so that a warp that gave
// up after a timeout cannot leave the others blocked for good.
__device__ __forceinline__ bool readout_sync(Shared* sh, uint32_t& nsync, const WaitCtx& wc) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) ptx::mbar_arrive(&sh->rsync);
  const bool ok = wait_warp(&sh->rsync, nsync & 1, wc);
  ++nsync;
  return ok;
}

// After this CTA wrote its partial of a split tile (every readout thread its
// weight row): count the arrival on the tile's counter.  The contributor
// that completes the count sums all partials of the tile in k order (so the
// result does not depend on who arrives last), adds the bias, rounds once to
// the output type and stores Y; it also resets the counter for the next
// launch.  Nobody waits for anybody: the last arrival finds every partial
// written.  On the CTA's last run (`defer`) the sum is left to wide_fixup,
// which all the CTA's warps run once their roles are done: the last arrival
// is most often a contributor finishing its last run, and the sum's time is
// the latency of loads that four warps alone keep too few of in flight.  (A
// sum in the middle of a run stays with the readout warps, where it overlaps
// the CTA's remaining units.)
template <int BA, bool F16, bool SW>
__device__ bool split_fixup(const Args& a, const Unit& u, const SplitInfo& si, Shared* sh, int row,
                            float bias_n, uint32_t& nsync, const WaitCtx& wc, bool defer) {
  __threadfence();   // this thread's partial row is visible to the whole GPU
  if (!readout_sync(sh, nsync, wc)) return false;
  if (threadIdx.x == 32 * kReadoutWarp0) {
    uint32_t* cnt = a.counters + u.sk_tile;
    // acquire-release: the last arrival observes every contributor's partial
    const uint32_t old = ptx::atom_add_acq_rel_gpu(cnt, 1u);
    const bool last = old == static_cast<uint32_t>(si.c_hi - si.c_lo);
    if (last) atomicExch(cnt, 0u);
    sh->fixup_last = last && !defer ? 1 : 0;
    if (last && defer) {
      sh->fix_tile = u.tile;
      sh->fix_clo = si.c_lo;
      sh->fix_chi = si.c_hi;
      sh->fix_slot = si.slot_lo;
      sh->fixup_defer = 1;
    }
  }
  if (!readout_sync(sh, nsync, wc)) return false;
  if (!sh->fixup_last) return true;
  __threadfence();
  const int n0 = (u.tile % a.n_tiles) * kTileW;
  const int m0 = (u.tile / a.n_tiles) * BA;
  const int n = n0 + row;
  const int mcols = min(BA, a.M - m0);
  constexpr int64_t kSlot = static_cast<int64_t>(BA) * kTileW;
  const float* lo = a.ws + (static_cast<int64_t>(si.c_lo) * 2 + si.slot_lo) * kSlot + row;
#pragma unroll 1
  for (int c0 = 0; c0 < mcols; c0 += 16) {
    float acc[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) acc[j] = __ldcg(lo + (c0 + j) * kTileW);
#pragma unroll 2
    for (int c = si.c_lo + 1; c <= si.c_hi; ++c) {
      const float* src = a.ws + static_cast<int64_t>(c) * 2 * kSlot + row;
#pragma unroll
      for (int j = 0; j < 16; ++j) acc[j] += __ldcg(src + (c0 + j) * kTileW);
    }
    if (SW && a.sw) {
#pragma unroll
      for (int j0 = 0; j0 < 16; j0 += 8) {
        float h[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) h[i] = acc[j0 + i] + bias_n;
        swiglu_vals(h);
        if (n < a.N && (n & 1) == 0) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if (c0 + j0 + i < mcols)
              a.Y[static_cast<int64_t>(m0 + c0 + j0 + i) * (a.N >> 1) + (n >> 1)] =
                  act_from_float<F16>(h[i]);
          }
        }
      }
    } else if (n < a.N) {
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        if (c0 + j < mcols)
          a.Y[static_cast<int64_t>(m0 + c0 + j) * a.N + n] = act_from_float<F16>(acc[j] + bias_n);
      }
    }
  }
  return true;
}

// The deferred sum of split_fixup, by every thread of the CTA after the
// teardown barrier: thread t takes weight row t % 128 and the columns
// t / 128 + P j (P = threads / 128) that hold activation rows, adding the
// contributors' partials in the same k order as split_fixup (so the result is
// the same bit for bit).  Up to 64 loads per thread are in flight.
template <int BA, bool F16, bool SW>
__device__ void wide_fixup(const Args& a, const Shared* sh) {
  constexpr int P = kWarps * 32 / kTileW;
  constexpr int kCols = BA / P;                   // columns per thread
  constexpr int kCh = kCols < 16 ? kCols : 16;     // columns per pass
  constexpr int kUnroll = 64 / kCh;                // contributors per round
  static_assert(BA % P == 0, "columns split evenly over the parts");
  __threadfence();
  const int row = static_cast<int>(threadIdx.x) % kTileW;
  const int part = static_cast<int>(threadIdx.x) / kTileW;
  const int tile = sh->fix_tile;
  const int c_lo = sh->fix_clo, c_hi = sh->fix_chi;
  const int n = (tile % a.n_tiles) * kTileW + row;
  const int m0 = (tile / a.n_tiles) * BA;
  const int mcols = min(BA, a.M - m0);
  const float bias_n = (a.bias != nullptr && n < a.N) ? act_to_float<F16>(a.bias[n]) : 0.0f;
  constexpr int64_t kSlot = static_cast<int64_t>(BA) * kTileW;
  const float* lo = a.ws + (static_cast<int64_t>(c_lo) * 2 + sh->fix_slot) * kSlot + row;
#pragma unroll 1
  for (int j0 = 0; j0 < kCols; j0 += kCh) {
    if (part + P * j0 >= mcols) break;
    float acc[kCh];
#pragma unroll
    for (int j = 0; j < kCh; ++j) {
      const int col = part + P * (j0 + j);
      acc[j] = col < mcols ? __ldcg(lo + col * kTileW) : 0.0f;
    }
#pragma unroll kUnroll
    for (int c = c_lo + 1; c <= c_hi; ++c) {
      const float* src = a.ws + static_cast<int64_t>(c) * 2 * kSlot + row;
#pragma unroll
      for (int j = 0; j < kCh; ++j) {
        const int col = part + P * (j0 + j);
        if (col < mcols) acc[j] += __ldcg(src + col * kTileW);
      }
    }
    if (SW && a.sw) {
      float h[kCh];
#pragma unroll
      for (int j = 0; j < kCh; ++j) h[j] = acc[j] + bias_n;
      swiglu_vals(h);
      if (n < a.N && (n & 1) == 0) {
#pragma unroll
        for (int j = 0; j < kCh; ++j) {
          const int col = part + P * (j0 + j);
          if (col < mcols) a.Y[static_cast<int64_t>(m0 + col) * (a.N >> 1) + (n >> 1)] = act_from_float<F16>(h[j]);
        }
      }
    } else if (n < a.N) {
#pragma unroll
      for (int j = 0; j < kCh; ++j) {
        const int col = part + P * (j0 + j);
        if (col < mcols) a.Y[static_cast<int64_t>(m0 + col) * a.N + n] = act_from_float<F16>(acc[j] + bias_n);
      }
    }
  }
}

// Cluster split-K reduction, by every thread of every CTA of the cluster at
// exit.  The csk CTAs of a cluster hold the partials of one tile (rank r:
// the r-th K range) in their shared memory.  After a cluster barrier (every
// CTA reaches it: all of the kernel's waits before it are bounded, and a CTA
// whose wait ran out still comes here), CTA r sums the r-th slice of the
// tile's 128 x BA values over the ranks in rank order, i.e. in k order (the
// result does not depend on timing), reading its peers' partials through
// distributed shared memory, adds the bias in fp32, rounds once and stores
// Y.  A second cluster barrier keeps every CTA's shared memory alive until
// its peers have read it.  A CTA whose kernel gave up (abort flag) stores
// nothing: the error word already reports the launch as failed.
template <int BA, bool F16>
__device__ void csk_reduce(const Args& a, const Shared* sh, int cta, float* sp) {
  ptx::cluster_sync();
  const int S = a.csk;
  const int t = cta / S, r = cta - t * S;
  const int n0 = (t % a.n_tiles) * kTileW;
  const int m0 = (t / a.n_tiles) * BA;
  constexpr int kE = BA * kTileW;   // values of a tile, column-major ([BA][128])
  const int e0 = (r * kE) / S, e1 = ((r + 1) * kE) / S;
  const uint32_t base = ptx::smem_u32(sp);
  const bool ok = *reinterpret_cast<const volatile int*>(&sh->abort_flag) == 0;
  for (int e = e0 + static_cast<int>(threadIdx.x); ok && e < e1; e += static_cast<int>(blockDim.x)) {
    const int col = e / kTileW, row = e - col * kTileW;
    const int m = m0 + col, n = n0 + row;
    if (m >= a.M || n >= a.N) continue;
    float sum = 0.0f;
    for (int q = 0; q < S; ++q) sum += ptx::ld_dsmem_f32(base + 4u * static_cast<uint32_t>(e), q);
    if (a.bias != nullptr) sum += act_to_float<F16>(a.bias[n]);
    a.Y[static_cast<int64_t>(m) * a.N + n] = act_from_float<F16>(sum);
  }
  ptx::cluster_sync();
}

template <int BA, int L, bool GRP, int STAGES, int UG, int WF, bool F16, int G, bool SW>
__global__ void __launch_bounds__(Cfg<BA, L, GRP, STAGES, UG, WF>::kThreads, 1)
    w4a16_gemm_tc_kernel(const __grid_constant__ GroupArgs<G> g) {
  static_assert(WF == kFmtInt4 || !F16, "INT8 and FP4 weights with bf16 activations");
  // this CTA's problem and its index in the problem's sub-grid
  int prob = 0;
  if constexpr (G > 1) {
    while (prob + 1 < g.count && static_cast<int>(blockIdx.x) >= g.cta_start[prob + 1]) ++prob;
  }
  const Args& a = g.a[prob];
  const int cta = static_cast<int>(blockIdx.x) - g.cta_start[prob];
  const int ctas = g.cta_start[prob + 1] - g.cta_start[prob];
  const CUtensorMap* const tm_act = &g.tm[prob][0];
  const CUtensorMap* const tm_w = &g.tm[prob][1];
  const CUtensorMap* const tm_s = &g.tm[prob][2];
  using C = Cfg<BA, L, GRP, STAGES, UG, WF>;
  constexpr int DB = C::kDB;
  constexpr int SL = C::kSL;
  constexpr int AL = C::kAL;
  constexpr int DL = C::kDL;
  constexpr int RL = C::kRL;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  Shared* sh = reinterpret_cast<Shared*>(smem + C::kRing);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // activation boxes of a stage; codes and scales of a stage (split rings:
  // of a code stage)
  auto act_box = [&](int stage, int box) -> uint8_t* {
    return smem + stage * C::kActStride + box * C::kActBox;
  };
  auto w_tile = [&](int stage) -> uint8_t* { return smem + C::kWBase + stage * C::kWStride; };
  auto s_tile = [&](int stage, int gi) -> __half* {
    return reinterpret_cast<__half*>(w_tile(stage) + C::kSRel + gi * C::kSB);
  };
  // FP4: block-scale bytes of group gi of a stage, [block][128 rows]
  auto s_bytes = [&](int stage, int gi) -> const uint8_t* {
    return w_tile(stage) + C::kSRel + gi * C::kSB;
  };
  // Resources of unit i (lane p, index j in the lane): the lanes own
  // interleaved shared-memory stages, TMEM weight stages and accumulators.
  auto stage_of = [&](int i) -> int {
    int p, j;
    lane_split<L>(i, p, j);
    return p + L * (j % SL);
  };
  // TMEM weight stages go round per group: group jg of lane p's groups
  // (jg = UG * j + gi for group gi of the lane's unit j).
  auto gstage_of = [&](int p, int jg) -> int { return p + L * (jg % AL); };
  // split rings (one lane): the code stage of unit i
  auto wstage_of = [&](int i) -> int { return C::kSplit ? i % (C::kCodeStages > 0 ? C::kCodeStages : 1) : 0; };
  // Completion of unit i's MMAs.  Group mode: the pair ring (lane 0's and
  // lane 1's j-th units complete together, one arrival each); one lane:
  // the unit ring.
  auto done_bar = [&](int i) -> uint64_t* {
    int p, j;
    lane_split<L>(i, p, j);
    if constexpr (GRP) return &sh->pair_done[j % kPairRing];
    return &sh->unit_done[p * RL + j % RL];
  };
  auto done_parity = [&](int i) -> uint32_t {
    int p, j;
    lane_split<L>(i, p, j);
    if constexpr (GRP) return static_cast<uint32_t>((j / kPairRing) & 1);
    return static_cast<uint32_t>((j / RL) & 1);
  };

  // ---------------------------------------------------------------- set-up
#ifdef W4A16_TRACE
  unsigned long long* const trace_cta = g_trace;
  unsigned long long* const trace_unit = blockIdx.x == 0 ? g_trace_units : nullptr;
#endif
  if (threadIdx.x == 0) W4A16_TRACE_POINT(0);
  if (threadIdx.x == 0) W4A16_TRACE_UNIT(9, 0);
  {
    // barriers initialised in parallel, one per thread (one thread doing all
    // of them in turn costs several hundred cycles of the launch's head)
    const int t = static_cast<int>(threadIdx.x);
    bool init = true;
    if (t < C::kActStages) {
      ptx::mbar_init(&sh->full[t], 1);
    } else if (C::kSplit && t >= 224 && t < 224 + C::kCodeStages) {
      ptx::mbar_init(&sh->wfull[t - 224], 1);
      ptx::mbar_init(&sh->wempty[t - 224], 4);   // the 4 warps of a dequant warpgroup
    } else if (t >= 32 && t < 32 + L * RL) {
      ptx::mbar_init(&sh->unit_done[t - 32], 1);
    } else if (t >= 64 && t < 64 + C::kAS) {
      ptx::mbar_init(&sh->afull[t - 64], 4);
    } else if (t >= 96 && t < 96 + DB) {
      // dequant mode: both lanes' MMA threads arrive (L = 2)
      ptx::mbar_init(&sh->dfull[t - 96], GRP ? 1 : L);
      ptx::mbar_init(&sh->dempty[t - 96], 4);
    } else if (t >= 128 && t < 128 + kPairRing) {
      ptx::mbar_init(&sh->pair_done[t - 128], 2);
    } else if (t == 160) {
      ptx::mbar_init(&sh->mma_done[0], 1);
      ptx::mbar_init(&sh->mma_done[1], 1);
      ptx::mbar_init(&sh->rsync, 4);
      sh->abort_flag = 0;
      sh->fixup_last = 0;
      sh->fixup_defer = 0;
    } else {
      init = false;
    }
    if (init) ptx::fence_mbar_init();
    if (t == 192) {
      ptx::prefetch_tmap(tm_act);
      ptx::prefetch_tmap(tm_w);
      ptx::prefetch_tmap(tm_s);
    }
  }
  if (warp == 1) {
    ptx::tmem_alloc(&sh->tmem_base, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = sh->tmem_base;
  const WaitCtx wc{a.err, a.timeout_ns, &sh->abort_flag};

  if (threadIdx.x == 0) W4A16_TRACE_POINT(1);
  if (threadIdx.x == 0) W4A16_TRACE_UNIT(9, 1);
  // The schedule depends on the launch only, so it is worked out while the
  // previous kernel on the stream may still run; the inputs may be that
  // kernel's outputs, so nothing is read before the dependency wait.
  Sched sched;
  sched.init(a, cta, ctas);
  const int total = sched.total;
#ifdef W4A16_TRACE
  if (threadIdx.x == 0 && trace_cta != nullptr) {
    // profiling builds: the CTA's problem, units and dp tiles next to its times
    trace_cta[blockIdx.x * 16 + 12] = static_cast<unsigned long long>(prob);
    trace_cta[blockIdx.x * 16 + 13] = static_cast<unsigned long long>(total);
    trace_cta[blockIdx.x * 16 + 14] = static_cast<unsigned long long>(sched.dp_iters);
  }
#endif
  // Every role but the producers waits for the previous kernel on the stream
  // here (its outputs may be this kernel's inputs); the producers wait in
  // their own branch, after any early weight copies.
  const bool producer = warp == 0 || warp == 2;
  if (!producer) {
    ptx::grid_dependency_wait();
    ptx::grid_launch_dependents();
  }
  if (threadIdx.x == 32) W4A16_TRACE_POINT(2);
  if (threadIdx.x == 32) W4A16_TRACE_UNIT(9, 2);

  if (producer) {
    // ----------------------------------------------------- TMA producers
    // Even units from warp 0, odd units from warp 2 (with two lanes: one
    // producer per lane).  A producer walks the CTA's runs (consecutive
    // units on one tile): a run's coordinates are worked out once, a unit's
    // by additions, so that the one issuing thread spends its time on the
    // copies.  With prefetch_w, the codes and scales of the first stages go
    // out before the dependency wait (the weights are not the previous
    // kernel's outputs) and the activations of those stages after it.
    if (lane != 0) {
      ptx::grid_dependency_wait();
    } else {
      const int mine = warp == 0 ? 0 : 1;
      int issued = -1;
      auto walk = [&](int limit, auto&& fn) -> bool {
        SegCursor cur;
        cur.init(sched);
        int i0 = 0;
        while (i0 < total && i0 < limit) {
          Unit r;
          int kb0, len;
          cur.next(r, kb0, len, a.dp_tiles);
          const int mt = r.tile / a.n_tiles;
          const int tn = r.tile - mt * a.n_tiles;
          const int m0 = mt * BA;
          const int wrow0 = tn * a.KB * UG * kTileW;
          const int sx = tn * kTileW;
          // split rings: one producer walks every unit (warp 0 the codes,
          // warp 2 the activations); else even units from warp 0, odd from 2
          constexpr int kStep = C::kSplit ? 1 : 2;
          for (int i = i0 + (!C::kSplit && (i0 & 1) != mine ? 1 : 0); i < i0 + len && i < limit;
               i += kStep) {
            const int g0 = (kb0 + i - i0) * UG;   // the unit's first group
            if (!fn(i, m0, wrow0 + g0 * kTileW, sx, g0)) return false;
          }
          i0 += len;
        }
        return true;
      };
      // the unit's codes (UG consecutive 8 KiB tiles of the tiled storage:
      // one contiguous block) and its scales
      auto issue_w = [&](int stage, int wrow, int sx, int g0) {
        ptx::mbar_arrive_expect_tx(&sh->full[stage], C::kTx);
        ptx::tma_load_2d(w_tile(stage), tm_w, &sh->full[stage], 0, wrow);
        ptx::tma_load_2d(s_tile(stage, 0), tm_s, &sh->full[stage], sx, g0 * wf_blocks(WF));
      };
      auto issue_a = [&](int stage, int m0, int g0) {
        if (a.act_3d) {
          ptx::tma_load_3d(act_box(stage, 0), tm_act, &sh->full[stage], 0, m0, g0 * 2);
        } else {
#pragma unroll
          for (int b = 0; b < 2 * UG; ++b)
            ptx::tma_load_2d(act_box(stage, b), tm_act, &sh->full[stage], g0 * kUnitK + 64 * b, m0);
        }
      };
      if constexpr (C::kSplit) {
        if (warp == 0) {
          // codes and scales of every unit into the code ring; with static
          // weights the whole ring is requested before the dependency wait
          auto issue_c = [&](int i, int wrow, int sx, int g0) {
            const int ws = wstage_of(i);
            ptx::mbar_arrive_expect_tx(&sh->wfull[ws], C::kTxCode);
            ptx::tma_load_2d(w_tile(ws), tm_w, &sh->wfull[ws], 0, wrow);
            ptx::tma_load_2d(s_tile(ws, 0), tm_s, &sh->wfull[ws], sx, g0 * wf_blocks(WF));
          };
          const int npre = a.prefetch_w > 0 ? C::kCodeStages : 0;
          if (npre > 0) {
            walk(npre, [&](int i, int, int wrow, int sx, int g0) {
              issue_c(i, wrow, sx, g0);
              issued = i;
              return true;
            });
          }
          ptx::grid_dependency_wait();
          ptx::grid_launch_dependents();
          walk(total, [&](int i, int, int wrow, int sx, int g0) {
            if (i < npre) return true;
            // the stage's previous unit (i - kCodeStages) was read by the dequant
            if (i >= C::kCodeStages &&
                !wait_one(&sh->wempty[wstage_of(i)], static_cast<uint32_t>((i / C::kCodeStages) - 1) & 1u,
                          wc))
              return false;
            issue_c(i, wrow, sx, g0);
            W4A16_TRACE_UNIT(0, i);
            issued = i;
            return true;
          });
          if (*reinterpret_cast<volatile int*>(&sh->abort_flag)) {
            // this producer's copies still in flight land before the CTA exits
            for (int i = issued; i >= 0 && i > issued - C::kCodeStages; --i) {
              const uint64_t t0 = ptx::globaltimer_ns();
              while (!ptx::mbar_try_wait(&sh->wfull[wstage_of(i)],
                                         static_cast<uint32_t>(i / C::kCodeStages) & 1u)) {
                if (ptx::globaltimer_ns() - t0 > a.timeout_ns) break;
              }
            }
          }
        } else {
          // activations of every unit into the activation ring; a stage is
          // free once the MMAs of its previous unit completed
          ptx::grid_dependency_wait();
          ptx::grid_launch_dependents();
          walk(total, [&](int i, int m0, int, int, int g0) {
            const int stage = stage_of(i);
            if (i >= C::kActStages &&
                !wait_one(done_bar(i - C::kActStages), done_parity(i - C::kActStages), wc))
              return false;
            ptx::mbar_arrive_expect_tx(&sh->full[stage], C::kTxAct);
            issue_a(stage, m0, g0);
            if (i <= 1) W4A16_TRACE_POINT(3);
            issued = i;
            return true;
          });
          if (*reinterpret_cast<volatile int*>(&sh->abort_flag)) {
            for (int i = issued; i >= 0 && i > issued - C::kActStages; --i) {
              const uint64_t t0 = ptx::globaltimer_ns();
              while (!ptx::mbar_try_wait(&sh->full[stage_of(i)],
                                         static_cast<uint32_t>(i / C::kActStages) & 1u)) {
                if (ptx::globaltimer_ns() - t0 > a.timeout_ns) break;
              }
            }
          }
        }
      } else {
      // a shallow prefetch: the copies of one TMA unit run in order, so every
      // early weight copy sits ahead of the first activation copy
      const int npre = a.prefetch_w < STAGES ? a.prefetch_w : STAGES;
      if (npre > 0) {
        walk(npre, [&](int i, int, int wrow, int sx, int g0) {
          issue_w(stage_of(i), wrow, sx, g0);
          return true;
        });
      }
      ptx::grid_dependency_wait();
      ptx::grid_launch_dependents();
      walk(total, [&](int i, int m0, int wrow, int sx, int g0) {
        const int stage = stage_of(i);
        if (i < npre) {
          issue_a(stage, m0, g0);
        } else {
          // the unit that last used this stage is i - STAGES (same producer)
          if (i >= STAGES && !wait_one(done_bar(i - STAGES), done_parity(i - STAGES), wc))
            return false;
          W4A16_TRACE_UNIT(13, i);
          issue_w(stage, wrow, sx, g0);
          issue_a(stage, m0, g0);
        }
        if (i <= 1) W4A16_TRACE_POINT(3);
        W4A16_TRACE_UNIT(0, i);
        issued = i;
        return true;
      });
      if (*reinterpret_cast<volatile int*>(&sh->abort_flag)) {
        // let this producer's copies still in flight land before the CTA exits
        for (int i = issued; i >= 0 && i > issued - STAGES; i -= 2) {
          int p, j;
          lane_split<L>(i, p, j);
          const uint64_t t0 = ptx::globaltimer_ns();
          while (!ptx::mbar_try_wait(&sh->full[stage_of(i)], (j / SL) & 1)) {
            if (ptx::globaltimer_ns() - t0 > a.timeout_ns) break;
          }
        }
      }
      }
    }
  } else if (warp == 1 || (L == 2 && warp == kMmaWarp2)) {
    // ------------------------------------------------------- MMA issuers
    // One thread per lane: one thread alone cannot issue small-N MMAs as
    // fast as the tensor pipe runs them.
    if (lane == 0) {
      const int mine = warp == 1 ? 0 : 1;
      constexpr uint32_t idesc = ptx::idesc_f16kind_f32(kTileW, BA, F16 ? 0u : 1u);
      const uint32_t smem0 = ptx::smem_u32(smem);
      if constexpr (GRP) {
        // this lane's units j = 0, 1, ...: unit i = 2 j + mine; every unit
        // starts a fresh accumulator (the readout applies the group scale)
        const int nj = (total - mine + 1) >> 1;
        bool ok = true;
        for (int j = 0; j < nj && ok; ++j) {
          const int stage = mine + 2 * (j % SL);
          const int dl = j % DL;
          const uint32_t b0 = smem0 + stage * C::kActStride;
#pragma unroll
          for (int gi = 0; gi < UG; ++gi) {
            const int jg = UG * j + gi;
            const int as = gstage_of(mine, jg);
            if (gi == 0) W4A16_TRACE_UNIT(23, 2 * j + mine);
            if (!wait_one(&sh->afull[as], (jg / AL) & 1, wc)) {
              ok = false;
              break;
            }
            if (gi == 0) W4A16_TRACE_UNIT(24, 2 * j + mine);
            // accumulator buffer dl of this lane is free once the readout
            // loaded the lane's unit j - DL (one barrier per buffer, so the
            // MMAs run up to DL units ahead of the readout)
            if (gi == 0 && j >= DL &&
                !wait_one(&sh->dempty[mine * DL + dl], ((j / DL) - 1) & 1, wc)) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            if (j == 0 && gi == 0) W4A16_TRACE_POINT(4);
            W4A16_TRACE_UNIT(gi == 0 ? 4 : 20, 2 * j + mine);
            // group gi of the unit: its own accumulator
            const uint32_t d_tmem = tmem + C::kDCol + ((mine + 2 * dl) * UG + gi) * BA;
            const uint32_t a_tmem = tmem + as * kAStageCols;
            const uint64_t bdesc = ptx::smem_desc_sw128(b0 + 2 * gi * C::kActBox);
#pragma unroll
            for (int kk = 0; kk < kUnitK / 16; ++kk) {
              // K step kk: 64-k half kk / 4, 32 bytes per 16 k inside it
              const uint32_t boff = ((kk >> 2) * C::kActBox + (kk & 3) * 32) >> 4;
              ptx::mma_f16kind_tmem_a(d_tmem, a_tmem + kk * 8, bdesc + boff, idesc,
                                      kk > 0 ? 1u : 0u);
            }
            W4A16_TRACE_UNIT(gi == 0 ? 21 : 22, 2 * j + mine);
          }
          if (!ok) break;
          // one arrival per lane on the pair's barrier; an unpaired last
          // unit (lane 0) arrives for both
          ptx::mma_commit(&sh->pair_done[j % kPairRing]);
          if (mine == 0 && 2 * j == total - 1) ptx::mma_commit(&sh->pair_done[j % kPairRing]);
          W4A16_TRACE_UNIT(5, 2 * j + mine);
        }
        if (nj > 0) W4A16_TRACE_POINT(5);
      } else {
        // Dequant mode: a run accumulates in TMEM across its units.  Each
        // lane accumulates its own units of the run in its own half of the
        // run's buffer; the readout adds the halves.
        int seg = 0;
        int db = 0;
        bool have = false;   // this lane issued into the current run's buffer
        UnitIter it;
        it.init(sched);
        for (int i = 0; i < total; ++i) {
          const Unit u = it.next();
          if (u.seg_first) {
            db = seg % DB;
            have = false;
          }
          int p, j;
          lane_split<L>(i, p, j);
          if (p == mine) {
            const int stage = stage_of(i);
            const uint32_t b0 = smem0 + stage * C::kActStride;
            const uint32_t d_tmem = tmem + C::kDCol + (db * L + mine) * BA;
            W4A16_TRACE_UNIT(8, i);
            bool ok = true;
            // split rings: the activations have a barrier of their own (the
            // dequant's arrival covers only the codes)
            if constexpr (C::kSplit) {
              if (!wait_one(&sh->full[stage], static_cast<uint32_t>(j / SL) & 1u, wc)) break;
            }
#pragma unroll
            for (int gi = 0; gi < UG; ++gi) {
              const int jg = UG * j + gi;
              const int as = gstage_of(mine, jg);
              if (!wait_one(&sh->afull[as], (jg / AL) & 1, wc)) {
                ok = false;
                break;
              }
              if (gi == 0) W4A16_TRACE_UNIT(10, i);
              // the buffer's previous run (seg - DB) was drained by the readout
              if (!have && seg >= DB &&
                  !wait_one(&sh->dempty[db], ((seg / DB) - 1) & 1, wc)) {
                ok = false;
                break;
              }
              ptx::tc_fence_after();
              if (i == 0 && gi == 0) W4A16_TRACE_POINT(4);
              if (i == total - 1 && gi == 0) W4A16_TRACE_POINT(5);
              if (gi == 0) W4A16_TRACE_UNIT(4, i);
              const uint32_t a_tmem = tmem + as * kAStageCols;
              const uint64_t bdesc = ptx::smem_desc_sw128(b0 + 2 * gi * C::kActBox);
              // the last activation tile: only its columns that hold rows
              const uint32_t id = u.tile >= a.tail_tile0
                                      ? ptx::idesc_f16kind_f32(kTileW, a.tail_n, F16 ? 0u : 1u)
                                      : idesc;
#pragma unroll
              for (int kk = 0; kk < kUnitK / 16; ++kk) {
                const uint32_t boff = ((kk >> 2) * C::kActBox + (kk & 3) * 32) >> 4;
                ptx::mma_f16kind_tmem_a(d_tmem, a_tmem + kk * 8, bdesc + boff, id,
                                        (kk > 0 || have) ? 1u : 0u);
              }
              have = true;
            }
            if (!ok) break;
            W4A16_TRACE_UNIT(11, i);
            ptx::mma_commit(done_bar(i));
          }
          if (u.seg_last) {
            if (have) {
              ptx::mma_commit(&sh->dfull[db]);
            } else {
              // no unit of this lane in the run: arrive without MMAs, once
              // the buffer's previous run was drained
              if (seg >= DB && !wait_one(&sh->dempty[db], ((seg / DB) - 1) & 1, wc)) break;
              ptx::mbar_arrive(&sh->dfull[db]);
            }
            ++seg;
            W4A16_TRACE_UNIT(5, i);
          }
        }
      }
      // all MMAs of this thread complete before TMEM is freed
      ptx::mma_commit(&sh->mma_done[mine]);
      const uint64_t t0 = ptx::globaltimer_ns();
      while (!ptx::mbar_try_wait(&sh->mma_done[mine], 0)) {
        if (ptx::globaltimer_ns() - t0 > a.timeout_ns) {
          wait_record_timeout(wc);
          break;
        }
      }
    }
  } else if (warp >= kReadoutWarp0 && warp < kReadoutWarp0 + 4) {
    // ------------------------------------------------------------ readout
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    if constexpr (GRP) {
      // Units come in pairs (lane 0's j-th unit, lane 1's j-th unit), behind
      // one barrier that both lanes' MMA threads arrive on.  Per pair: one
      // wait, both accumulators loaded, then acc += s * D for each unit in
      // order.  Per unit only a countdown; tile, row and scale addresses are
      // computed once per run ("segment") of the CTA.
      float acc[BA];
      // Scales: copied from global memory into a ring in shared memory
      // kScaleAhead pairs before they are needed (per-thread asynchronous
      // copies; each even lane copies its row's and the next row's scale).
      uint16_t* const sring =
          reinterpret_cast<uint16_t*>(reinterpret_cast<uint8_t*>(sh) + sizeof(Shared));
      SegCursor pf_cur;
      pf_cur.init(sched);
      int pf_left = 0;
      const __half* pf_ptr = a.scales;
      bool pf_ok = false;
      auto prefetch_unit = [&](int jj) {
        if (jj >= total) return;
        if (pf_left == 0) {
          Unit v;
          int kb0;
          pf_cur.next(v, kb0, pf_left, a.dp_tiles);
          const int nn = (v.tile % a.n_tiles) * kTileW + row;
          pf_ok = nn < a.N;   // N % 8 == 0: row nn + 1 exists too
          pf_ptr = a.scales + static_cast<int64_t>(kb0) * UG * a.N + nn;
        } else {
          pf_ptr += static_cast<int64_t>(UG) * a.N;
        }
        --pf_left;
        if ((lane & 1) == 0 && pf_ok) {
#pragma unroll
          for (int gi = 0; gi < UG; ++gi)
            ptx::cp_async_4(ptx::smem_u32(sring + ((jj % kScaleRing) * UG + gi) * kTileW + row),
                            pf_ptr + static_cast<int64_t>(gi) * a.N);
        }
      };
#pragma unroll
      for (int q = 0; q < kScaleAhead; ++q) {
        prefetch_unit(2 * q);
        prefetch_unit(2 * q + 1);
        ptx::cp_async_commit();
      }
      // the current run
      SegCursor cur;
      cur.init(sched);
      Unit seg;
      SplitInfo si{0, 0, 0};
      int seg_left = 0;
      bool first = true;
      float bias_f = 0.0f;
      uint32_t nsync = 0;
      bool ok = true;
      auto open_run = [&]() {
        int kb0;
        cur.next(seg, kb0, seg_left, a.dp_tiles);
        const int n = (seg.tile % a.n_tiles) * kTileW + row;
        bias_f = (a.bias != nullptr && n < a.N) ? act_to_float<F16>(a.bias[n]) : 0.0f;
        if (!seg.whole && a.csk <= 1) si = split_info(a, seg.sk_tile, ctas);
        first = true;
      };
      if (total > 0) open_run();
      // acc (+)= scale * D for one group, 16 columns at a time (`first`:
      // the run's first group sets acc); emits at the end of a run
      auto accumulate = [&](float scale, const uint32_t* d, int c0) {
#pragma unroll
        for (int c = 0; c < 16; ++c)
          acc[c0 + c] = first ? scale * __uint_as_float(d[c]) : fmaf(scale, __uint_as_float(d[c]), acc[c0 + c]);
      };
      auto scale_at = [&](int i, int gi) -> float {
        return __half2float(
            __ushort_as_half(sring[((i % kScaleRing) * UG + gi) * kTileW + row]));
      };
      auto finish_unit = [&](int i) {
        first = false;
        if (--seg_left == 0) {
          emit_cols<BA, BA, F16, SW>(a, seg, row, 0, acc, bias_f, cta, csk_partial(smem));
          if (!seg.whole && a.csk <= 1)
            ok = split_fixup<BA, F16, SW>(a, seg, si, sh, row, bias_f, nsync, wc, i + 1 == total);
          if (i + 1 < total) open_run();
        }
      };
      const int pairs = (total + 1) >> 1;
      for (int q = 0; q < pairs; ++q) {
        const int i0 = 2 * q;
        const bool has1 = i0 + 1 < total;
        const int dl = q % DL;
        prefetch_unit(2 * (q + kScaleAhead));
        prefetch_unit(2 * (q + kScaleAhead) + 1);
        ptx::cp_async_commit();
        ptx::cp_async_wait<kScaleAhead>();   // this pair's copies landed
        __syncwarp();
        float s0[UG], s1[UG];
#pragma unroll
        for (int gi = 0; gi < UG; ++gi) {
          s0[gi] = scale_at(i0, gi);
          s1[gi] = scale_at(i0 + 1, gi);
        }
        if (threadIdx.x == 32 * kReadoutWarp0) W4A16_TRACE_UNIT(12, i0);
        if (!wait_warp(&sh->pair_done[q % kPairRing], (q / kPairRing) & 1, wc)) break;
        if (threadIdx.x == 32 * kReadoutWarp0 && q == 0) W4A16_TRACE_POINT(8);
        if (threadIdx.x == 32 * kReadoutWarp0 && q == pairs - 1) W4A16_TRACE_POINT(9);
        if (threadIdx.x == 32 * kReadoutWarp0) W4A16_TRACE_UNIT(6, i0);
        ptx::tc_fence_after();
        // unit accumulators: UG groups of BA columns each
        const uint32_t d0 = lane_base + C::kDCol + (0 + 2 * dl) * UG * BA;
        const uint32_t d1 = lane_base + C::kDCol + (1 + 2 * dl) * UG * BA;
        auto release = [&]() {
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            ptx::mbar_arrive(&sh->dempty[dl]);
            if (has1) ptx::mbar_arrive(&sh->dempty[DL + dl]);
          }
          if (threadIdx.x == 32 * kReadoutWarp0) W4A16_TRACE_UNIT(7, i0);
        };
        if constexpr (BA == 16) {
          // both units' accumulators (all their groups) with one TMEM wait
          uint32_t r0[16 * UG], r1[16 * UG];
          if constexpr (UG == 1) {
            ptx::tmem_ld2_x16_sync(d0, d1, r0, r1);
          } else {
            ptx::tmem_ld2_x32_sync(d0, d1, r0, r1);
          }
          release();
#pragma unroll
          for (int gi = 0; gi < UG; ++gi) {
            accumulate(s0[gi], r0 + 16 * gi, 0);
            first = false;
          }
          finish_unit(i0);
          if (has1) {
#pragma unroll
            for (int gi = 0; gi < UG; ++gi) {
              accumulate(s1[gi], r1 + 16 * gi, 0);
              first = false;
            }
            finish_unit(i0 + 1);
          }
        } else {
          // one unit at a time, one group at a time, 16 columns per TMEM load
#pragma unroll 1
          for (int h = 0; h <= (has1 ? 1 : 0); ++h) {
#pragma unroll
            for (int gi = 0; gi < UG; ++gi) {
#pragma unroll
              for (int c0 = 0; c0 < BA; c0 += 16) {
                uint32_t r[16];
                ptx::tmem_ld_x16_sync((h ? d1 : d0) + gi * BA + c0, r);
                accumulate(h ? s1[gi] : s0[gi], r, c0);
              }
              first = false;
            }
            if (h == (has1 ? 1 : 0)) release();
            finish_unit(i0 + h);
          }
        }
        if (!ok) break;
      }
      ptx::cp_async_wait<0>();   // no copy may land after exit
    } else {
      uint16_t bias_raw = 0;
      int seg = 0;
      int i_first = 0;
      uint32_t nsync = 0;
      // NVFP4: g multiplies every fp32 sum (partials too: the fixup adds
      // scaled partials) before the bias
      float g_t = 1.0f;
      if constexpr (WF == kFmtNvfp4) g_t = __ldg(a.out_scale);
      UnitIter it;
      it.init(sched);
      for (int i = 0; i < total; ++i) {
        const Unit u = it.next();
        if (u.seg_first) {
          const int n = (u.tile % a.n_tiles) * kTileW + row;
          bias_raw = (a.bias != nullptr && n < a.N) ? a.bias[n] : static_cast<uint16_t>(0);
          i_first = i;
        }
        if (!u.seg_last) continue;
        const int db = seg % DB;
        if (!wait_warp(&sh->dfull[db], (seg / DB) & 1, wc)) break;
        ++seg;
        ptx::tc_fence_after();
        const float bias_f = act_to_float<F16>(bias_raw);
        // the lanes that hold units of this run (a run of one unit has one)
        const bool has0 = L == 1 || i > i_first || (i_first & 1) == 0;
        const bool has1 = L == 2 && (i > i_first || (i_first & 1) == 1);
        const uint32_t buf = lane_base + C::kDCol + db * L * BA;
        // columns past the last activation row were not computed (M-tail)
        const int mcols = min(BA, a.M - (u.tile / a.n_tiles) * BA);
#pragma unroll 1
        for (int c0 = 0; c0 < BA; c0 += C::kChunk) {
          if (c0 >= mcols) break;
          float v[C::kChunk];
          load_cols<C::kChunk>(buf + (has0 ? 0 : BA) + c0, v);
          if (has0 && has1) {
            float w[C::kChunk];
            load_cols<C::kChunk>(buf + BA + c0, w);
#pragma unroll
            for (int c = 0; c < C::kChunk; ++c) v[c] += w[c];
          }
          if constexpr (WF == kFmtNvfp4) {
#pragma unroll
            for (int c = 0; c < C::kChunk; ++c) v[c] *= g_t;
          }
          emit_cols<BA, C::kChunk, F16, SW>(a, u, row, c0, v, bias_f, cta, csk_partial(smem));
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&sh->dempty[db]);
        if (!u.whole && a.csk <= 1 &&
            !split_fixup<BA, F16, SW>(a, u, split_info(a, u.sk_tile, ctas), sh, row, bias_f, nsync, wc,
                                  i + 1 == total))
          break;
      }
    }
  } else if (warp >= kDequantWarp0 && warp < kDequantWarp0 + 8) {
    // ------------------------------------------------------------ dequant
    // warpgroup wg converts units wg, wg + 2, ... (with two lanes: lane wg's
    // units): every thread its whole row of 128 codes per unit
    const int wg = (warp - kDequantWarp0) >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    // a row of a group's codes: 64 B (INT4, 64-byte swizzle: 16-byte chunk c
    // of row r at c ^ ((r >> 1) & 3)) or 128 B (INT8, 128-byte swizzle:
    // chunk c at c ^ (r & 7))
    constexpr int kRowBytes = wf_bits(WF) * 16;
    constexpr int kChunks = kRowBytes / 16;
    const uint32_t wrow0 = ptx::smem_u32(w_tile(0)) + row * kRowBytes;
    const uint32_t swz = wf_bits(WF) == 4 ? ((row >> 1) & 3) : (row & 7);
    for (int i = wg; i < total; i += 2) {
      int p, j;
      lane_split<L>(i, p, j);
      // the stage holding unit i's codes (split rings: its code stage)
      const int stage = C::kSplit ? wstage_of(i) : stage_of(i);
      if constexpr (!C::kSplit && L == 1 && (STAGES & 1) != 0) {
        // With an odd stage count the uses of one stage alternate between
        // the two warpgroups, so this warpgroup did not see the stage's
        // previous phase (unit i - STAGES, the other warpgroup's), and a
        // parity wait cannot tell that phase from this unit's.  The producer
        // refills the stage only after the MMAs of unit i - STAGES completed,
        // so waiting for those first proves the previous phase complete.
        if (i >= STAGES && !wait_warp(done_bar(i - STAGES), done_parity(i - STAGES), wc)) break;
      }
      if (threadIdx.x == 32 * kDequantWarp0) W4A16_TRACE_UNIT(25, i);
      if constexpr (C::kSplit) {
        if (!wait_warp(&sh->wfull[stage], static_cast<uint32_t>(i / C::kCodeStages) & 1u, wc)) break;
      } else {
        if (!wait_warp(&sh->full[stage], (j / SL) & 1, wc)) break;
      }
      if (i == 0 && threadIdx.x == 32 * kDequantWarp0) W4A16_TRACE_POINT(6);
      if (threadIdx.x == 32 * kDequantWarp0) W4A16_TRACE_UNIT(1, i);
      bool ok = true;
      // the row's codes of every group of the unit
      uint32_t words[UG][4 * kChunks];
#pragma unroll
      for (int gi = 0; gi < UG; ++gi) {
        const uint32_t wrow = wrow0 + stage * C::kWStride + gi * C::kWB;
#pragma unroll
        for (int q = 0; q < kChunks; ++q) {
          const uint4 v = ptx::lds128(wrow + ((q ^ swz) << 4));
          words[gi][4 * q + 0] = v.x;
          words[gi][4 * q + 1] = v.y;
          words[gi][4 * q + 2] = v.z;
          words[gi][4 * q + 3] = v.w;
        }
      }
      // split rings: the row's scales too, then the code stage goes back to
      // the producer (the values are in registers)
      __half sv[UG];
      if constexpr (C::kSplit) {
#pragma unroll
        for (int gi = 0; gi < UG; ++gi) sv[gi] = s_tile(stage, gi)[row];
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&sh->wempty[stage]);
      }
      if (threadIdx.x == 32 * kDequantWarp0) W4A16_TRACE_UNIT(16, i);
#pragma unroll
      for (int gi = 0; gi < UG; ++gi) {
        // the TMEM stage is free once the MMAs of its previous group (jg - AL
        // of this lane) completed: the completion of the unit that group
        // belongs to (one commit per unit and issuer serves the stage, the
        // shared-memory stage and the readout; a commit costs an issuing
        // thread about as much as two MMAs)
        const int jg = UG * j + gi;
        const int as = gstage_of(p, jg);
        if (jg >= AL) {
          const int iprev = L * ((jg - AL) / UG) + p;
          if (!wait_warp(done_bar(iprev), done_parity(iprev), wc)) {
            ok = false;
            break;
          }
        }
        if (threadIdx.x == 32 * kDequantWarp0) W4A16_TRACE_UNIT(gi == 0 ? 2 : 17, i);
        ptx::tc_fence_after();
        const uint32_t a_addr = lane_base + as * kAStageCols;
        uint32_t s_hi2 = 0, s_lo2 = 0;
        float s_w8 = 0.0f;
        if constexpr (wf_fp4(WF)) {
          // the block scales are read per block below
        } else if constexpr (!GRP && WF == kFmtInt8) {
          s_w8 = __half2float(C::kSplit ? sv[gi] : s_tile(stage, gi)[row]);
        } else if constexpr (!GRP) {
          if constexpr (F16) {
            // fp16 operand: fp16_rn(q * s) is one fused multiply-add (q and
            // s are both fp16)
            const uint32_t sb = static_cast<uint32_t>(__half_as_ushort(s_tile(stage, gi)[row]));
            s_hi2 = sb | (sb << 16);
          } else {
            const float scale = __half2float(s_tile(stage, gi)[row]);
            const __nv_bfloat16 hi = __float2bfloat16_rn(scale);
            const float lo_f = scale - __bfloat162float(hi);        // exact
            const __nv_bfloat16 lo = __float2bfloat16_rn(lo_f);     // exact
            const uint32_t hi_bits = static_cast<uint32_t>(__bfloat16_as_ushort(hi));
            const uint32_t lo_bits = static_cast<uint32_t>(__bfloat16_as_ushort(lo));
            s_hi2 = hi_bits | (hi_bits << 16);
            s_lo2 = lo_bits | (lo_bits << 16);
          }
        }
        // convert and store 16 columns (4 code words) at a time
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t opnd[16];
          if constexpr (wf_fp4(WF)) {
            // 32 K values: one MXFP4 block, or two NVFP4 blocks (words 4 q,
            // 4 q + 1 and 4 q + 2, 4 q + 3)
#pragma unroll
            for (int w = 0; w < 4; ++w) {
              constexpr int kWordsPerBlock = WF == kFmtMxfp4 ? 4 : 2;
              const int blk = (4 * q + w) / kWordsPerBlock;
              const uint32_t sc = s_bytes(stage, gi)[blk * kTileW + row];
              uint32_t h2, off2;
              if constexpr (WF == kFmtMxfp4) {
                mx_half_scale(sc, h2, off2);
              } else {
                nv_half_scale(sc, h2, off2);
              }
              e2m1_to_operand(words[gi][4 * q + w], h2, off2, &opnd[4 * w]);
            }
          } else if constexpr (WF == kFmtInt4) {
#pragma unroll
            for (int w = 0; w < 4; ++w) codes_to_operand<F16>(words[gi][4 * q + w], &opnd[4 * w]);
          } else {
#pragma unroll
            for (int w = 0; w < 8; ++w) bytes_to_operand_bf16(words[gi][8 * q + w], &opnd[2 * w]);
          }
          if constexpr (wf_fp4(WF)) {
            // scaled during the conversion
          } else if constexpr (!GRP && WF == kFmtInt8) {
#pragma unroll
            for (int c = 0; c < 16; ++c) opnd[c] = scale_pair_bf16_f32(opnd[c], s_w8);
          } else if constexpr (!GRP) {
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              if constexpr (F16) {
                opnd[c] = x2_fma<true>(opnd[c], s_hi2, 0x80008000u);   // q * s + (-0)
              } else {
                opnd[c] = scale_pair_bf16(opnd[c], s_hi2, s_lo2);
              }
            }
          }
          ptx::tmem_st_x16(a_addr + 16 * q, opnd);
        }
      }
      if (!ok) break;
      // one wait for all groups' TMEM stores (the stores of one group
      // complete while the next one converts), then one arrival per group
      if (threadIdx.x == 32 * kDequantWarp0) W4A16_TRACE_UNIT(18, i);
      ptx::tmem_st_wait();
      if (threadIdx.x == 32 * kDequantWarp0) W4A16_TRACE_UNIT(19, i);
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
#pragma unroll
        for (int gi = 0; gi < UG; ++gi) ptx::mbar_arrive(&sh->afull[gstage_of(p, UG * j + gi)]);
      }
      if (!ok) break;
      if (threadIdx.x == 32 * kDequantWarp0) W4A16_TRACE_UNIT(3, i);
      if (i >= total - 2 && threadIdx.x == 32 * kDequantWarp0) W4A16_TRACE_POINT(7);
    }
  }

  // ------------------------------------------------------------- teardown
  if (threadIdx.x == 32 * kReadoutWarp0) W4A16_TRACE_POINT(10);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem, kTmemCols);
  if (sh->fixup_defer) wide_fixup<BA, F16, SW>(a, sh);
  if (a.csk > 1) csk_reduce<BA, F16>(a, sh, cta, csk_partial(smem));
  if (threadIdx.x == 32) W4A16_TRACE_POINT(11);
}

template <int BA, int L, bool GRP, int STAGES, int UG, int WF, bool F16, int G, bool SW = false>
cudaError_t launch_instance(const GemmGroup& grp, bool use_pdl, cudaStream_t stream) {
  using C = Cfg<BA, L, GRP, STAGES, UG, WF>;
  auto kernel = w4a16_gemm_tc_kernel<BA, L, GRP, STAGES, UG, WF, F16, G, SW>;
  if (grp.count < 1 || grp.count > G) return cudaErrorInvalidValue;

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

  constexpr CUtensorMapDataType kActType =
      F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  GroupArgs<G> g{};
  int start = 0;
  for (int i = 0; i < grp.count; ++i) {
    const GemmProblem& p = grp.p[i];
    const GemmSchedule& s = grp.s[i];
    if ((p.K / kUnitK) % UG != 0) return cudaErrorInvalidValue;
    // Activations as [K/64][M][64]: one box {64, BA, 2 * UG} brings all
    // 64-wide K pieces of a unit, in the same shared-memory order as 2 * UG
    // 2-D boxes.
    int act_3d = 1;
    if (encode_tmap_3d(&g.tm[i][0], kActType, p.A, 64, p.M, p.K / 64, p.K * 2, 128, 64, BA,
                       2 * UG, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS) {
      act_3d = 0;
      if (encode_tmap_2d(&g.tm[i][0], kActType, p.A, p.K, p.M, p.K * 2, 64, BA,
                         CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    }
    // tiled code storage viewed as rows of 64 bytes (INT4) or 128 bytes
    // (INT8): tile (tn, g) is rows (tn * K/128 + g) * 128 .. + 127; a unit's
    // UG tiles are one box
    const uint64_t w_rows =
        static_cast<uint64_t>((p.N + kTileW - 1) / kTileW) * (p.K / kUnitK) * kTileW;
    constexpr uint32_t kRowBytes = wf_bits(WF) * 16;
    if (encode_tmap_2d(&g.tm[i][1], CU_TENSOR_MAP_DATA_TYPE_UINT8, p.packed, kRowBytes, w_rows,
                       kRowBytes, kRowBytes, kTileW * UG,
                       wf_bits(WF) == 4 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B) !=
        CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    if constexpr (wf_fp4(WF)) {
      // block-scale bytes [K/32 or K/16][N]: a unit's blocks for 128 rows
      // are one box {128, UG * blocks per group}
      if (p.tensor_scale == nullptr && WF == kFmtNvfp4) return cudaErrorInvalidValue;
      if (encode_tmap_2d(&g.tm[i][2], CU_TENSOR_MAP_DATA_TYPE_UINT8, p.scales, p.N,
                         p.K / kUnitK * wf_blocks(WF), p.N, kTileW, UG * wf_blocks(WF),
                         CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    } else {
      if (encode_tmap_2d(&g.tm[i][2], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, p.scales, p.N,
                         p.K / kGroup, p.N * 2, kTileW, UG, CU_TENSOR_MAP_SWIZZLE_NONE) !=
          CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    }

    Args& a = g.a[i];
    a.M = static_cast<int>(p.M);
    a.N = static_cast<int>(p.N);
    a.K = static_cast<int>(p.K);
    a.KB = static_cast<int>(p.K / kUnitK / UG);   // units per tile
    a.n_tiles = static_cast<int>((p.N + kTileW - 1) / kTileW);
    a.dp_tiles = s.dp_tiles;
    a.sk_units = static_cast<int>(s.sk_units);
    a.act_3d = act_3d;
    a.csk = s.cluster > 1 ? s.cluster : 0;
    a.sw = SW && p.swiglu ? 1 : 0;
    // two units per producer: deeper early copies sit ahead of the first
    // activation copy in the TMA queue and delay the start (measured)
    a.prefetch_w = p.weights_static ? 4 : 0;
    {
      // M-tail (dequant mode): the last activation tile's MMAs cover its
      // rows rounded up to 16 (a valid kind::f16 N for 128-row MMAs)
      const int m_tiles = static_cast<int>((p.M + BA - 1) / BA);
      const int rows = static_cast<int>(p.M) - (m_tiles - 1) * BA;
      const int tn = (rows + 15) / 16 * 16;
      a.tail_n = tn < BA ? tn : BA;
      a.tail_tile0 = (!GRP && tn < BA) ? (m_tiles - 1) * a.n_tiles : 0x7FFFFFFF;
    }
    a.scales = static_cast<const __half*>(p.scales);
    a.out_scale = p.tensor_scale;
    a.bias = static_cast<const uint16_t*>(p.bias);
    a.Y = static_cast<uint16_t*>(p.Y);
    a.counters = p.counters != nullptr ? p.counters : static_cast<uint32_t*>(p.workspace);
    a.ws = p.partials != nullptr
               ? p.partials
               : reinterpret_cast<float*>(static_cast<uint8_t*>(p.workspace) + kCounterBytes);
    a.err = p.error_word;
    a.timeout_ns = p.timeout_ns;
    g.cta_start[i] = start;
    start += s.grid;
  }
  g.cta_start[grp.count] = start;
  g.count = grp.count;

  // cluster split-K: one problem, its grid a whole number of clusters
  const int cluster = grp.s[0].cluster > 1 ? grp.s[0].cluster : 0;
  if (cluster > 0 && (grp.count != 1 || start % cluster != 0 || cluster > 8))
    return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(start));
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (use_pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (cluster > 0) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, kernel, g);
}

// The compiled configurations: {act_tile, lanes, group_scale, stages,
// unit_groups}.
#define W4A16_GEMM_INSTANCES(X) \
  X(16, 2, true, 16, 1)         \
  X(32, 2, true, 12, 1)         \
  X(64, 2, true, 8, 1)          \
  X(16, 2, false, 16, 1)        \
  X(32, 2, false, 12, 1)        \
  X(64, 2, false, 8, 1)         \
  X(128, 2, false, 4, 1)        \
  X(64, 1, false, 8, 1)         \
  X(128, 1, false, 5, 1)        \
  X(256, 1, false, 3, 1)        \
  X(16, 2, true, 8, 2)          \
  X(16, 2, false, 8, 2)         \
  X(32, 2, false, 6, 2)         \
  X(64, 2, false, 4, 2)

// INT8 weights (bf16 activations, single problems): {act_tile, lanes,
// group_scale, stages, unit_groups}.
#define W8A16_GEMM_INSTANCES(X) \
  X(16, 2, true, 10, 1)         \
  X(32, 2, true, 8, 1)          \
  X(64, 2, false, 6, 1)         \
  X(128, 1, false, 4, 1)        \
  X(256, 1, false, 2, 1)        \
  X(256, 1, false, 130, 1)

// FP4 weights (MXFP4 or NVFP4, bf16 activations, single problems; dequant
// mode only): {act_tile, lanes, group_scale, stages, unit_groups}.
#define FP4A16_GEMM_INSTANCES(X) \
  X(16, 2, false, 16, 1)         \
  X(32, 2, false, 12, 1)         \
  X(64, 2, false, 8, 1)          \
  X(128, 1, false, 5, 1)         \
  X(256, 1, false, 3, 1)         \
  X(16, 2, false, 8, 2)

template <int WF>
cudaError_t launch_gemm_tc_fp4_typed(const GemmKernelConfig& c, const GemmGroup& grp,
                                     bool use_pdl, cudaStream_t stream) {
#define FP4A16_LAUNCH_CASE(BA, L, GRP, ST, UG)                                   \
  if (c.act_tile == BA && c.lanes == L && c.group_scale == GRP && c.stages == ST && \
      c.unit_groups == UG && c.weight_format == WF)                                 \
    return launch_instance<BA, L, GRP, ST, UG, WF, false, 1>(grp, use_pdl, stream);
  FP4A16_GEMM_INSTANCES(FP4A16_LAUNCH_CASE)
#undef FP4A16_LAUNCH_CASE
  return cudaErrorInvalidConfiguration;
}

// (a template, so that only the unit that calls it compiles these kernels)
template <int WF>
cudaError_t launch_gemm_tc_w8_typed(const GemmKernelConfig& c, const GemmGroup& grp, bool use_pdl,
                                    cudaStream_t stream) {
  static_assert(WF == kFmtInt8, "INT8 weights");
#define W8A16_LAUNCH_CASE(BA, L, GRP, ST, UG)                                    \
  if (c.act_tile == BA && c.lanes == L && c.group_scale == GRP && c.stages == ST && \
      c.unit_groups == UG && c.weight_format == kFmtInt8)                                    \
    return launch_instance<BA, L, GRP, ST, UG, kFmtInt8, false, 1>(grp, use_pdl, stream);
  W8A16_GEMM_INSTANCES(W8A16_LAUNCH_CASE)
#undef W8A16_LAUNCH_CASE
  return cudaErrorInvalidConfiguration;
}

// All compiled configurations of one activation type and group size (SW:
// the SwiGLU epilogue).
template <bool F16, int G, bool SW = false>
cudaError_t launch_gemm_tc_typed(const GemmKernelConfig& c, const GemmGroup& grp, bool use_pdl,
                                 cudaStream_t stream) {
#define W4A16_LAUNCH_CASE(BA, L, GRP, ST, UG)                                    \
  if (c.act_tile == BA && c.lanes == L && c.group_scale == GRP && c.stages == ST && \
      c.unit_groups == UG && c.weight_format == kFmtInt4)                                    \
    return launch_instance<BA, L, GRP, ST, UG, kFmtInt4, F16, G, SW>(grp, use_pdl, stream);
  W4A16_GEMM_INSTANCES(W4A16_LAUNCH_CASE)
#undef W4A16_LAUNCH_CASE
  return cudaErrorInvalidConfiguration;
}

}  // namespace
}  // namespace w4a16
