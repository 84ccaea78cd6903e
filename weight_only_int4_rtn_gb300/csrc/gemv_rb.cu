// W4A16 GEMM for M <= 16: a row-block kernel with warp-level MMA (sm_103a),
// bf16 or fp16 activations.
//
// "Kernel dispatch and Humming quantization in PhyAI", section "Humming makes
// the separation useful": INT4 round-to-nearest weights, group 128 along K,
// BF16 (or FP16) activations; the packed layout runs only through the kernels
// that understand it.  At M <= 16 the GEMM does at most 32 flops per 0.52
// bytes of codes and scales: it is bound by streaming the weight from HBM,
// and the tcgen05 path's fixed costs per 128 x 128 unit (the converted
// operand's TMEM round trip, MMA issue and commit, barrier hand-offs between
// roles) are what limits it there.  This kernel has no pipeline roles: every
// warp feeds itself, converts its codes in registers and multiplies them
// with synchronous warp MMAs (mma.sync m16n8k16, fp32 accumulators), whose
// 8 columns take up to 8 activation rows at no extra cost; for M = 9 .. 16
// each converted code fragment feeds two MMAs (activation rows 0-7 and
// 8-15), so the conversion, the kernel's main cost, is shared by 16 rows.
//
// Work split.  An item is one row block (RB = 32 consecutive weight rows of
// one 128-row storage tile) times up to two groups of 128 codes along K (one
// for M = 8): 2 KiB of contiguous codes per group in the tiled storage, the
// 32 rows' scales, the groups' activations.  Persistent form: the grid is
// the resident CTAs (or fewer), teams of WK warps (1, 2, 4, 8) take row
// blocks round-robin and split each row block's K range into WK equal runs
// of groups; the host picks WK so that the busiest SM has the least work.
// Cluster form, for shapes with few row blocks and long K: one CTA-wide team
// per (row block, cluster rank), the K range split over the S CTAs of a
// thread-block cluster and summed through distributed shared memory.
// Grouped launches: up to 8 independent problems, problem p on its own
// sub-grid of CTAs in the persistent form (one launch, one head, for the
// projections of a decode step).
//
// Streaming.  Each warp owns a ring of two shared-memory stages (three for
// M <= 16, whose CTA has an SM to itself) of one item each, whose copies
// complete on a per-stage mbarrier, so the next item is
// in flight while one is computed, without holding a register: the codes
// and scales by non-tensor bulk copies (cp.async.bulk), the activations by
// one bulk copy per row for M <= 2 and by one tensor copy per group for all
// rows for M <= 4 and 8 (each copy instruction costs the issuing warp time,
// and per-row copies made M = 8 the slowest form).  With static weights the
// first stages' codes and scales are requested before the wait for the
// previous kernel (whose output may be A).  Waits are time-bounded: a warp
// that gives up records the error, walks its remaining items without
// waiting (so its team's barriers still match) and lets its copies in
// flight land before it exits.
//
// Arithmetic.  The row block is two 16-row MMA tiles (A: weight rows x k),
// the activations are B (k x 8 columns, column m = activation row m).  A
// lane (gq, tq) = (lane / 4, lane % 4) reads, of its rows gq and gq + 8, the
// 32 codes k = 32 tq .. 32 tq + 31 with one 16-byte load per row.  One
// shift and one AND-XOR turn nibbles s and s + 4 of a code word into two
// 16-bit values x + q under the exponent whose unit is bit 0 (sign bit
// flipped: n ^ 8 = q + 8), x = 136 for bf16 and 1032 for fp16, both exact;
// each word gives the A fragments of two MMAs.  The MMA's k order within a
// group is a permutation of the storage's; B takes the activations in the
// same order (byte permutes of the 16-byte activation loads), so each
// product is unchanged.  Products of x + q (at most 11 significant bits)
// with an activation are exact in fp32.  An MMA of an all-ones A gives the
// group's activation sums per column, and x times those is taken off before
// the group's fp32 scale multiplies the partial into the row's total (for
// M <= 16 one MMA of the activations as A, rows gq and gq + 8 = activation
// rows gq and 8 + gq, against an all-ones B gives the sums of all 16 rows;
// each lane fetches its columns' sums from the lanes that hold them).  With
// fp16 activations the 10-bit mantissa also holds a nibble at bits 4-7: the
// MMAs of a word split into a class of nibbles 0, 2, 4, 6 (1032 + q) and one
// of nibbles 1, 3, 5, 7 (1152 + 16 q under 0x6480, exact), so one shift by 8
// per word serves both, and the second class's partial, less 1152 times its
// activation sum, is scaled by 1/16 (exact) before the group scale.
//
// Reduction.  A team's warps add their totals in k order through shared
// memory after a named barrier; with a cluster the CTAs' sums are added in
// rank order; the bias is added in fp32 and Y rounded once.  The result
// does not depend on timing.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"
#include "waits.cuh"
#include "warp_mma.cuh"

namespace w4a16 {
namespace {

constexpr int kRbWarps = kRbWarpsPerCta;
constexpr int kRbRows = 32;       // rows per block: two 16-row MMA tiles

struct RbArgs {
  CUtensorMap amap;        // M >= 4: A as [M][K], boxes of 136 values x MT rows
  const uint16_t* A;       // [M, K] activation type
  const uint8_t* packed;   // tiled codes
  const __half* scales;    // [K/128, N]
  const uint16_t* bias;    // [N] or null
  uint16_t* Y;             // [M, N]
  int M, N, K, KB;         // KB: groups along K
  int NB;                  // row blocks
  int team;                // warps that split one row block's K range (1, 2, 4, 8)
  int cluster;             // CTAs of a cluster splitting K (1: none; then team = 8)
  int static_w;            // codes and scales are not written by the kernel before
                           // this one: the first copies of them may precede the
                           // grid-dependency wait
  uint32_t* err;           // device error word
  uint64_t timeout_ns;     // limit of one wait
};

// A launch: G problems, problem p on CTAs cta_start[p] .. cta_start[p+1]-1
// (G = 1: a single problem; the cluster form only then).
template <int G>
struct RbLaunch {
  RbArgs p[G];
  int cta_start[G + 1];
  int count;
};

// MT: activation rows (M <= MT; the MMA's 8 columns, twice for MT = 16).
// An item holds up to UG groups of one row block (2 for M <= 4; 1 for
// M = 8 and 16, whose activation rows fill the shared memory).  One stage holds the item's codes (2 KiB per
// group), its rows' scales (64 B per group) and MT activation rows of the
// item's groups.  M <= 2: the codes, the scales, then each activation row's
// UG groups (contiguous in A: 256 B per group), padded by 16 B for M = 2.
// M <= 4, 8 and 16 (kTensor): per group, the activations as one tensor copy
// of MT rows x 136 values (272-byte rows: the lanes' 16-byte loads of
// different rows fall in different bank groups; rows >= M and values past K
// are zero) followed by the group's scales, then the codes.
template <int MT>
struct RbCfg {
  static constexpr bool kTensor = MT >= 4;
  static constexpr int kUG = MT <= 4 ? 2 : 1;
  static constexpr int kCodeBytes = kRbRows * 64;                 // one group
  static constexpr int kScaleBytes = kRbRows * 2;                 // one group
  static constexpr int kActRow = kTensor ? 272 : kUG * kGroup * 2 + (MT > 1 ? 16 : 0);
  static constexpr int kActBox = MT * 272;                        // one group's tensor copy
  static constexpr int kGrpBytes = (kActBox + kScaleBytes + 127) / 128 * 128;
  static constexpr int kCodeOff = kTensor ? kUG * kGrpBytes : 0;
  static constexpr int kScaleOff = kTensor ? kActBox : kUG * kCodeBytes;
  static constexpr int kScaleStride = kTensor ? kGrpBytes : kScaleBytes;
  static constexpr int kActOff = kTensor ? 0 : kScaleOff + kUG * kScaleBytes;
  static constexpr int kActGroup = kTensor ? kGrpBytes : kGroup * 2;   // to group gi's values
  static constexpr int kStage =
      kTensor ? (kCodeOff + kUG * kCodeBytes + 127) / 128 * 128 : kActOff + MT * kActRow;
  static constexpr int kNT = MT > 8 ? 2 : 1;                      // MMA column tiles
  // Two CTAs an SM (registers <= 128, shared memory <= 113 KB) with two
  // stages a warp; MT = 16 (32 KB of team totals, 6.5 KB stages, about 165
  // registers): one CTA an SM with three stages a warp (48 KiB of codes in
  // flight per SM against 64 KiB with two CTAs)
  static constexpr int kCtasPerSm = MT > 8 ? 1 : 2;
  static constexpr int kDepth = MT > 8 ? 3 : 2;                   // stages per warp
  static constexpr int kBarOff = kRbWarps * kDepth * kStage;
  static constexpr int kSmem = kBarOff + kRbWarps * kDepth * 8 + 128;   // + alignment of the base
  static constexpr int kStatic = kRbWarps * 2 * kRbRows * MT * 4 + kRbRows * MT * 4 + 16;
  static_assert(kActOff % 16 == 0 && kCodeOff % 16 == 0 && kStage % 16 == 0,
                "bulk-copy destinations 16-byte aligned");
  static_assert(!kTensor || (kGrpBytes % 128 == 0 && kStage % 128 == 0),
                "tensor-copy destinations 128-byte aligned");
  static_assert(MT == 1 || MT == 2 || MT == 4 || MT == 8 || MT == 16,
                "the MMA has 8 columns, taken once or twice");
  static_assert(kCtasPerSm * (kSmem + kStatic + 1024) <= 228 * 1024, "shared memory of an SM");
};

// Walks a warp's items for the copies: the row blocks of its team (rb = T,
// T + TT, ...) and, in each, the warp's groups k0 .. k1 - 1 in items of up
// to UG groups, with the item's copy sources and transaction bytes
// (stepped, not recomputed, inside a row block).
template <int UG>
struct RbWalk {
  int rb, g, ng;             // row block, first group, groups in the item
  const uint8_t* codes;      // the first group's kRbRows x 64 bytes
  const __half* scales;      // the first group's nv values
  const uint16_t* act;       // row 0's values of the item's groups
  uint32_t scale_bytes;      // one group's
  __device__ bool valid(int NB) const { return rb < NB; }
  // the item's transaction bytes, given one group's activation bytes
  __device__ uint32_t bytes(uint32_t act_group) const {
    return static_cast<uint32_t>(ng) * (kRbRows * 64 + scale_bytes + act_group);
  }
  __device__ void start(const RbArgs& a, int rb_, int k0, int k1) {
    rb = rb_;
    g = k0;
    ng = k1 - k0 < UG ? k1 - k0 : UG;
    if (rb >= a.NB) return;
    const int r0 = rb * kRbRows;
    const int tn = r0 / kTileW;
    const int nv = a.N - r0 < kRbRows ? a.N - r0 : kRbRows;   // a multiple of 8
    codes = a.packed + ((static_cast<int64_t>(tn) * a.KB + k0) * kTileW + (r0 - tn * kTileW)) * 64;
    scales = a.scales + static_cast<int64_t>(k0) * a.N + r0;
    act = a.A + static_cast<int64_t>(k0) * kGroup;
    scale_bytes = 2u * static_cast<uint32_t>(nv);
  }
  __device__ void next(const RbArgs& a, int k0, int k1, int TT) {
    g += ng;
    if (g >= k1) {
      start(a, rb + TT, k0, k1);
    } else {
      codes += static_cast<int64_t>(ng) * kTileW * 64;
      scales += static_cast<int64_t>(ng) * a.N;
      act += ng * kGroup;
      ng = k1 - g < UG ? k1 - g : UG;
    }
  }
};

template <int MT, bool F16, int G>
__global__ void __launch_bounds__(kRbWarps * 32, RbCfg<MT>::kCtasPerSm)
    gemv_rb_kernel(const __grid_constant__ RbLaunch<G> L) {
  using C = RbCfg<MT>;
  constexpr int NT = C::kNT;
  // this CTA's problem and its index in the problem's sub-grid
  int prob = 0;
  if constexpr (G > 1) {
    while (prob + 1 < L.count && static_cast<int>(blockIdx.x) >= L.cta_start[prob + 1]) ++prob;
  }
  const RbArgs& g = L.p[prob];
  const int cta = static_cast<int>(blockIdx.x) - L.cta_start[prob];
  const int ctas = L.cta_start[prob + 1] - L.cta_start[prob];
  constexpr int D = C::kDepth;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                             ~static_cast<uintptr_t>(127));
  // per warp, per row-block parity: its rows' totals (a team's flush)
  __shared__ float tbuf[kRbWarps][2][kRbRows][MT];
  __shared__ float csum[kRbRows][MT];   // cluster split: the CTA's totals
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, tq = lane & 3;        // MMA fragment row group, column pair
  const int WK = g.team, S = g.cluster;
  const int tpc = kRbWarps / WK;                  // teams per CTA
  const int team = warp / WK, wt = warp - team * WK;

  // the team's first row block and stride; with a cluster split the CTA is
  // one team on one row block and its rank takes a share of K
  int T, TT, rank = 0, cg0 = 0, cg1 = g.KB;
  if (S > 1) {
    T = cta / S;
    rank = cta - T * S;
    TT = g.NB;
    cg0 = (rank * g.KB) / S;
    cg1 = ((rank + 1) * g.KB) / S;
  } else {
    T = cta * tpc + team;
    TT = ctas * tpc;
  }
  const int k0 = cg0 + (wt * (cg1 - cg0)) / WK;
  const int k1 = cg0 + ((wt + 1) * (cg1 - cg0)) / WK;

  uint8_t* ring = smem + warp * D * C::kStage;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kBarOff) + warp * D;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    if constexpr (C::kTensor) ptx::prefetch_tmap(&g.amap);
  }
  if (lane == 0) {
    for (int s = 0; s < D; ++s) ptx::mbar_init(&full[s], 1);
    ptx::fence_mbar_init();
  }
  __syncthreads();
  const WaitCtx wc{g.err, g.timeout_ns, &abort_flag};

  // an item's copies, issued by lane 0: weights (each group's codes and the
  // valid rows' scales) and activations (M <= 2: each of the M rows' values
  // of the item's groups, one contiguous run; else one tensor copy of MT
  // rows per group)
  constexpr int UG = C::kUG;
  using Walk = RbWalk<UG>;
  auto issue_w = [&](const Walk& it, uint8_t* st, uint64_t* bar) {
    ptx::mbar_arrive_expect_tx(
        bar, it.bytes(C::kTensor ? static_cast<uint32_t>(C::kActBox) : static_cast<uint32_t>(g.M) * kGroup * 2));
    for (int gi = 0; gi < it.ng; ++gi) {
      ptx::bulk_g2s(st + C::kCodeOff + gi * C::kCodeBytes, it.codes + static_cast<int64_t>(gi) * kTileW * 64,
                    C::kCodeBytes, bar);
      ptx::bulk_g2s(st + C::kScaleOff + gi * C::kScaleStride, it.scales + static_cast<int64_t>(gi) * g.N,
                    it.scale_bytes, bar);
    }
  };
  auto issue_a = [&](const Walk& it, uint8_t* st, uint64_t* bar) {
    const uint32_t bytes = static_cast<uint32_t>(it.ng) * kGroup * 2;
    if constexpr (C::kTensor) {
      for (int gi = 0; gi < it.ng; ++gi)
        ptx::tma_load_2d(st + gi * C::kGrpBytes, &g.amap, bar, (it.g + gi) * kGroup, 0);
    } else if constexpr (MT == 1) {
      ptx::bulk_g2s(st + C::kActOff, it.act, bytes, bar);
    } else {
      for (int m = 0; m < g.M; ++m)
        ptx::bulk_g2s(st + C::kActOff + m * C::kActRow, it.act + static_cast<int64_t>(m) * g.K, bytes, bar);
    }
  };

  // (the launch guarantees KB >= team x cluster: no warp's range is empty)
  const int first = k1 > k0 ? T : g.NB;
  Walk pre;
  pre.start(g, first, k0, k1);
  // the first D items; with static weights their codes and scales are
  // requested before the wait for the previous kernel
  int issued = 0;
  if (lane == 0 && g.static_w) {
    Walk q = pre;
    for (int s = 0; s < D && q.valid(g.NB); ++s, q.next(g, k0, k1, TT))
      issue_w(q, ring + s * C::kStage, &full[s]);
  }
  ptx::grid_dependency_wait();
  ptx::grid_launch_dependents();
  for (; issued < D && pre.valid(g.NB); ++issued, pre.next(g, k0, k1, TT)) {
    if (lane == 0) {
      if (!g.static_w) issue_w(pre, ring + issued * C::kStage, &full[issued]);
      issue_a(pre, ring + issued * C::kStage, &full[issued]);
    }
  }

  // the lane's totals of the block's two 16-row tiles: rows gq, gq + 8 of
  // tile tau, columns (activation rows) 8 nt + 2 tq, 8 nt + 2 tq + 1
  float acc[2][NT][4] = {};

  // One item.  Code word j of a row (k = 32 tq + 8 j ..) gives the A
  // fragments of MMAs 2 j + h, h = 0, 1: fragment columns (2 tq, 2 tq + 1)
  // <- k = 32 tq + 8 j + 2 h + (0, 4), columns (2 tq + 8, 2 tq + 9) <- + (1,
  // 5); B's fragment rows take the same k from the activations.
  auto compute_group = [&](uint32_t st, int gi) {
    constexpr uint32_t kOne = wmma16::CodeOffset<F16>::kOnes;
    constexpr float kOff = wmma16::CodeOffset<F16>::kOff;
    // B fragments of column tile nt: activation row 8 nt + gq (for MT < 8
    // rows >= MT repeat row MT - 1: columns >= M are never stored)
    uint32_t b[NT][8][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int mrow = NT > 1 ? 8 * nt + gq : (gq < MT ? gq : MT - 1);
      uint32_t u[16];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 v =
            ptx::lds128(st + C::kActOff + mrow * C::kActRow + gi * C::kActGroup + 64 * tq + 16 * i);
        u[4 * i] = v.x;
        u[4 * i + 1] = v.y;
        u[4 * i + 2] = v.z;
        u[4 * i + 3] = v.w;
      }
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if constexpr (F16) {
            // class h of word j: k = k0 + h + (0, 4) and k0 + h + (2, 6)
            b[nt][2 * j + h][0] = ptx::prmt(u[4 * j], u[4 * j + 2], h ? 0x7632u : 0x5410u);
            b[nt][2 * j + h][1] = ptx::prmt(u[4 * j + 1], u[4 * j + 3], h ? 0x7632u : 0x5410u);
          } else {
            b[nt][2 * j + h][0] = ptx::prmt(u[4 * j + h], u[4 * j + h + 2], 0x5410u);
            b[nt][2 * j + h][1] = ptx::prmt(u[4 * j + h], u[4 * j + h + 2], 0x7632u);
          }
        }
    }
    // the group's activation sums over the k of class h (the MMAs 2 j + h)
    // for the lane's columns: sum[h][nt][c] for column 8 nt + 2 tq + c; the
    // MMAs run as independent accumulation chains, added at the end
    float sum[2][NT][2];
    if constexpr (NT == 1) {
      float sa[4] = {}, sb[4] = {};
#pragma unroll
      for (int mu = 0; mu < 8; mu += 2) {
        wmma16::mma16816<F16>(sa, kOne, kOne, kOne, kOne, b[0][mu][0], b[0][mu][1]);
        wmma16::mma16816<F16>(sb, kOne, kOne, kOne, kOne, b[0][mu + 1][0], b[0][mu + 1][1]);
      }
      sum[0][0][0] = sa[0];
      sum[0][0][1] = sa[1];
      sum[1][0][0] = sb[0];
      sum[1][0][1] = sb[1];
    } else {
      // the activations as A (row gq: activation row gq, row gq + 8:
      // activation row 8 + gq), all-ones B: every column holds the row sums;
      // activation row 8 nt + 2 tq + c is row 2 tq + c (+ 8) of lane
      // 4 (2 tq + c)
      float sa[4] = {}, sb[4] = {};
#pragma unroll
      for (int mu = 0; mu < 8; mu += 2) {
        wmma16::mma16816<F16>(sa, b[0][mu][0], b[1][mu][0], b[0][mu][1], b[1][mu][1], kOne, kOne);
        wmma16::mma16816<F16>(sb, b[0][mu + 1][0], b[1][mu + 1][0], b[0][mu + 1][1], b[1][mu + 1][1],
                              kOne, kOne);
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int src = 4 * (2 * tq + c);
          sum[0][nt][c] = __shfl_sync(0xFFFFFFFFu, sa[2 * nt], src);
          sum[1][nt][c] = __shfl_sync(0xFFFFFFFFu, sb[2 * nt], src);
        }
    }
    uint32_t W[2][2][4];   // [tile][row gq, gq + 8][word]
#pragma unroll
    for (int tau = 0; tau < 2; ++tau)
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const uint4 v =
            ptx::lds128(st + C::kCodeOff + gi * C::kCodeBytes + (16 * tau + 8 * half + gq) * 64 + 16 * tq);
        W[tau][half][0] = v.x;
        W[tau][half][1] = v.y;
        W[tau][half][2] = v.z;
        W[tau][half][3] = v.w;
      }
    float d[2][2][NT][4] = {};   // [tile][h][column tile]
    if constexpr (F16) {
      // fp16 (10 mantissa bits): nibbles s and s + 4 as 1032 + q (class 0,
      // bits 0-3 of each half) or 16 (72 + q) = 1152 + 16 q (class 1, bits
      // 4-7 under 0x6480), so one shift by 8 serves nibbles 2, 3, 6, 7;
      // class 1's products are exact and its partial is scaled by 1/16
      constexpr uint32_t kLoMask = 0x000F000Fu, kHiMask = 0x00F000F0u;
      constexpr uint32_t kLoMagic = 0x64086408u, kHiMagic = 0x64806480u;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t w[2][2], w8[2][2];
#pragma unroll
        for (int tau = 0; tau < 2; ++tau)
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            w[tau][half] = W[tau][half][j];
            w8[tau][half] = W[tau][half][j] >> 8;
          }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t mask = h ? kHiMask : kLoMask, magic = h ? kHiMagic : kLoMagic;
#pragma unroll
          for (int tau = 0; tau < 2; ++tau) {
            const uint32_t a0 = ptx::and_xor(w[tau][0], mask, magic);
            const uint32_t a1 = ptx::and_xor(w[tau][1], mask, magic);
            const uint32_t a2 = ptx::and_xor(w8[tau][0], mask, magic);
            const uint32_t a3 = ptx::and_xor(w8[tau][1], mask, magic);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
              wmma16::mma16816<F16>(d[tau][h][nt], a0, a1, a2, a3, b[nt][2 * j + h][0], b[nt][2 * j + h][1]);
          }
        }
      }
#pragma unroll
      for (int tau = 0; tau < 2; ++tau) {
        const int r = 16 * tau + gq;
        const float s0 = wmma16::lds_scale(st + C::kScaleOff + gi * C::kScaleStride + 2 * r);
        const float s1 = wmma16::lds_scale(st + C::kScaleOff + gi * C::kScaleStride + 2 * (r + 8));
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float q = fmaf(0.0625f, fmaf(-1152.0f, sum[1][nt][e & 1], d[tau][1][nt][e]),
                                 fmaf(-1032.0f, sum[0][nt][e & 1], d[tau][0][nt][e]));
            acc[tau][nt][e] = fmaf(e < 2 ? s0 : s1, q, acc[tau][nt][e]);
          }
      }
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int tau = 0; tau < 2; ++tau) {
            const uint32_t a0 = wmma16::code_pair16<F16>(W[tau][0][j], 2 * h);
            const uint32_t a1 = wmma16::code_pair16<F16>(W[tau][1][j], 2 * h);
            const uint32_t a2 = wmma16::code_pair16<F16>(W[tau][0][j], 2 * h + 1);
            const uint32_t a3 = wmma16::code_pair16<F16>(W[tau][1][j], 2 * h + 1);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
              wmma16::mma16816<F16>(d[tau][h][nt], a0, a1, a2, a3, b[nt][2 * j + h][0], b[nt][2 * j + h][1]);
          }
#pragma unroll
      for (int tau = 0; tau < 2; ++tau) {
        const int r = 16 * tau + gq;
        const float s0 = wmma16::lds_scale(st + C::kScaleOff + gi * C::kScaleStride + 2 * r);
        const float s1 = wmma16::lds_scale(st + C::kScaleOff + gi * C::kScaleStride + 2 * (r + 8));
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const float sum0 = sum[0][nt][0] + sum[1][nt][0], sum1 = sum[0][nt][1] + sum[1][nt][1];
          acc[tau][nt][0] = fmaf(s0, fmaf(-kOff, sum0, d[tau][0][nt][0] + d[tau][1][nt][0]), acc[tau][nt][0]);
          acc[tau][nt][1] = fmaf(s0, fmaf(-kOff, sum1, d[tau][0][nt][1] + d[tau][1][nt][1]), acc[tau][nt][1]);
          acc[tau][nt][2] = fmaf(s1, fmaf(-kOff, sum0, d[tau][0][nt][2] + d[tau][1][nt][2]), acc[tau][nt][2]);
          acc[tau][nt][3] = fmaf(s1, fmaf(-kOff, sum1, d[tau][0][nt][3] + d[tau][1][nt][3]), acc[tau][nt][3]);
        }
      }
    }
  };

  // The row block's totals: with a team of one and no cluster straight to Y
  // (bias added in fp32, one rounding); else through shared memory, the
  // team's warps in k order, into Y or (cluster split) csum.
  int nflush = 0;
  auto flush = [&](int rb) {
    const int r0 = rb * kRbRows;
    if (WK == 1 && S == 1) {
#pragma unroll
      for (int tau = 0; tau < 2; ++tau)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int n = r0 + 16 * tau + gq + (e >= 2 ? 8 : 0);
            const int m = 8 * nt + 2 * tq + (e & 1);
            if (m < g.M && n < g.N) {
              float t = acc[tau][nt][e];
              if (g.bias != nullptr) t += wmma16::act_to_f32<F16>(g.bias[n]);
              g.Y[static_cast<int64_t>(m) * g.N + n] = wmma16::f32_to_out<F16>(t);
            }
          }
    } else {
#pragma unroll
      for (int tau = 0; tau < 2; ++tau)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int m = 8 * nt + 2 * tq + (e & 1);
            if (m < MT) tbuf[warp][nflush & 1][16 * tau + gq + (e >= 2 ? 8 : 0)][m] = acc[tau][nt][e];
          }
      ptx::named_barrier_sync(1 + team, WK * 32);
      if (wt == 0) {
        for (int e = lane; e < kRbRows * MT; e += 32) {
          const int row = e / MT, m = e - row * MT;
          float t = 0.0f;
          for (int w = 0; w < WK; ++w) t += tbuf[team * WK + w][nflush & 1][row][m];
          if (S > 1) {
            csum[row][m] = t;
          } else {
            const int n = r0 + row;
            if (n < g.N && m < g.M) {
              if (g.bias != nullptr) t += wmma16::act_to_f32<F16>(g.bias[n]);
              g.Y[static_cast<int64_t>(m) * g.N + n] = wmma16::f32_to_out<F16>(t);
            }
          }
        }
      }
    }
#pragma unroll
    for (int tau = 0; tau < 2; ++tau)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[tau][nt][e] = 0.0f;
    ++nflush;
  };

  // the ring: item i in stage i % D; once computed, the stage takes item i + D
  bool ok = true;
  int s = 0;
  uint32_t phase = 0;
  int waited = 0;   // items whose copies have landed
  const uint32_t ring_u32 = ptx::smem_u32(ring);
  uint32_t st = ring_u32;
  const int per_block = (k1 - k0 + UG - 1) / UG;   // items per row block
  const int last_ng = k1 - k0 - (per_block - 1) * UG;  // groups in a row block's last item
  int left = per_block;   // items left in the current row block
#pragma unroll 1
  for (int rb = first; rb < g.NB;) {
    if (ok) {
      if (wait_warp(&full[s], phase, wc))
        ++waited;
      else
        ok = false;
    }
    compute_group(st, 0);
    if (UG > 1 && (left > 1 || last_ng > 1)) compute_group(st, 1);
    if (ok && pre.valid(g.NB)) {
      // the lanes' reads of the stage have returned (their values are
      // consumed above): the copy may overwrite it
      __syncwarp();
      if (lane == 0) {
        issue_w(pre, ring + s * C::kStage, &full[s]);
        issue_a(pre, ring + s * C::kStage, &full[s]);
      }
      pre.next(g, k0, k1, TT);
      ++issued;
    }
    if (--left == 0) {
      flush(rb);
      left = per_block;
      rb += TT;
    }
    st += C::kStage;
    if (++s == D) {
      s = 0;
      st = ring_u32;
      phase ^= 1u;
    }
  }
  if (!ok && lane == 0) {
    // gave up: the copies in flight land before the CTA exits
    for (int i = waited; i < issued; ++i) {
      const int si = i % D;
      const uint32_t ph = static_cast<uint32_t>(i / D) & 1u;
      const uint64_t t0 = ptx::globaltimer_ns();
      while (!ptx::mbar_try_wait(&full[si], ph))
        if (ptx::globaltimer_ns() - t0 > g.timeout_ns) break;
    }
  }

  if (S > 1) {
    // CTAs of the cluster in rank (k) order; rank q stores rows q, q + S, ...
    ptx::cluster_sync();
    const uint32_t base = ptx::smem_u32(&csum[0][0]);
    const int r0 = T * kRbRows;
    for (int e = threadIdx.x; e < kRbRows * MT; e += blockDim.x) {
      const int row = e / MT, m = e - row * MT;
      if (row % S != rank) continue;
      const int n = r0 + row;
      if (n >= g.N || m >= g.M) continue;
      float t = 0.0f;
      for (int q = 0; q < S; ++q) t += ptx::ld_dsmem_f32(base + 4u * static_cast<uint32_t>(e), q);
      if (g.bias != nullptr) t += wmma16::act_to_f32<F16>(g.bias[n]);
      g.Y[static_cast<int64_t>(m) * g.N + n] = wmma16::f32_to_out<F16>(t);
    }
    ptx::cluster_sync();   // every CTA's sums stay alive until read
  }
}

// One problem's kernel arguments under schedule s (false: the problem or
// the schedule is not one this kernel runs).
template <int MT, bool F16>
bool rb_args(const GemmProblem& p, const GemmSchedule& s, RbArgs& g) {
  using C = RbCfg<MT>;
  const int64_t blocks = (p.N + kRbRows - 1) / kRbRows;
  const int S = s.cluster > 1 ? s.cluster : 1;
  const int WK = s.team;
  const int64_t KB = p.K / kGroup;
  // every warp gets at least one group; a cluster split is one CTA-wide team
  // per row block
  if (p.M > MT || S > 8 || (WK != 1 && WK != 2 && WK != 4 && WK != 8) || KB < WK * S ||
      (S > 1 && (WK != kRbWarps || s.grid != blocks * S)) || s.grid < 1)
    return false;
  g = RbArgs{};
  g.A = static_cast<const uint16_t*>(p.A);
  g.packed = static_cast<const uint8_t*>(p.packed);
  g.scales = static_cast<const __half*>(p.scales);
  g.bias = static_cast<const uint16_t*>(p.bias);
  g.Y = static_cast<uint16_t*>(p.Y);
  g.M = static_cast<int>(p.M);
  g.N = static_cast<int>(p.N);
  g.K = static_cast<int>(p.K);
  g.KB = static_cast<int>(KB);
  g.NB = static_cast<int>(blocks);
  g.team = WK;
  g.cluster = S;
  g.static_w = p.weights_static ? 1 : 0;
  g.err = p.error_word;
  g.timeout_ns = p.timeout_ns;
  if constexpr (C::kTensor) {
    // A as [M][K]: a box of 136 values (one group and 8 more, which keep the
    // rows 272 bytes apart in shared memory) by MT rows, zero past K and M
    constexpr CUtensorMapDataType kActType =
        F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    if (encode_tmap_2d(&g.amap, kActType, p.A, p.K, p.M, p.K * 2, C::kActRow / 2, MT,
                       CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
      return false;
  }
  return true;
}

template <int MT, bool F16, int G>
cudaError_t launch_rb(const GemmGroup& grp, bool use_pdl, cudaStream_t stream) {
  using C = RbCfg<MT>;
  if (grp.count < 1 || grp.count > G) return cudaErrorInvalidValue;
  RbLaunch<G> L{};
  L.count = grp.count;
  int total = 0;
  for (int i = 0; i < grp.count; ++i) {
    if (!rb_args<MT, F16>(grp.p[i], grp.s[i], L.p[i])) return cudaErrorInvalidValue;
    // the cluster form (one cluster size per launch) takes a single problem
    if (grp.count > 1 && L.p[i].cluster > 1) return cudaErrorInvalidValue;
    L.cta_start[i] = total;
    total += grp.s[i].grid;
  }
  L.cta_start[grp.count] = total;
  const int S = L.p[0].cluster;
  auto kernel = gemv_rb_kernel<MT, F16, G>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static bool attr_set[64] = {};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(total));
  cfg.blockDim = dim3(kRbWarps * 32);
  cfg.dynamicSmemBytes = C::kSmem;
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
  return cudaLaunchKernelEx(&cfg, kernel, L);
}

template <int MT, bool F16>
cudaError_t launch_rb_any(const GemmGroup& grp, bool use_pdl, cudaStream_t stream) {
  return grp.count == 1 ? launch_rb<MT, F16, 1>(grp, use_pdl, stream)
                        : launch_rb<MT, F16, kMaxGemmGroup>(grp, use_pdl, stream);
}

}  // namespace

int gemv_rb_rows(int act_tile) {
  (void)act_tile;
  return kRbRows;
}

int gemv_rb_ctas_per_sm(int act_tile) {
  return act_tile > 8 ? RbCfg<16>::kCtasPerSm : RbCfg<8>::kCtasPerSm;
}

size_t gemv_rb_smem_bytes(int act_tile) {
  switch (act_tile) {
    case 1: return RbCfg<1>::kSmem;
    case 2: return RbCfg<2>::kSmem;
    case 4: return RbCfg<4>::kSmem;
    case 8: return RbCfg<8>::kSmem;
    case 16: return RbCfg<16>::kSmem;
    default: return 0;
  }
}

cudaError_t launch_gemv_rb(const GemmKernelConfig& c, const GemmGroup& grp, bool use_pdl,
                           cudaStream_t stream) {
  if (grp.count < 1 || grp.count > kMaxGemmGroup) return cudaErrorInvalidValue;
  for (int i = 0; i < grp.count; ++i) {
    // the fused epilogue is the tcgen05 path's; one activation type a launch
    if (grp.p[i].swiglu || grp.p[i].act_f16 != grp.p[0].act_f16) return cudaErrorInvalidValue;
  }
  const bool f16 = grp.p[0].act_f16;
  switch (c.act_tile) {
    case 1: return f16 ? launch_rb_any<1, true>(grp, use_pdl, stream) : launch_rb_any<1, false>(grp, use_pdl, stream);
    case 2: return f16 ? launch_rb_any<2, true>(grp, use_pdl, stream) : launch_rb_any<2, false>(grp, use_pdl, stream);
    case 4: return f16 ? launch_rb_any<4, true>(grp, use_pdl, stream) : launch_rb_any<4, false>(grp, use_pdl, stream);
    case 8: return f16 ? launch_rb_any<8, true>(grp, use_pdl, stream) : launch_rb_any<8, false>(grp, use_pdl, stream);
    case 16: return f16 ? launch_rb_any<16, true>(grp, use_pdl, stream) : launch_rb_any<16, false>(grp, use_pdl, stream);
    default: return cudaErrorInvalidConfiguration;
  }
}

}  // namespace w4a16
