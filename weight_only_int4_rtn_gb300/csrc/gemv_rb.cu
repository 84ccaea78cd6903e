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
// are what limits it.  This kernel has no pipeline roles: every warp feeds
// itself and converts its codes in registers.
//
// Work split.  An item is one row block (RB = 16 consecutive weight rows of
// one 128-row storage tile) times one group of 128 codes along K: 1 KiB of
// contiguous codes in the tiled storage, the 16 rows' scales, the group's
// activations.  Persistent form: the grid is the resident CTAs (or fewer),
// teams of WK warps (1, 2, 4, 8) take row blocks round-robin and split each
// row block's K range into WK equal runs of groups; the host picks WK so
// that the busiest warp has the fewest items.  Cluster form, for shapes
// with few row blocks and long K: one CTA-wide team per (row block, cluster
// rank), the K range split over the S CTAs of a thread-block cluster and
// summed through distributed shared memory.
//
// Streaming.  Each warp owns a ring of D shared-memory stages (one item
// each) filled by non-tensor bulk copies (cp.async.bulk) that complete on a
// per-stage mbarrier, so D items per warp are in flight without holding a
// register: 16 warps x D KiB per SM cover the HBM latency.  With static
// weights the first stages' codes and scales are requested before the wait
// for the previous kernel (whose output may be A).  Waits are time-bounded:
// a warp that gives up records the error, walks its remaining items without
// waiting (so its team's barriers still match) and lets its copies in
// flight land before it exits.
//
// Arithmetic.  A lane owns a chunk of CH = 16 codes (8 bytes of a 64-byte
// tile row) of RPL = 4 rows, r = lane / 8 + 4 j, and reads its activations
// once per item for those rows.  One shift of a code word puts two
// neighbouring nibbles at bits 12..15 and 16..19; one AND-XOR each places
// them under the exponent of 2048 (bits 12..15) or 128 (bits 16..19) with
// the nibble's sign bit flipped (n ^ 8 = q + 8), so a code of even k reads
// 2056 + q and one of odd k reads 136 + q, exactly: twelve operations per
// eight codes.  Products with a bf16 or fp16 activation are exact in fp32
// (at most 12 + 11 significant bits), and per chunk
//   sum_k q_k a_k = sum_k x_k a_k - 2056 sum_even a - 136 sum_odd a,
// the two activation sums formed once per item and shared by the lane's
// rows.  The item's partial times the fp32 scale goes to the row's total.
//
// Reduction.  Lanes of one row sum their totals by shuffles (fixed order);
// a team's warps add theirs in k order through shared memory after a named
// barrier; with a cluster the CTAs' sums are added in rank order; the bias
// is added in fp32 and Y rounded once.  The result does not depend on
// timing.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"
#include "waits.cuh"

namespace w4a16 {
namespace {

constexpr int kRbWarps = kRbWarpsPerCta;

struct RbArgs {
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

template <bool F16>
__device__ __forceinline__ float rb_act(uint16_t b) {
  if constexpr (F16) {
    return __half2float(__ushort_as_half(b));
  } else {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
  }
}

template <bool F16>
__device__ __forceinline__ uint16_t rb_out(float x) {
  if constexpr (F16) {
    return __half_as_ushort(__float2half_rn(x));
  } else {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
  }
}

// Activations of one chunk: CH values (CH / 2 words of two 16-bit values,
// k even in the low half) to CH / 2 (even k, odd k) pairs.
template <int CH, bool F16>
__device__ __forceinline__ void rb_acts(const uint32_t (&w)[CH / 2], float2 (&a)[CH / 2]) {
#pragma unroll
  for (int i = 0; i < CH / 2; ++i) {
    if constexpr (F16) {
      a[i] = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
    } else {
      a[i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xFFFF0000u));
    }
  }
}

// A nibble at bits p..p+3 of v, as the float 2^(23-p) + (n ^ 8) = 2^(23-p)
// + 8 + q: one AND-XOR puts it under the exponent whose unit is bit p, with
// the sign bit of the two's-complement nibble flipped.
template <int P>
__device__ __forceinline__ float rb_nib(uint32_t v) {
  constexpr uint32_t kMagic = (static_cast<uint32_t>(150 - P) << 23) | (8u << P);
  return __uint_as_float(ptx::and_xor(v, 0xFu << P, kMagic));
}
template <int P>
__device__ __forceinline__ constexpr float rb_off() {
  return static_cast<float>((1u << (23 - P)) + 8u);
}

// The 8 codes of one word as exact (q_k, q_k+1) pairs, k even: nibbles 0..4
// sit at bits 0, 4, 8, 12, 16 of w, nibbles 5..7 at bits 8, 12, 16 of w >>
// 12 (one shift); one packed subtraction of the exponents' offsets per pair
// is exact (x and its offset share a binade).
__device__ __forceinline__ void rb_codes(uint32_t w, float2 (&q)[4]) {
  const uint32_t v = w >> 12;
  q[0] = __fadd2_rn(make_float2(rb_nib<0>(w), rb_nib<4>(w)), make_float2(-rb_off<0>(), -rb_off<4>()));
  q[1] = __fadd2_rn(make_float2(rb_nib<8>(w), rb_nib<12>(w)), make_float2(-rb_off<8>(), -rb_off<12>()));
  q[2] = __fadd2_rn(make_float2(rb_nib<16>(w), rb_nib<8>(v)), make_float2(-rb_off<16>(), -rb_off<8>()));
  q[3] = __fadd2_rn(make_float2(rb_nib<12>(v), rb_nib<16>(v)), make_float2(-rb_off<12>(), -rb_off<16>()));
}

// MT: activation rows (M <= MT); CH: codes per lane chunk; RPL: rows per lane.
template <int MT, int CH, int RPL>
struct RbCfg {
  static constexpr int kLPR = kGroup / CH;           // lanes per row
  static constexpr int kRowsPerPass = 32 / kLPR;     // rows one warp instruction covers
  static constexpr int kRB = kRowsPerPass * RPL;     // rows per block
  static constexpr int kWords = CH / 8;              // code words per lane-chunk
  static_assert(kGroup % kRB == 0, "a row block sits inside one 128-row tile");
  // one stage: the item's codes, its rows' scales, MT activation rows
  static constexpr int kCodeBytes = kRB * 64;
  static constexpr int kScaleOff = kCodeBytes;
  static constexpr int kActOff = kScaleOff + kRB * 2;
  static constexpr int kStage = kActOff + MT * kGroup * 2;
  static constexpr int kDepth = MT <= 1 ? 5 : MT <= 2 ? 7 : 6;   // stages per warp
  static constexpr int kBarOff = kRbWarps * kDepth * kStage;
  static constexpr int kSmem = kBarOff + kRbWarps * kDepth * 8;
  static_assert(kActOff % 16 == 0 && kStage % 16 == 0, "bulk-copy destinations 16-byte aligned");
};

// Two CTAs of 8 warps per SM (registers <= 128, shared memory <= 113 KB each).
constexpr int kRbCtasPerSm = 2;

// Walks a warp's items for the copies: the row blocks of its team (rb = T,
// T + TT, ...) and, in each, the warp's groups k0 .. k1 - 1, with the item's
// copy sources and transaction bytes (stepped, not recomputed, inside a
// row block).
template <int RB, int MT>
struct RbWalk {
  int rb, g;
  const uint8_t* codes;      // RB x 64 bytes
  const __half* scales;      // nv values
  const uint16_t* act;       // row 0's 128 values
  uint32_t scale_bytes, bytes;
  __device__ bool valid(int NB) const { return rb < NB; }
  __device__ void start(const RbArgs& a, int rb_, int k0) {
    rb = rb_;
    g = k0;
    if (rb >= a.NB) return;
    const int r0 = rb * RB;
    const int tn = r0 / kTileW;
    const int nv = a.N - r0 < RB ? a.N - r0 : RB;   // a multiple of 8
    codes = a.packed + ((static_cast<int64_t>(tn) * a.KB + k0) * kTileW + (r0 - tn * kTileW)) * 64;
    scales = a.scales + static_cast<int64_t>(k0) * a.N + r0;
    act = a.A + static_cast<int64_t>(k0) * kGroup;
    scale_bytes = 2u * static_cast<uint32_t>(nv);
    bytes = RB * 64 + scale_bytes + static_cast<uint32_t>(a.M) * kGroup * 2;
  }
  __device__ void next(const RbArgs& a, int k0, int k1, int TT) {
    if (++g == k1) {
      start(a, rb + TT, k0);
    } else {
      codes += kTileW * 64;
      scales += a.N;
      act += kGroup;
    }
  }
};

__device__ __forceinline__ uint32_t lds_u16(uint32_t saddr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(saddr));
  return v;
}

template <int MT, int CH, int RPL, bool F16>
__global__ void __launch_bounds__(kRbWarps * 32, kRbCtasPerSm)
    gemv_rb_kernel(const __grid_constant__ RbArgs g) {
  using C = RbCfg<MT, CH, RPL>;
  constexpr int W = C::kWords;
  constexpr int D = C::kDepth;
  extern __shared__ __align__(128) uint8_t smem[];
  // per warp, per row-block parity: its rows' totals (a team's flush)
  __shared__ float tbuf[kRbWarps][2][C::kRB][MT];
  __shared__ float csum[C::kRB][MT];   // cluster split: the CTA's totals
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int WK = g.team, S = g.cluster;
  const int tpc = kRbWarps / WK;                  // teams per CTA
  const int team = warp / WK, wt = warp - team * WK;
  const int c = lane % C::kLPR;                   // the lane's chunk
  const int rl = lane / C::kLPR;                  // the lane's first row in a block

  // the team's first row block and stride; with a cluster split the CTA is
  // one team on one row block and its rank takes a share of K
  int T, TT, rank = 0, cg0 = 0, cg1 = g.KB;
  if (S > 1) {
    T = static_cast<int>(blockIdx.x) / S;
    rank = static_cast<int>(blockIdx.x) - T * S;
    TT = g.NB;
    cg0 = (rank * g.KB) / S;
    cg1 = ((rank + 1) * g.KB) / S;
  } else {
    T = static_cast<int>(blockIdx.x) * tpc + team;
    TT = static_cast<int>(gridDim.x) * tpc;
  }
  const int k0 = cg0 + (wt * (cg1 - cg0)) / WK;
  const int k1 = cg0 + ((wt + 1) * (cg1 - cg0)) / WK;

  uint8_t* ring = smem + warp * D * C::kStage;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kBarOff) + warp * D;
  if (threadIdx.x == 0) abort_flag = 0;
  if (lane == 0) {
    for (int s = 0; s < D; ++s) ptx::mbar_init(&full[s], 1);
    ptx::fence_mbar_init();
  }
  __syncthreads();
  const WaitCtx wc{g.err, g.timeout_ns, &abort_flag};

  // an item's copies, issued by lane 0: weights (codes and the valid rows'
  // scales) and activations (the M rows' 128 values)
  using Walk = RbWalk<C::kRB, MT>;
  auto issue_w = [&](const Walk& it, uint8_t* st, uint64_t* bar) {
    ptx::mbar_arrive_expect_tx(bar, it.bytes);
    ptx::bulk_g2s(st, it.codes, C::kCodeBytes, bar);
    ptx::bulk_g2s(st + C::kScaleOff, it.scales, it.scale_bytes, bar);
  };
  auto issue_a = [&](const Walk& it, uint8_t* st, uint64_t* bar) {
    if constexpr (MT == 1) {
      ptx::bulk_g2s(st + C::kActOff, it.act, kGroup * 2, bar);
    } else {
      for (int m = 0; m < g.M; ++m)
        ptx::bulk_g2s(st + C::kActOff + m * kGroup * 2, it.act + static_cast<int64_t>(m) * g.K, kGroup * 2, bar);
    }
  };

  // (the launch guarantees KB >= team x cluster: no warp's range is empty)
  const int first = k1 > k0 ? T : g.NB;
  Walk pre;
  pre.start(g, first, k0);
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

  float acc[RPL][MT];
#pragma unroll
  for (int j = 0; j < RPL; ++j)
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[j][m] = 0.0f;

  auto compute = [&](uint32_t st) {
    uint32_t cw[RPL][W];
    float sc[RPL];
#pragma unroll
    for (int j = 0; j < RPL; ++j) {
      const int r = rl + C::kRowsPerPass * j;
      const uint2 v = ptx::lds64(st + r * 64 + c * (CH / 2));
      cw[j][0] = v.x;
      cw[j][1] = v.y;
      sc[j] = __half2float(__ushort_as_half(static_cast<uint16_t>(lds_u16(st + C::kScaleOff + 2 * r))));
    }
    float2 a[MT][CH / 2];
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      uint32_t aw[CH / 2];
#pragma unroll
      for (int q = 0; q < CH / 8; ++q) {
        // rows m >= M were not copied: their values are never stored
        const uint4 v = ptx::lds128(st + C::kActOff + m * kGroup * 2 + c * CH * 2 + 16 * q);
        aw[4 * q] = v.x;
        aw[4 * q + 1] = v.y;
        aw[4 * q + 2] = v.z;
        aw[4 * q + 3] = v.w;
      }
      rb_acts<CH, F16>(aw, a[m]);
    }
#pragma unroll
    for (int j = 0; j < RPL; ++j) {
      float2 p[MT];
#pragma unroll
      for (int m = 0; m < MT; ++m) p[m] = make_float2(0.0f, 0.0f);
#pragma unroll
      for (int wi = 0; wi < W; ++wi) {
        float2 q[4];
        rb_codes(cw[j][wi], q);
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int m = 0; m < MT; ++m) p[m] = __ffma2_rn(q[i], a[m][4 * wi + i], p[m]);
      }
#pragma unroll
      for (int m = 0; m < MT; ++m) acc[j][m] = fmaf(sc[j], p[m].x + p[m].y, acc[j][m]);
    }
  };

  // The row block's totals: the chunk lanes of a row in a fixed order, then
  // the team's warps in k order; stored to Y (bias added in fp32, one
  // rounding), or with a cluster split left in csum for the cluster sum.
  int nflush = 0;
  auto flush = [&](int rb) {
#pragma unroll
    for (int j = 0; j < RPL; ++j)
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int o = 1; o < C::kLPR; o <<= 1) acc[j][m] += __shfl_xor_sync(0xFFFFFFFFu, acc[j][m], o);
    const int r0 = rb * C::kRB;
    if (WK == 1 && S == 1) {
      if (c == 0) {
#pragma unroll
        for (int j = 0; j < RPL; ++j) {
          const int n = r0 + rl + C::kRowsPerPass * j;
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            if (n < g.N && m < g.M) {
              float t = acc[j][m];
              if (g.bias != nullptr) t += rb_act<F16>(g.bias[n]);
              g.Y[static_cast<int64_t>(m) * g.N + n] = rb_out<F16>(t);
            }
          }
        }
      }
    } else {
      if (c == 0) {
#pragma unroll
        for (int j = 0; j < RPL; ++j)
#pragma unroll
          for (int m = 0; m < MT; ++m) tbuf[warp][nflush & 1][rl + C::kRowsPerPass * j][m] = acc[j][m];
      }
      ptx::named_barrier_sync(1 + team, WK * 32);
      if (wt == 0) {
        for (int e = lane; e < C::kRB * MT; e += 32) {
          const int row = e / MT, m = e - row * MT;
          float t = 0.0f;
          for (int w = 0; w < WK; ++w) t += tbuf[team * WK + w][nflush & 1][row][m];
          if (S > 1) {
            csum[row][m] = t;
          } else {
            const int n = r0 + row;
            if (n < g.N && m < g.M) {
              if (g.bias != nullptr) t += rb_act<F16>(g.bias[n]);
              g.Y[static_cast<int64_t>(m) * g.N + n] = rb_out<F16>(t);
            }
          }
        }
      }
    }
#pragma unroll
    for (int j = 0; j < RPL; ++j)
#pragma unroll
      for (int m = 0; m < MT; ++m) acc[j][m] = 0.0f;
    ++nflush;
  };

  // the ring: item i in stage i % D; once computed, the stage takes item i + D
  bool ok = true;
  int s = 0;
  uint32_t phase = 0;
  int waited = 0;   // items whose copies have landed
  const uint32_t ring_u32 = ptx::smem_u32(ring);
  uint32_t st = ring_u32;
  const int per_block = k1 - k0;
  int left = per_block;   // items left in the current row block
#pragma unroll 1
  for (int rb = first; rb < g.NB;) {
    if (ok) {
      if (wait_warp(&full[s], phase, wc))
        ++waited;
      else
        ok = false;
    }
    compute(st);
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
    const int r0 = T * C::kRB;
    for (int e = threadIdx.x; e < C::kRB * MT; e += blockDim.x) {
      const int row = e / MT, m = e - row * MT;
      if (row % S != rank) continue;
      const int n = r0 + row;
      if (n >= g.N || m >= g.M) continue;
      float t = 0.0f;
      for (int q = 0; q < S; ++q) t += ptx::ld_dsmem_f32(base + 4u * static_cast<uint32_t>(e), q);
      if (g.bias != nullptr) t += rb_act<F16>(g.bias[n]);
      g.Y[static_cast<int64_t>(m) * g.N + n] = rb_out<F16>(t);
    }
    ptx::cluster_sync();   // every CTA's sums stay alive until read
  }
}

template <int MT, int CH, int RPL, bool F16>
cudaError_t launch_rb(const GemmProblem& p, const GemmSchedule& s, bool use_pdl, cudaStream_t stream) {
  using C = RbCfg<MT, CH, RPL>;
  const int64_t blocks = (p.N + C::kRB - 1) / C::kRB;
  const int S = s.cluster > 1 ? s.cluster : 1;
  const int WK = s.team;
  const int64_t KB = p.K / kGroup;
  // every warp gets at least one group; a cluster split is one CTA-wide team
  // per row block
  if (p.M > MT || S > 8 || (WK != 1 && WK != 2 && WK != 4 && WK != 8) || KB < WK * S ||
      (S > 1 && (WK != kRbWarps || s.grid != blocks * S)) || s.grid < 1)
    return cudaErrorInvalidValue;
  RbArgs g{};
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
  auto kernel = gemv_rb_kernel<MT, CH, RPL, F16>;
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
  cfg.gridDim = dim3(static_cast<unsigned>(s.grid));
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
  return cudaLaunchKernelEx(&cfg, kernel, g);
}

}  // namespace

int gemv_rb_rows(int act_tile) {
  return act_tile <= 1 ? RbCfg<1, 16, 8>::kRB : RbCfg<4, 16, 4>::kRB;
}

int gemv_rb_ctas_per_sm(int act_tile) {
  (void)act_tile;
  return kRbCtasPerSm;
}

size_t gemv_rb_smem_bytes(int act_tile) {
  switch (act_tile) {
    case 1: return RbCfg<1, 16, 8>::kSmem;
    case 2: return RbCfg<2, 16, 4>::kSmem;
    case 4: return RbCfg<4, 16, 4>::kSmem;
    default: return 0;
  }
}

cudaError_t launch_gemv_rb(const GemmKernelConfig& c, const GemmGroup& grp, bool use_pdl,
                           cudaStream_t stream) {
  if (grp.count != 1) return cudaErrorInvalidValue;
  const GemmProblem& p = grp.p[0];
  const GemmSchedule& s = grp.s[0];
  if (p.swiglu) return cudaErrorInvalidValue;   // the fused epilogue is the tcgen05 path's
  const bool f16 = p.act_f16;
  switch (c.act_tile) {
    case 1: return f16 ? launch_rb<1, 16, 8, true>(p, s, use_pdl, stream)
                       : launch_rb<1, 16, 8, false>(p, s, use_pdl, stream);
    case 2: return f16 ? launch_rb<2, 16, 4, true>(p, s, use_pdl, stream)
                       : launch_rb<2, 16, 4, false>(p, s, use_pdl, stream);
    case 4: return f16 ? launch_rb<4, 16, 4, true>(p, s, use_pdl, stream)
                       : launch_rb<4, 16, 4, false>(p, s, use_pdl, stream);
    default: return cudaErrorInvalidConfiguration;
  }
}

}  // namespace w4a16
