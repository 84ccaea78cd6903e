// W4A16 GEMM on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
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
// partial tile to the workspace and increments that tile's counter; the CTA
// whose increment completes the count sums the partials in k order
// (deterministic), adds the bias and stores Y, then resets the counter.
// Nothing ever waits on another CTA.
//
// Warp roles (blockDim = 224 + 128 * dequant_wgs):
//   warps 0, 2  TMA producers (one lane each; even and odd units, because one
//               thread can only complete a few mbarrier phases per
//               microsecond, fewer than the weight stream needs)
//   warp 1      TMEM allocator; MMA issuer (one lane)
//   warps 3-6   readout: accumulator -> registers / output, stream-K fixup
//   warps 7..   dequant: packed codes (shared memory) -> weight operand (TMEM)
// A warp may only touch TMEM lanes 32 * (warp % 4) .. + 31, so each readout
// and dequant thread owns weight row 32 * (warp % 4) + lane.  The dequant
// warps never wait on accumulators: they run up to four units ahead of the
// MMA, which runs up to DB units ahead of the readout.
//
// Every wait on an mbarrier is bounded by a time limit; on expiry the kernel
// records an error word, lets every role leave its loop, waits (bounded) for
// its own copies and MMAs in flight, frees TMEM and returns.
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
__device__ unsigned long long* g_trace = nullptr;
__device__ unsigned long long* g_trace_units = nullptr;
#define W4A16_TRACE_POINT(id)                                                           \
  do {                                                                                  \
    if (trace_cta != nullptr) trace_cta[blockIdx.x * 16 + (id)] = ptx::globaltimer_ns(); \
  } while (0)
#define W4A16_TRACE_UNIT(role, i)                                                       \
  do {                                                                                  \
    if (trace_unit != nullptr && (i) < 64)                                             \
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
constexpr int kWBytes = kTileW * kUnitK / 2;   // packed codes per unit: 8 KiB
constexpr int kSBytes = kTileW * 2;            // scales per unit: 256 B
constexpr int kAStages = 4;                    // weight-operand stages in TMEM
constexpr int kAStageCols = kUnitK / 2;        // 64 TMEM columns per stage
constexpr int kDCol = kAStages * kAStageCols;  // accumulators start at column 256
constexpr int kDCols = 512 - kDCol;            // 256 accumulator columns
constexpr uint32_t kTmemCols = 512;
constexpr int kReadoutWarp0 = 3;
constexpr int kDequantWarp0 = 7;

struct Args {
  int M, N, K, KB;
  int n_tiles;
  int dp_tiles;
  int sk_units;
  int act_3d;                  // activation map is 3-D: both 64-k halves in one copy
  const __half* scales;        // [K/128, N]; the group-mode readout reads its scales here
  const __nv_bfloat16* bias;
  __nv_bfloat16* Y;
  float* ws;
  uint32_t* counters;
  uint32_t* err;
  uint64_t timeout_ns;
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

  __device__ void init(const Args& a) {
    c = blockIdx.x;
    C = gridDim.x;
    KB = a.KB;
    dp_tiles = a.dp_tiles;
    dp_iters = (dp_tiles > c) ? (dp_tiles - c + C - 1) / C : 0;
    u0 = static_cast<int>((static_cast<int64_t>(c) * a.sk_units) / C);
    u1 = static_cast<int>((static_cast<int64_t>(c + 1) * a.sk_units) / C);
    total = dp_iters * KB + (u1 - u0);
  }

  __device__ Unit get(int i) const {
    Unit r;
    const int ndp = dp_iters * KB;
    if (i < ndp) {
      const int it = i / KB;
      r.tile = it * C + c;
      r.kb = i - it * KB;
      r.seg_first = (r.kb == 0);
      r.seg_last = (r.kb == KB - 1);
      r.whole = true;
      r.slot = 0;
      r.sk_tile = -1;
    } else {
      const int u = u0 + (i - ndp);
      const int tl = u / KB;
      r.tile = dp_tiles + tl;
      r.kb = u - tl * KB;
      const int seg_lo = max(u0, tl * KB);
      const int seg_hi = min(u1, (tl + 1) * KB);   // exclusive
      r.seg_first = (u == seg_lo);
      r.seg_last = (u == seg_hi - 1);
      r.whole = (seg_lo == tl * KB) && (seg_hi == (tl + 1) * KB);
      r.slot = (tl == u0 / KB) ? 0 : 1;
      r.sk_tile = tl;
    }
    return r;
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

// CTA that owns stream-K unit u under the balanced split.
__device__ __forceinline__ int sk_owner(int u, int C, int sk_units) {
  return static_cast<int>(((static_cast<int64_t>(u) + 1) * C - 1) / sk_units);
}

struct Shared {
  uint64_t full[16];
  uint64_t empty[16];
  uint64_t afull[kAStages];
  uint64_t aempty[kAStages];
  uint64_t dfull[4];
  uint64_t dempty[4];
  uint64_t unit_done[16];     // ring: phase completes when a unit's MMAs completed
  uint64_t mma_done;
  uint64_t wsync;             // readout-only barrier (bounded waits, unlike bar.sync)
  uint32_t tmem_base;
  int abort_flag;
  int fixup_last;
};

// ------------------------------------------------------- code -> bf16 pairs
// Eight 4-bit codes (one 32-bit word, code k in nibble k) to four bf16x2
// words holding the code pairs (k0,k1), (k2,k3), (k4,k5), (k6,k7) as exact
// bf16 integers.  0x4300 | (nibble ^ 8) is the bf16 value 136 + q; one fused
// multiply-add subtracts 136.
__device__ __forceinline__ uint32_t bf16x2_fma(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

__device__ __forceinline__ void codes_to_bf16(uint32_t w, uint32_t* out) {
  const uint32_t v = w >> 4;
  const uint32_t one = 0x3F803F80u;       // (1.0, 1.0)
  const uint32_t m136 = 0xC308C308u;      // (-136, -136)
  out[0] = bf16x2_fma(ptx::and_xor(ptx::prmt(w, v, 0x0400), 0x000F000Fu, 0x43084308u), one, m136);
  out[1] = bf16x2_fma(ptx::and_xor(ptx::prmt(w, v, 0x0501), 0x000F000Fu, 0x43084308u), one, m136);
  out[2] = bf16x2_fma(ptx::and_xor(ptx::prmt(w, v, 0x0602), 0x000F000Fu, 0x43084308u), one, m136);
  out[3] = bf16x2_fma(ptx::and_xor(ptx::prmt(w, v, 0x0703), 0x000F000Fu, 0x43084308u), one, m136);
}

// bf16_rn(q * s) for both halves: q * s_lo is exact (<= 7 significant bits),
// so fma(q, s_hi, q * s_lo) rounds the exact product once.
__device__ __forceinline__ uint32_t scale_pair(uint32_t q, uint32_t s_hi2, uint32_t s_lo2) {
  const uint32_t lo = bf16x2_fma(q, s_lo2, 0x80008000u);   // q * s_lo + (-0)
  return bf16x2_fma(q, s_hi2, lo);
}

template <int BA, int NWG, bool GRP, int STAGES, int NACC>
struct Cfg {
  static constexpr int kActBox = BA * 128;                        // bytes per 64-k box
  static constexpr int kStageRaw = 2 * kActBox + kWBytes + kSBytes;
  static constexpr int kStage = (kStageRaw + 1023) / 1024 * 1024;
  static constexpr int kThreads = 32 * kDequantWarp0 + 128 * NWG;   // 15 warps: <= 128 registers
  static constexpr int kWords = 16;                               // code words per thread per unit
  // Each accumulator buffer holds NACC partial accumulators of BA columns:
  // k-step kk of a unit goes to partial kk % NACC, so NACC independent MMA
  // dependency chains overlap in the tensor pipe (with a small N a single
  // chain is bound by the MMA latency, not its throughput); the readout sums
  // the partials.
  static constexpr int kBufCols = BA * NACC;
  static constexpr int kDB = (kDCols / kBufCols) < 4 ? (kDCols / kBufCols) : 4;
  static constexpr int kChunk = BA < (GRP ? 16 : 32) ? BA : (GRP ? 16 : 32);
  static constexpr size_t kSmem = static_cast<size_t>(STAGES) * kStage + 1024 + sizeof(Shared);
  static constexpr uint32_t kTx = 2 * kActBox + kWBytes + kSBytes;
  static_assert(BA % 16 == 0 && BA >= 16 && BA <= 256, "tcgen05 N for M=128");
  static_assert(kDB >= 1, "accumulators fit in TMEM");
  static_assert(NACC == 1 || NACC == 2 || NACC == 4, "partial accumulators divide the 8 k-steps");
  static_assert(!GRP || BA <= 64, "group mode keeps BA fp32 accumulators per thread");
  static_assert(STAGES <= 16, "barrier arrays");
  static_assert(NWG == 1 || NWG == 2, "dequant warpgroups");
};

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

// CNT accumulator columns of this thread's lane, summed over the NACC
// partial accumulators (BA columns apart).
template <int CNT, int NACC, int BA>
__device__ __forceinline__ void load_partials(uint32_t taddr, float (&v)[CNT]) {
  uint32_t r[CNT];
  tmem_ld_cols<CNT>(taddr, r);
#pragma unroll
  for (int j = 0; j < CNT; ++j) v[j] = __uint_as_float(r[j]);
#pragma unroll
  for (int p = 1; p < NACC; ++p) {
    tmem_ld_cols<CNT>(taddr + p * BA, r);
#pragma unroll
    for (int j = 0; j < CNT; ++j) v[j] += __uint_as_float(r[j]);
  }
}

// Write accumulator columns [col0, col0 + CNT) of this thread's weight row
// either to Y (whole tile) or to this CTA's partial slot.
template <int BA, int CNT>
__device__ __forceinline__ void emit_cols(const Args& a, const Unit& u, int row, int col0,
                                          const float (&v)[CNT], float bias_n) {
  const int n0 = (u.tile % a.n_tiles) * kTileW;
  const int m0 = (u.tile / a.n_tiles) * BA;
  if (u.whole) {
    const int n = n0 + row;
    if (n < a.N) {
#pragma unroll
      for (int j = 0; j < CNT; ++j) {
        const int m = m0 + col0 + j;
        if (m < a.M) a.Y[static_cast<int64_t>(m) * a.N + n] = __float2bfloat16_rn(v[j] + bias_n);
      }
    }
  } else {
    // partial slot, row-major: this thread's row holds BA contiguous floats
    float* slot = a.ws + (static_cast<int64_t>(blockIdx.x) * 2 + u.slot) * (BA * kTileW) +
                  row * BA + col0;
#pragma unroll
    for (int j = 0; j < CNT; j += 4)
      *reinterpret_cast<float4*>(slot + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
  }
}

// Barrier among the readout warps built on an mbarrier, so that a warp that
// gave up after a timeout cannot leave the others blocked forever.
__device__ bool readout_sync(Shared* sh, uint32_t& nsync, const WaitCtx& wc) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) ptx::mbar_arrive(&sh->wsync);
  const bool ok = wait_warp(&sh->wsync, nsync & 1, wc);
  ++nsync;
  return ok;
}

// After this CTA wrote a partial tile: count the arrival; the CTA that
// completes the count sums every partial of the tile in k order and stores Y.
template <int BA>
__device__ bool stream_k_fixup(const Args& a, const Unit& u, Shared* sh, int row, float bias_n,
                               uint32_t& nsync, const WaitCtx& wc) {
  constexpr int kSub = BA < 16 ? BA : 16;   // columns summed together
  const int C = gridDim.x;
  __threadfence();
  if (!readout_sync(sh, nsync, wc)) return false;
  const int KB = a.KB;
  const int c_lo = sk_owner(u.sk_tile * KB, C, a.sk_units);
  const int c_hi = sk_owner(u.sk_tile * KB + KB - 1, C, a.sk_units);
  if (threadIdx.x == 32 * kReadoutWarp0) {
    const uint32_t old = atomicAdd(&a.counters[u.sk_tile], 1u);
    const bool last = (old == static_cast<uint32_t>(c_hi - c_lo));
    if (last) atomicExch(&a.counters[u.sk_tile], 0u);
    sh->fixup_last = last ? 1 : 0;
  }
  if (!readout_sync(sh, nsync, wc)) return false;
  if (!sh->fixup_last) return true;
  __threadfence();
  const int n0 = (u.tile % a.n_tiles) * kTileW;
  const int m0 = (u.tile / a.n_tiles) * BA;
  const int n = n0 + row;
  const float* base = a.ws + row * BA;
  for (int c0 = 0; c0 < BA; c0 += kSub) {
    float acc[kSub];
#pragma unroll
    for (int j = 0; j < kSub; ++j) acc[j] = 0.0f;
#pragma unroll 4
    for (int cc = c_lo; cc <= c_hi; ++cc) {
      // slot 0 when the tile is the first stream-K tile of CTA cc, else 1
      const int first_tile = static_cast<int>((static_cast<int64_t>(cc) * a.sk_units) / C) / KB;
      const int slot = (u.sk_tile == first_tile) ? 0 : 1;
      const float4* src = reinterpret_cast<const float4*>(
          base + (static_cast<int64_t>(cc) * 2 + slot) * (BA * kTileW) + c0);
      float4 v[kSub / 4];
#pragma unroll
      for (int j = 0; j < kSub / 4; ++j) v[j] = __ldcg(src + j);
#pragma unroll
      for (int j = 0; j < kSub / 4; ++j) {
        acc[4 * j] += v[j].x;
        acc[4 * j + 1] += v[j].y;
        acc[4 * j + 2] += v[j].z;
        acc[4 * j + 3] += v[j].w;
      }
    }
    if (n < a.N) {
#pragma unroll
      for (int j = 0; j < kSub; ++j) {
        const int m = m0 + c0 + j;
        if (m < a.M) a.Y[static_cast<int64_t>(m) * a.N + n] = __float2bfloat16_rn(acc[j] + bias_n);
      }
    }
  }
  return true;
}

template <int BA, int NWG, bool GRP, int STAGES, int NACC>
__global__ void __launch_bounds__(Cfg<BA, NWG, GRP, STAGES, NACC>::kThreads, 1)
    w4a16_gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_act,
                         const __grid_constant__ CUtensorMap tm_w,
                         const __grid_constant__ CUtensorMap tm_s, const Args a) {
  using C = Cfg<BA, NWG, GRP, STAGES, NACC>;
  constexpr int DB = C::kDB;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  Shared* sh = reinterpret_cast<Shared*>(smem + STAGES * C::kStage);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  auto act_box = [&](int stage, int box) -> uint8_t* {
    return smem + stage * C::kStage + box * C::kActBox;
  };
  auto w_tile = [&](int stage) -> uint8_t* { return smem + stage * C::kStage + 2 * C::kActBox; };
  auto s_tile = [&](int stage) -> __half* {
    return reinterpret_cast<__half*>(smem + stage * C::kStage + 2 * C::kActBox + kWBytes);
  };

  // ---------------------------------------------------------------- set-up
#ifdef W4A16_TRACE
  unsigned long long* const trace_cta = g_trace;
  unsigned long long* const trace_unit = blockIdx.x == 0 ? g_trace_units : nullptr;
#endif
  // Barriers.  full[s]: a stage's copies landed.  unit_done[i % R]: all MMAs
  // of unit i completed (one tcgen05.commit per unit); it frees the
  // shared-memory stage and the TMEM weight stage of unit i and tells the
  // group-mode readout that the unit's partial sum is ready.  afull: the
  // weight operand is in TMEM (the dequant warps waited on full before, so
  // the MMA thread need not).  dempty: the readout drained an accumulator
  // buffer.  dfull (dequant mode): a run on a tile is fully accumulated.
  // Each mbarrier check costs about a hundred cycles even when the phase is
  // already complete, so the single MMA thread makes as few as it can.
  constexpr int R = STAGES > kAStages ? STAGES : kAStages;
  if (threadIdx.x == 0) W4A16_TRACE_POINT(0);
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&sh->full[s], 1);
      ptx::mbar_init(&sh->empty[s], 4);
    }
    for (int s = 0; s < R; ++s) ptx::mbar_init(&sh->unit_done[s], 1);
    for (int s = 0; s < kAStages; ++s) ptx::mbar_init(&sh->afull[s], 4);
    for (int s = 0; s < DB; ++s) {
      ptx::mbar_init(&sh->dfull[s], 1);
      ptx::mbar_init(&sh->dempty[s], 4);
    }
    ptx::mbar_init(&sh->mma_done, 1);
    ptx::mbar_init(&sh->wsync, 4);
    sh->abort_flag = 0;
    sh->fixup_last = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tmap(&tm_act);
    ptx::prefetch_tmap(&tm_w);
    ptx::prefetch_tmap(&tm_s);
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
  // Inputs may be produced by the previous kernel on the stream.
  ptx::grid_dependency_wait();
  ptx::grid_launch_dependents();
  if (threadIdx.x == 0) W4A16_TRACE_POINT(2);

  Sched sched;
  sched.init(a);
  UnitIter it;
  it.init(sched);
  const int total = sched.total;

  if (warp == 0 || warp == 2) {
    // ----------------------------------------------------- TMA producers
    if (lane == 0) {
      const int mine = warp == 0 ? 0 : 1;
      int issued = -1;
      for (int i = 0; i < total; ++i) {
        const Unit u = it.next();
        if ((i & 1) != mine) continue;
        const int stage = i % STAGES;
        if (i >= STAGES) {
          const int j = i - STAGES;   // the unit that last used this stage
          if (!wait_one(&sh->unit_done[j % R], (j / R) & 1, wc)) break;
        }
        const int m0 = (u.tile / a.n_tiles) * BA;
        ptx::mbar_arrive_expect_tx(&sh->full[stage], C::kTx);
        if (a.act_3d) {
          ptx::tma_load_3d(act_box(stage, 0), &tm_act, &sh->full[stage], 0, m0, u.kb * 2);
        } else {
          ptx::tma_load_2d(act_box(stage, 0), &tm_act, &sh->full[stage], u.kb * kUnitK, m0);
          ptx::tma_load_2d(act_box(stage, 1), &tm_act, &sh->full[stage], u.kb * kUnitK + 64, m0);
        }
        // the unit's codes: one contiguous 8 KiB tile of the tiled storage
        ptx::tma_load_2d(w_tile(stage), &tm_w, &sh->full[stage], 0,
                         ((u.tile % a.n_tiles) * a.KB + u.kb) * kTileW);
        ptx::tma_load_2d(s_tile(stage), &tm_s, &sh->full[stage], (u.tile % a.n_tiles) * kTileW,
                         u.kb);
        if (i <= 1) W4A16_TRACE_POINT(3);
        W4A16_TRACE_UNIT(0, i);
        issued = i;
      }
      if (*reinterpret_cast<volatile int*>(&sh->abort_flag)) {
        // let this producer's copies still in flight land before the CTA exits
        for (int i = issued; i >= 0 && i > issued - STAGES; i -= 2) {
          const uint64_t t0 = ptx::globaltimer_ns();
          while (!ptx::mbar_try_wait(&sh->full[i % STAGES], (i / STAGES) & 1)) {
            if (ptx::globaltimer_ns() - t0 > a.timeout_ns) break;
          }
        }
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(kTileW, BA);
      const uint32_t smem0 = ptx::smem_u32(smem);
      int seg = 0;
      int db = 0;
      for (int i = 0; i < total; ++i) {
        const Unit u = it.next();
        const int stage = i % STAGES;
        const int as = i % kAStages;
        W4A16_TRACE_UNIT(8, i);
        if (!wait_one(&sh->afull[as], (i / kAStages) & 1, wc)) break;
        W4A16_TRACE_UNIT(10, i);
        bool fresh;
        if constexpr (GRP) {
          db = i % DB;
          // the readout frees buffers in unit order: once unit i-1 is read
          // out, the buffers of units i .. i+DB-1 are all free
          if (db == 0 && i >= DB && !wait_one(&sh->dempty[DB - 1], ((i / DB) - 1) & 1, wc)) break;
          fresh = true;
        } else {
          fresh = u.seg_first;
          if (u.seg_first) {
            db = seg % DB;
            if (seg >= DB && !wait_one(&sh->dempty[db], ((seg / DB) - 1) & 1, wc)) break;
          }
        }
        ptx::tc_fence_after();
        if (i == 0) W4A16_TRACE_POINT(4);
        if (i == total - 1) W4A16_TRACE_POINT(5);
        W4A16_TRACE_UNIT(4, i);
        const uint32_t d_tmem = tmem + kDCol + db * C::kBufCols;
        const uint32_t a_tmem = tmem + as * kAStageCols;
        const uint32_t b0 = smem0 + stage * C::kStage;
#pragma unroll
        for (int kk = 0; kk < kUnitK / 16; ++kk) {
          const uint32_t baddr = b0 + (kk >> 2) * C::kActBox + (kk & 3) * 32;
          ptx::mma_bf16_tmem_a(d_tmem + (kk % NACC) * BA, a_tmem + kk * 8,
                               ptx::smem_desc_sw128(baddr), idesc,
                               (kk >= NACC || !fresh) ? 1u : 0u);
        }
        W4A16_TRACE_UNIT(11, i);
        ptx::mma_commit(&sh->unit_done[i % R]);
        if constexpr (!GRP) {
          if (u.seg_last) {
            ptx::mma_commit(&sh->dfull[db]);
            ++seg;
          }
        }
        W4A16_TRACE_UNIT(5, i);
      }
      // all MMAs of this CTA complete before TMEM is freed
      ptx::mma_commit(&sh->mma_done);
      const uint64_t t0 = ptx::globaltimer_ns();
      while (!ptx::mbar_try_wait(&sh->mma_done, 0)) {
        if (ptx::globaltimer_ns() - t0 > a.timeout_ns) {
          wait_record_timeout(wc);
          break;
        }
      }
    }
  } else if (warp < kDequantWarp0) {
    // ------------------------------------------------------------ readout
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    uint32_t nsync = 0;
    float acc[GRP ? BA : 1];
    float bias_n = 0.0f;
    int seg = 0;
    // group mode: the unit's scales come from global memory (L2: the TMA just
    // brought them), fetched two units ahead
    UnitIter ahead = it;
    float s_next = 0.0f, s_next2 = 0.0f;
    auto fetch_scale = [&](int j) -> float {
      if (j >= total) return 0.0f;
      const Unit v = ahead.next();
      const int nn = (v.tile % a.n_tiles) * kTileW + row;
      return nn < a.N ? __half2float(a.scales[static_cast<int64_t>(v.kb) * a.N + nn]) : 0.0f;
    };
    if constexpr (GRP) {
      s_next = fetch_scale(0);
      s_next2 = fetch_scale(1);
    }
    for (int i = 0; i < total; ++i) {
      const Unit u = it.next();
      const int n = (u.tile % a.n_tiles) * kTileW + row;
      if (u.seg_first)
        bias_n = (a.bias != nullptr && n < a.N) ? __bfloat162float(a.bias[n]) : 0.0f;
      if constexpr (GRP) {
        const int db = i % DB;
        const float scale = s_next;
        s_next = s_next2;
        s_next2 = fetch_scale(i + 2);
        if (!wait_warp(&sh->unit_done[i % R], (i / R) & 1, wc)) break;
        if (threadIdx.x == 32 * kReadoutWarp0 && i == 0) W4A16_TRACE_POINT(8);
        if (threadIdx.x == 32 * kReadoutWarp0 && i == total - 1) W4A16_TRACE_POINT(9);
        if (threadIdx.x == 32 * kReadoutWarp0) W4A16_TRACE_UNIT(6, i);
        ptx::tc_fence_after();
#pragma unroll
        for (int c0 = 0; c0 < BA; c0 += C::kChunk) {
          float d[C::kChunk];
          load_partials<C::kChunk, NACC, BA>(lane_base + kDCol + db * C::kBufCols + c0, d);
#pragma unroll
          for (int j = 0; j < C::kChunk; ++j)
            acc[c0 + j] = u.seg_first ? scale * d[j] : fmaf(scale, d[j], acc[c0 + j]);
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0 && db == DB - 1) ptx::mbar_arrive(&sh->dempty[DB - 1]);
        if (threadIdx.x == 32 * kReadoutWarp0) W4A16_TRACE_UNIT(7, i);
        if (u.seg_last) {
          emit_cols<BA, BA>(a, u, row, 0, acc, bias_n);
          if (!u.whole && !stream_k_fixup<BA>(a, u, sh, row, bias_n, nsync, wc)) break;
        }
      } else {
        if (!u.seg_last) continue;
        const int db = seg % DB;
        if (!wait_warp(&sh->dfull[db], (seg / DB) & 1, wc)) break;
        ++seg;
        ptx::tc_fence_after();
#pragma unroll 1
        for (int c0 = 0; c0 < BA; c0 += C::kChunk) {
          float v[C::kChunk];
          load_partials<C::kChunk, NACC, BA>(lane_base + kDCol + db * C::kBufCols + c0, v);
          emit_cols<BA, C::kChunk>(a, u, row, c0, v, bias_n);
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&sh->dempty[db]);
        if (!u.whole && !stream_k_fixup<BA>(a, u, sh, row, bias_n, nsync, wc)) break;
      }
    }
  } else {
    // ------------------------------------------------------------ dequant
    // warpgroup wg converts units wg, wg + NWG, ...: every thread its whole
    // row of 128 codes per unit
    const int wg = (warp - kDequantWarp0) >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t wrow0 = ptx::smem_u32(w_tile(0)) + row * 64;
    const uint32_t swz = (row >> 1) & 3;
    for (int i = wg; i < total; i += NWG) {
      const int stage = i % STAGES;
      const int as = i % kAStages;
      if (!wait_warp(&sh->full[stage], (i / STAGES) & 1, wc)) break;
      if (i == 0 && threadIdx.x == 32 * kDequantWarp0) W4A16_TRACE_POINT(6);
      if (threadIdx.x == 32 * kDequantWarp0) W4A16_TRACE_UNIT(1, i);

      // the row's 64 B of packed codes, stored with the 64-byte swizzle:
      // 16-byte chunk c of row r sits at chunk position c ^ ((r >> 1) & 3)
      const uint32_t wrow = wrow0 + stage * C::kStage;
      uint32_t words[16];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 v = ptx::lds128(wrow + ((q ^ swz) << 4));
        words[4 * q + 0] = v.x;
        words[4 * q + 1] = v.y;
        words[4 * q + 2] = v.z;
        words[4 * q + 3] = v.w;
      }
      float scale = 0.0f;
      if constexpr (!GRP) scale = __half2float(s_tile(stage)[row]);

      // the TMEM stage is free once the MMAs of the unit that used it completed
      if (i >= kAStages) {
        const int j = i - kAStages;
        if (!wait_warp(&sh->unit_done[j % R], (j / R) & 1, wc)) break;
      }
      if (threadIdx.x == 32 * kDequantWarp0) W4A16_TRACE_UNIT(2, i);
      ptx::tc_fence_after();
      const uint32_t a_addr = lane_base + as * kAStageCols;
      uint32_t s_hi2 = 0, s_lo2 = 0;
      if constexpr (!GRP) {
        const __nv_bfloat16 hi = __float2bfloat16_rn(scale);
        const float lo_f = scale - __bfloat162float(hi);        // exact
        const __nv_bfloat16 lo = __float2bfloat16_rn(lo_f);     // exact
        const uint32_t hi_bits = static_cast<uint32_t>(__bfloat16_as_ushort(hi));
        const uint32_t lo_bits = static_cast<uint32_t>(__bfloat16_as_ushort(lo));
        s_hi2 = hi_bits | (hi_bits << 16);
        s_lo2 = lo_bits | (lo_bits << 16);
      }
      // convert and store 16 columns (4 code words) at a time
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t opnd[16];
#pragma unroll
        for (int w = 0; w < 4; ++w) codes_to_bf16(words[4 * q + w], &opnd[4 * w]);
        if constexpr (!GRP) {
#pragma unroll
          for (int c = 0; c < 16; ++c) opnd[c] = scale_pair(opnd[c], s_hi2, s_lo2);
        }
        ptx::tmem_st_x16(a_addr + 16 * q, opnd);
      }
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&sh->afull[as]);
      if (threadIdx.x == 32 * kDequantWarp0) W4A16_TRACE_UNIT(3, i);
      if (i >= total - NWG && threadIdx.x == 32 * kDequantWarp0) W4A16_TRACE_POINT(7);
    }
  }

  // ------------------------------------------------------------- teardown
  if (threadIdx.x == 32 * kReadoutWarp0) W4A16_TRACE_POINT(10);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem, kTmemCols);
  if (threadIdx.x == 32) W4A16_TRACE_POINT(11);
}

// One-thread kernel whose wait can never complete: exercises the bounded
// wait and the error word without faulting or hanging the GPU.
__global__ void wait_timeout_selftest_kernel(uint32_t* err, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    ptx::fence_mbar_init();
    abort_flag = 0;
    const WaitCtx wc{err, timeout_ns, &abort_flag};
    (void)wait_one(&bar, 0, wc);   // nobody arrives: times out
  }
}

template <int BA, int NWG, bool GRP, int STAGES, int NACC>
cudaError_t launch_instance(const GemmSchedule& s, const GemmProblem& p, bool use_pdl,
                            cudaStream_t stream) {
  using C = Cfg<BA, NWG, GRP, STAGES, NACC>;
  auto kernel = w4a16_gemm_tc_kernel<BA, NWG, GRP, STAGES, NACC>;

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

  CUtensorMap tm_act, tm_w, tm_s;
  // Activations as [K/64][M][64]: one box {64, BA, 2} brings both 64-wide K
  // halves of a unit, in the same shared-memory order as two 2-D boxes.
  int act_3d = 1;
  if (encode_tmap_3d(&tm_act, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.A, 64, p.M, p.K / 64, p.K * 2, 128,
                     64, BA, 2, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS) {
    act_3d = 0;
    if (encode_tmap_2d(&tm_act, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.A, p.K, p.M, p.K * 2, 64, BA,
                       CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  // tiled code storage viewed as rows of 64 bytes: tile (tn, g) is rows
  // (tn * K/128 + g) * 128 .. + 127
  const uint64_t w_rows = static_cast<uint64_t>((p.N + kTileW - 1) / kTileW) * (p.K / kUnitK) * kTileW;
  if (encode_tmap_2d(&tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.packed, 64, w_rows, 64, 64, kTileW,
                     CU_TENSOR_MAP_SWIZZLE_64B) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  if (encode_tmap_2d(&tm_s, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, p.scales, p.N, p.K / kGroup, p.N * 2,
                     kTileW, 1, CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;

  Args a{};
  a.M = static_cast<int>(p.M);
  a.N = static_cast<int>(p.N);
  a.K = static_cast<int>(p.K);
  a.KB = static_cast<int>(p.K / kUnitK);
  a.n_tiles = static_cast<int>((p.N + kTileW - 1) / kTileW);
  a.dp_tiles = s.dp_tiles;
  a.sk_units = static_cast<int>(s.sk_units);
  a.act_3d = act_3d;
  a.scales = static_cast<const __half*>(p.scales);
  a.bias = static_cast<const __nv_bfloat16*>(p.bias);
  a.Y = static_cast<__nv_bfloat16*>(p.Y);
  a.counters = static_cast<uint32_t*>(p.workspace);
  a.ws = reinterpret_cast<float*>(static_cast<uint8_t*>(p.workspace) + kCounterBytes);
  a.err = p.error_word;
  a.timeout_ns = p.timeout_ns;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(s.grid));
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = use_pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, tm_act, tm_w, tm_s, a);
}

// The compiled configurations:
//   {act_tile, dequant_wgs, group_scale, stages, partial accumulators}.
#define W4A16_GEMM_INSTANCES(X) \
  X(16, 2, true, 16, 1)         \
  X(32, 2, true, 12, 1)         \
  X(64, 2, true, 8, 1)          \
  X(64, 2, false, 8, 1)         \
  X(128, 2, false, 5, 1)        \
  X(256, 2, false, 3, 1)

}  // namespace

size_t gemm_smem_bytes(const GemmKernelConfig& c) {
#define W4A16_SMEM_CASE(BA, NWG, GRP, ST, NA)                                            \
  if (c.act_tile == BA && c.worker_wgs == NWG && c.group_scale == GRP && c.stages == ST && \
      c.accumulators == NA)                                                                \
    return Cfg<BA, NWG, GRP, ST, NA>::kSmem;
  W4A16_GEMM_INSTANCES(W4A16_SMEM_CASE)
#undef W4A16_SMEM_CASE
  return 0;
}

bool gemm_config_available(const GemmKernelConfig& c) { return gemm_smem_bytes(c) != 0; }

size_t gemm_workspace_bytes(const GemmKernelConfig& c, const GemmSchedule& s, int64_t M,
                            int64_t N, int64_t K) {
  (void)M;
  (void)N;
  (void)K;
  if (s.sk_units == 0) return 0;
  return kCounterBytes + static_cast<size_t>(s.grid) * 2 * c.act_tile * kTileW * sizeof(float);
}

cudaError_t launch_gemm_tc(const GemmKernelConfig& c, const GemmSchedule& s,
                           const GemmProblem& p, bool use_pdl, cudaStream_t stream) {
#define W4A16_LAUNCH_CASE(BA, NWG, GRP, ST, NA)                                          \
  if (c.act_tile == BA && c.worker_wgs == NWG && c.group_scale == GRP && c.stages == ST && \
      c.accumulators == NA)                                                                \
    return launch_instance<BA, NWG, GRP, ST, NA>(s, p, use_pdl, stream);
  W4A16_GEMM_INSTANCES(W4A16_LAUNCH_CASE)
#undef W4A16_LAUNCH_CASE
  return cudaErrorInvalidConfiguration;
}

#ifdef W4A16_TRACE
extern "C" int w4a16_debug_set_trace(unsigned long long* buf) {
  return cudaMemcpyToSymbol(g_trace, &buf, sizeof(buf)) == cudaSuccess ? 0 : 1;
}
extern "C" int w4a16_debug_set_trace_units(unsigned long long* buf) {
  return cudaMemcpyToSymbol(g_trace_units, &buf, sizeof(buf)) == cudaSuccess ? 0 : 1;
}
#endif

cudaError_t launch_wait_timeout_selftest(uint32_t* error_word, uint64_t timeout_ns,
                                         cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(32);
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, wait_timeout_selftest_kernel, error_word, timeout_ns);
}

}  // namespace w4a16
