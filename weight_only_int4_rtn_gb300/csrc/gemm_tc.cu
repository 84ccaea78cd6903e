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
//     unit: TMA brings the packed codes (128 rows x 64 B), the 128 scales of
//     that group and the activation slice; the workers convert; one thread
//     issues 8 MMAs of K = 16.
//
// Two scaling modes:
//   group_scale = true:  the weight operand holds the integer codes (exact in
//     bf16); each unit's MMA result D_g is the integer-code partial sum of one
//     group, which the workers read back and accumulate as acc += s[g, n] *
//     D_g in fp32 registers.  Cheapest conversion; used for small act_tile.
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
// Warp roles (blockDim = 64 + 128 * worker_wgs):
//   warp 0      TMA producer (one lane)
//   warp 1      TMEM allocator; MMA issuer (one lane)
//   warps 2..   workers: dequant into TMEM, read accumulators, epilogue.
//               A warp may only touch TMEM lanes 32 * (warp % 4) .. + 31, so
//               each worker thread owns weight row 32 * (warp % 4) + lane.
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

namespace w4a16 {

namespace {

constexpr int kUnitK = 128;               // K values per unit (one group)
constexpr int kWBytes = kTileW * kUnitK / 2;   // packed codes per unit: 8 KiB
constexpr int kSBytes = kTileW * 2;            // scales per unit: 256 B
constexpr int kAStages = 4;                    // weight-operand stages in TMEM
constexpr int kAStageCols = kUnitK / 2;        // 64 TMEM columns per stage
constexpr int kDCol = kAStages * kAStageCols;  // accumulators start at column 256
constexpr uint32_t kTmemCols = 512;

struct Args {
  int M, N, K, KB;
  int n_tiles;
  int dp_tiles;
  int sk_units;
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

// CTA that owns stream-K unit u under the balanced split.
__device__ __forceinline__ int sk_owner(int u, int C, int sk_units) {
  return static_cast<int>(((static_cast<int64_t>(u) + 1) * C - 1) / sk_units);
}

struct Shared {
  uint64_t full[16];
  uint64_t empty[16];
  uint64_t afull[kAStages];
  uint64_t aempty[kAStages];
  uint64_t dfull[2];
  uint64_t dempty[2];
  uint64_t mma_done;
  uint64_t wsync;             // worker-only barrier (bounded waits, unlike bar.sync)
  uint32_t tmem_base;
  int abort_flag;
  int fixup_last;
};

// ------------------------------------------------------------- bounded waits
__device__ __forceinline__ void record_timeout(const Args& a, Shared* sh) {
  *reinterpret_cast<volatile int*>(&sh->abort_flag) = 1;
  atomicOr(a.err, 1u);
}

// Single-thread wait.  false = gave up (timeout, or another role gave up).
__device__ bool wait_one(uint64_t* bar, uint32_t parity, const Args& a, Shared* sh) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t spin = 1;; ++spin) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((spin & 31) == 0) {
      if (*reinterpret_cast<volatile int*>(&sh->abort_flag)) return false;
      if (ptx::globaltimer_ns() - t0 > a.timeout_ns) {
        record_timeout(a, sh);
        return false;
      }
    }
  }
}

// Warp-uniform wait: every lane observes the phase; the give-up decision is
// lane 0's and is shared, so the warp stays converged for .sync.aligned ops.
__device__ bool wait_warp(uint64_t* bar, uint32_t parity, const Args& a, Shared* sh) {
  const int lane = threadIdx.x & 31;
  uint64_t t0 = 0;
  for (uint32_t spin = 0;; ++spin) {
    const bool ok = ptx::mbar_try_wait(bar, parity);
    if (__all_sync(0xffffffffu, ok)) return true;
    if ((spin & 31) == 31) {
      int give_up = 0;
      if (lane == 0) {
        const uint64_t now = ptx::globaltimer_ns();
        if (t0 == 0) t0 = now;
        if (*reinterpret_cast<volatile int*>(&sh->abort_flag)) {
          give_up = 1;
        } else if (now - t0 > a.timeout_ns) {
          record_timeout(a, sh);
          give_up = 1;
        }
      }
      give_up = __shfl_sync(0xffffffffu, give_up, 0);
      if (give_up) return false;
    }
  }
}

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

__device__ __forceinline__ float bits_f32(uint32_t u) { return __uint_as_float(u); }

template <int BA, int NWG, bool GRP, int STAGES>
struct Cfg {
  static constexpr int kActBox = BA * 128;                        // bytes per 64-k box
  static constexpr int kStageRaw = 2 * kActBox + kWBytes + kSBytes;
  static constexpr int kStage = (kStageRaw + 1023) / 1024 * 1024;
  static constexpr int kThreads = 64 + 128 * NWG;
  static constexpr int kColsPerWg = BA / NWG;                     // D columns per worker WG
  static constexpr int kDequantCols = kAStageCols / NWG;          // A-stage columns per WG
  static constexpr int kChunk = kColsPerWg < 32 ? kColsPerWg : 32;
  static constexpr size_t kSmem = static_cast<size_t>(STAGES) * kStage + 1024 + sizeof(Shared);
  static constexpr uint32_t kTx = 2 * kActBox + kWBytes + kSBytes;
  static_assert(BA % 16 == 0 && BA >= 16 && BA <= 256, "tcgen05 N for M=128");
  static_assert(GRP ? (2 * BA <= 256) : (BA <= 256), "accumulators fit in TMEM");
  static_assert(STAGES <= 16, "barrier arrays");
  static_assert(kColsPerWg >= 8, "at least 8 accumulator columns per worker warpgroup");
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

// Write `cnt` accumulator columns [col0, col0 + cnt) of this thread's weight
// row either to Y (whole tile) or to this CTA's partial slot.
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
    float* slot = a.ws + (static_cast<int64_t>(blockIdx.x) * 2 + u.slot) * (BA * kTileW);
#pragma unroll
    for (int j = 0; j < CNT; ++j) slot[(col0 + j) * kTileW + row] = v[j];
  }
}

// Barrier among the worker warps built on an mbarrier, so that a worker warp
// that gave up after a timeout cannot leave the others blocked forever.
__device__ bool worker_sync(Shared* sh, uint32_t& nsync, const Args& a) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) ptx::mbar_arrive(&sh->wsync);
  const bool ok = wait_warp(&sh->wsync, nsync & 1, a, sh);
  ++nsync;
  return ok;
}

// After this CTA wrote a partial tile: count the arrival; the CTA that
// completes the count sums every partial of the tile in k order and stores Y.
template <int BA, int NWG>
__device__ bool stream_k_fixup(const Args& a, const Unit& u, Shared* sh, int row, int wg,
                               uint32_t& nsync) {
  constexpr int kCols = BA / NWG;
  const int C = gridDim.x;
  __threadfence();
  if (!worker_sync(sh, nsync, a)) return false;
  const int KB = a.KB;
  const int c_lo = sk_owner(u.sk_tile * KB, C, a.sk_units);
  const int c_hi = sk_owner(u.sk_tile * KB + KB - 1, C, a.sk_units);
  if (threadIdx.x == 64) {
    const uint32_t old = atomicAdd(&a.counters[u.sk_tile], 1u);
    const bool last = (old == static_cast<uint32_t>(c_hi - c_lo));
    if (last) atomicExch(&a.counters[u.sk_tile], 0u);
    sh->fixup_last = last ? 1 : 0;
  }
  if (!worker_sync(sh, nsync, a)) return false;
  if (!sh->fixup_last) return true;
  __threadfence();
  const int n0 = (u.tile % a.n_tiles) * kTileW;
  const int m0 = (u.tile / a.n_tiles) * BA;
  const int n = n0 + row;
  const float bias_n = (a.bias != nullptr && n < a.N) ? __bfloat162float(a.bias[n]) : 0.0f;
  const int col_begin = wg * kCols;
  for (int j = 0; j < kCols; ++j) {
    const int col = col_begin + j;
    float acc = 0.0f;
    for (int cc = c_lo; cc <= c_hi; ++cc) {
      const int first_tile_of_cc =
          static_cast<int>((static_cast<int64_t>(cc) * a.sk_units) / C) / KB;
      const int slot = (u.sk_tile == first_tile_of_cc) ? 0 : 1;
      const float* src = a.ws + (static_cast<int64_t>(cc) * 2 + slot) * (BA * kTileW);
      acc += __ldcg(src + col * kTileW + row);
    }
    const int m = m0 + col;
    if (n < a.N && m < a.M) a.Y[static_cast<int64_t>(m) * a.N + n] = __float2bfloat16_rn(acc + bias_n);
  }
  return true;
}

template <int BA, int NWG, bool GRP, int STAGES>
__global__ void __launch_bounds__(Cfg<BA, NWG, GRP, STAGES>::kThreads, 1)
    w4a16_gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_act,
                         const __grid_constant__ CUtensorMap tm_w,
                         const __grid_constant__ CUtensorMap tm_s, const Args a) {
  using C = Cfg<BA, NWG, GRP, STAGES>;
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
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&sh->full[s], 1);
      ptx::mbar_init(&sh->empty[s], 1);
    }
    for (int s = 0; s < kAStages; ++s) {
      ptx::mbar_init(&sh->afull[s], 4 * NWG);
      ptx::mbar_init(&sh->aempty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&sh->dfull[s], 1);
      ptx::mbar_init(&sh->dempty[s], 4 * NWG);
    }
    ptx::mbar_init(&sh->mma_done, 1);
    ptx::mbar_init(&sh->wsync, 4 * NWG);
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

  // Inputs may be produced by the previous kernel on the stream.
  ptx::grid_dependency_wait();
  ptx::grid_launch_dependents();

  Sched sched;
  sched.init(a);

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      int issued = 0;
      for (int i = 0; i < sched.total; ++i) {
        const int stage = i % STAGES;
        const uint32_t ph = (i / STAGES) & 1;
        if (!wait_one(&sh->empty[stage], ph ^ 1, a, sh)) break;
        const Unit u = sched.get(i);
        const int n0 = (u.tile % a.n_tiles) * kTileW;
        const int m0 = (u.tile / a.n_tiles) * BA;
        ptx::mbar_arrive_expect_tx(&sh->full[stage], C::kTx);
        ptx::tma_load_2d(act_box(stage, 0), &tm_act, &sh->full[stage], u.kb * kUnitK, m0);
        ptx::tma_load_2d(act_box(stage, 1), &tm_act, &sh->full[stage], u.kb * kUnitK + 64, m0);
        ptx::tma_load_2d(w_tile(stage), &tm_w, &sh->full[stage], u.kb * (kUnitK / 2), n0);
        ptx::tma_load_2d(s_tile(stage), &tm_s, &sh->full[stage], n0, u.kb);
        issued = i + 1;
      }
      if (*reinterpret_cast<volatile int*>(&sh->abort_flag)) {
        // let the copies still in flight land before the CTA exits
        const int first = issued > STAGES ? issued - STAGES : 0;
        for (int i = first; i < issued; ++i) {
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
      int seg = 0;
      for (int i = 0; i < sched.total; ++i) {
        const int stage = i % STAGES;
        const int as = i % kAStages;
        const Unit u = sched.get(i);
        if (!wait_one(&sh->full[stage], (i / STAGES) & 1, a, sh)) break;
        if (!wait_one(&sh->afull[as], (i / kAStages) & 1, a, sh)) break;
        int db = 0;
        bool fresh;
        if (GRP) {
          db = i & 1;
          if (!wait_one(&sh->dempty[db], ((i >> 1) & 1) ^ 1, a, sh)) break;
          fresh = true;
        } else {
          fresh = u.seg_first;
          if (u.seg_first && !wait_one(&sh->dempty[0], (seg & 1) ^ 1, a, sh)) break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem + kDCol + db * BA;
        const uint32_t a_tmem = tmem + as * kAStageCols;
        const uint32_t b0 = ptx::smem_u32(act_box(stage, 0));
        const uint32_t b1 = ptx::smem_u32(act_box(stage, 1));
#pragma unroll
        for (int kk = 0; kk < kUnitK / 16; ++kk) {
          const uint32_t baddr = (kk < 4 ? b0 : b1) + (kk & 3) * 32;
          ptx::mma_bf16_tmem_a(d_tmem, a_tmem + kk * 8, ptx::smem_desc_sw128(baddr), idesc,
                               (kk > 0 || !fresh) ? 1u : 0u);
        }
        ptx::mma_commit(&sh->empty[stage]);
        ptx::mma_commit(&sh->aempty[as]);
        if (GRP) {
          ptx::mma_commit(&sh->dfull[db]);
        } else if (u.seg_last) {
          ptx::mma_commit(&sh->dfull[0]);
          ++seg;
        }
      }
      // all MMAs of this CTA complete before TMEM is freed
      ptx::mma_commit(&sh->mma_done);
      const uint64_t t0 = ptx::globaltimer_ns();
      while (!ptx::mbar_try_wait(&sh->mma_done, 0)) {
        if (ptx::globaltimer_ns() - t0 > a.timeout_ns) {
          record_timeout(a, sh);
          break;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ workers
    const int wg = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    constexpr int kWords = 16 / NWG;                 // 32-bit code words per thread per unit
    constexpr int kCols = C::kColsPerWg;

    float acc[GRP ? kCols : 1];
    struct Pending {
      bool valid;
      Unit u;
      int i;
      int seg;
      float scale;
    } pend;
    pend.valid = false;
    int seg = 0;
    uint32_t nsync = 0;
    bool ok = true;

    // D -> acc (group mode) or D -> output (dequant mode) for a finished unit.
    auto finish = [&](const Pending& p) -> bool {
      const int n = (p.u.tile % a.n_tiles) * kTileW + row;
      const float bias_n =
          (a.bias != nullptr && n < a.N) ? __bfloat162float(a.bias[n]) : 0.0f;
      if constexpr (GRP) {
        const int db = p.i & 1;
        if (!wait_warp(&sh->dfull[db], (p.i >> 1) & 1, a, sh)) return false;
        ptx::tc_fence_after();
#pragma unroll
        for (int c0 = 0; c0 < kCols; c0 += C::kChunk) {
          uint32_t r[C::kChunk];
          tmem_ld_cols<C::kChunk>(lane_base + kDCol + db * BA + wg * kCols + c0, r);
#pragma unroll
          for (int j = 0; j < C::kChunk; ++j) {
            const float d = bits_f32(r[j]);
            acc[c0 + j] = p.u.seg_first ? p.scale * d : fmaf(p.scale, d, acc[c0 + j]);
          }
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&sh->dempty[db]);
        if (p.u.seg_last) {
          emit_cols<BA, kCols>(a, p.u, row, wg * kCols, acc, bias_n);
          if (!p.u.whole && !stream_k_fixup<BA, NWG>(a, p.u, sh, row, wg, nsync)) return false;
        }
      } else {
        if (!wait_warp(&sh->dfull[0], p.seg & 1, a, sh)) return false;
        ptx::tc_fence_after();
#pragma unroll 1
        for (int c0 = 0; c0 < kCols; c0 += C::kChunk) {
          uint32_t r[C::kChunk];
          float v[C::kChunk];
          tmem_ld_cols<C::kChunk>(lane_base + kDCol + wg * kCols + c0, r);
#pragma unroll
          for (int j = 0; j < C::kChunk; ++j) v[j] = bits_f32(r[j]);
          emit_cols<BA, C::kChunk>(a, p.u, row, wg * kCols + c0, v, bias_n);
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&sh->dempty[0]);
        if (!p.u.whole && !stream_k_fixup<BA, NWG>(a, p.u, sh, row, wg, nsync)) return false;
      }
      return true;
    };

    for (int i = 0; i < sched.total && ok; ++i) {
      const int stage = i % STAGES;
      const int as = i % kAStages;
      const Unit u = sched.get(i);
      if (!wait_warp(&sh->full[stage], (i / STAGES) & 1, a, sh)) { ok = false; break; }

      // this thread's 64 B of packed codes, stored with the 64-byte swizzle:
      // 16-byte chunk c of row r sits at chunk position c ^ ((r >> 1) & 3)
      const uint32_t wrow = ptx::smem_u32(w_tile(stage)) + row * 64;
      uint32_t words[kWords];
#pragma unroll
      for (int q = 0; q < kWords / 4; ++q) {
        const int chunk = wg * (kWords / 4) + q;
        const uint4 v = ptx::lds128(wrow + ((chunk ^ ((row >> 1) & 3)) << 4));
        words[4 * q + 0] = v.x;
        words[4 * q + 1] = v.y;
        words[4 * q + 2] = v.z;
        words[4 * q + 3] = v.w;
      }
      const float scale = __half2float(s_tile(stage)[row]);

      uint32_t opnd[4 * kWords];
#pragma unroll
      for (int q = 0; q < kWords; ++q) codes_to_bf16(words[q], &opnd[4 * q]);
      if constexpr (!GRP) {
        const __nv_bfloat16 hi = __float2bfloat16_rn(scale);
        const float lo_f = scale - __bfloat162float(hi);        // exact
        const __nv_bfloat16 lo = __float2bfloat16_rn(lo_f);     // exact
        const uint32_t hi_bits = static_cast<uint32_t>(__bfloat16_as_ushort(hi));
        const uint32_t lo_bits = static_cast<uint32_t>(__bfloat16_as_ushort(lo));
        const uint32_t s_hi2 = hi_bits | (hi_bits << 16);
        const uint32_t s_lo2 = lo_bits | (lo_bits << 16);
#pragma unroll
        for (int q = 0; q < 4 * kWords; ++q) opnd[q] = scale_pair(opnd[q], s_hi2, s_lo2);
      }

      if (!wait_warp(&sh->aempty[as], ((i / kAStages) & 1) ^ 1, a, sh)) { ok = false; break; }
      ptx::tc_fence_after();
      const uint32_t a_addr = lane_base + as * kAStageCols + wg * C::kDequantCols;
#pragma unroll
      for (int q = 0; q < (4 * kWords) / 16; ++q) ptx::tmem_st_x16(a_addr + 16 * q, &opnd[16 * q]);
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&sh->afull[as]);

      if (pend.valid) {
        if (!finish(pend)) { ok = false; break; }
        pend.valid = false;
      }
      if (GRP || u.seg_last) {
        pend.valid = true;
        pend.u = u;
        pend.i = i;
        pend.seg = seg;
        pend.scale = scale;
      }
      if (!GRP && u.seg_last) ++seg;
    }
    if (ok && pend.valid) finish(pend);
  }

  // ------------------------------------------------------------- teardown
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem, kTmemCols);
}

// One-thread kernel whose wait can never complete: exercises the bounded
// wait and the error word without faulting or hanging the GPU.
__global__ void wait_timeout_selftest_kernel(uint32_t* err, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ Shared sh;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    ptx::fence_mbar_init();
    sh.abort_flag = 0;
    Args a{};
    a.err = err;
    a.timeout_ns = timeout_ns;
    (void)wait_one(&bar, 0, a, &sh);   // nobody arrives: times out
  }
}

template <int BA, int NWG, bool GRP, int STAGES>
cudaError_t launch_instance(const GemmSchedule& s, const GemmProblem& p, bool use_pdl,
                            cudaStream_t stream) {
  using C = Cfg<BA, NWG, GRP, STAGES>;
  auto kernel = w4a16_gemm_tc_kernel<BA, NWG, GRP, STAGES>;

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
  if (encode_tmap_2d(&tm_act, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.A, p.K, p.M, p.K * 2, 64, BA,
                     CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  if (encode_tmap_2d(&tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.packed, p.K / 2, p.N, p.K / 2, 64,
                     kTileW, CU_TENSOR_MAP_SWIZZLE_64B) != CUDA_SUCCESS)
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
  a.bias = static_cast<const __nv_bfloat16*>(p.bias);
  a.Y = static_cast<__nv_bfloat16*>(p.Y);
  a.ws = static_cast<float*>(p.workspace);
  a.counters = reinterpret_cast<uint32_t*>(
      static_cast<uint8_t*>(p.workspace) +
      static_cast<size_t>(s.grid) * 2 * BA * kTileW * sizeof(float));
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

// The compiled configurations: {act_tile, worker_wgs, group_scale, stages}.
#define W4A16_GEMM_INSTANCES(X) \
  X(16, 2, true, 16)            \
  X(32, 2, true, 12)            \
  X(64, 2, true, 8)             \
  X(64, 2, false, 8)            \
  X(128, 2, true, 5)            \
  X(128, 2, false, 5)           \
  X(256, 2, false, 3)

}  // namespace

size_t gemm_smem_bytes(const GemmKernelConfig& c) {
#define W4A16_SMEM_CASE(BA, NWG, GRP, ST)                                                      \
  if (c.act_tile == BA && c.worker_wgs == NWG && c.group_scale == GRP && c.stages == ST) \
    return Cfg<BA, NWG, GRP, ST>::kSmem;
  W4A16_GEMM_INSTANCES(W4A16_SMEM_CASE)
#undef W4A16_SMEM_CASE
  return 0;
}

bool gemm_config_available(const GemmKernelConfig& c) { return gemm_smem_bytes(c) != 0; }

size_t gemm_workspace_bytes(const GemmKernelConfig& c, const GemmSchedule& s, int64_t M,
                            int64_t N, int64_t K) {
  (void)K;
  if (s.sk_units == 0) return 0;
  const int64_t tiles = gemm_tiles(c, M, N);
  const int64_t sk_tiles = tiles - s.dp_tiles;
  const size_t slots = static_cast<size_t>(s.grid) * 2 * c.act_tile * kTileW * sizeof(float);
  const size_t counters = static_cast<size_t>(sk_tiles) * sizeof(uint32_t);
  return slots + ((counters + 255) / 256) * 256;
}

cudaError_t launch_gemm_tc(const GemmKernelConfig& c, const GemmSchedule& s,
                           const GemmProblem& p, bool use_pdl, cudaStream_t stream) {
#define W4A16_LAUNCH_CASE(BA, NWG, GRP, ST)                                                    \
  if (c.act_tile == BA && c.worker_wgs == NWG && c.group_scale == GRP && c.stages == ST) \
    return launch_instance<BA, NWG, GRP, ST>(s, p, use_pdl, stream);
  W4A16_GEMM_INSTANCES(W4A16_LAUNCH_CASE)
#undef W4A16_LAUNCH_CASE
  return cudaErrorInvalidConfiguration;
}

cudaError_t launch_wait_timeout_selftest(uint32_t* error_word, uint64_t timeout_ns,
                                         cudaStream_t stream) {
  wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(error_word, timeout_ns);
  return cudaGetLastError();
}

}  // namespace w4a16
