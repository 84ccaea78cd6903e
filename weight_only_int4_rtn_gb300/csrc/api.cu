// C ABI of the W4A16 library: argument checks (metadata only), the GEMM
// variant catalogue and its per-shape table, tuning by measurement, the
// device error word and the TMA descriptor encoder.
//
// The per-shape table mirrors the cached, frozen, optionally autotuned kernel
// choice of "Kernel dispatch and Humming quantization in PhyAI", sections
// "Keep selection work out of repeated inference" (prepared selections are
// memoized and reused) and "Put deployment choices in a policy" (an error,
// never a silent fallback, when no implementation is usable).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cctype>
#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <fstream>
#include <map>
#include <mutex>
#include <sstream>
#include <string>
#include <tuple>
#include <vector>

#include "../../include/w4a16.h"
#include "kernels.h"

namespace w4a16 {

// Device error word: bit 0 = a bounded wait ran out.  One per device that
// loads this library.
__device__ uint32_t g_error_word;

namespace {

std::atomic<uint64_t> g_timeout_ns{2000000000ull};
// w4a16_set_weights_static: GEMM launches may read their weights before the
// dependency wait of programmatic dependent launch
std::atomic<int> g_weights_static{0};
thread_local char g_error_detail[256] = "";

// Record a failed CUDA call for w4a16_last_error_detail and clear the
// runtime's per-thread last error, so that it does not surface in an
// unrelated later call of this library or of the caller.
int cuda_failure(cudaError_t e, const char* where) {
  std::snprintf(g_error_detail, sizeof(g_error_detail), "%s: %s (%d)", where,
                cudaGetErrorString(e), static_cast<int>(e));
  (void)cudaGetLastError();
  if (std::getenv("W4A16_LOG") != nullptr) std::fprintf(stderr, "w4a16: %s\n", g_error_detail);
  return W4A16_ERR_CUDA;
}
std::atomic<uint64_t> g_launches{0};

constexpr int kMaxDevices = 64;

// SM count assumed by host-only queries when no CUDA device is visible
// (GB300: 152 SMs); launches always use the device's own count.
constexpr int kDefaultSms = 152;

struct DeviceInfo {
  bool ready = false;
  int num_sms = 0;
  uint32_t* error_word = nullptr;
  // clusters of 2, 4, 8 CTAs that each need a whole SM (every tcgen05 GEMM
  // instance) the GPU holds at once; -1: unknown
  int whole_sm_clusters[3] = {-1, -1, -1};
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mutex;

// Never launched: the occupancy query's stand-in for a CTA that needs a
// whole SM (512 threads, more than half of the shared memory).
__global__ void whole_sm_cta_kernel() {}
constexpr int kWholeSmSmem = 200 * 1024;

// Clusters of `cluster` whole-SM CTAs resident at once on the current device
// (a cluster's CTAs share one GPC, so this can be below SMs / cluster).
int query_whole_sm_clusters(int cluster) {
  if (cudaFuncSetAttribute(whole_sm_cta_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kWholeSmSmem) != cudaSuccess)
    return -1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(cluster));
  cfg.blockDim = dim3(512);
  cfg.dynamicSmemBytes = kWholeSmSmem;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = static_cast<unsigned>(cluster);
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, whole_sm_cta_kernel, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    return -1;
  }
  return n;
}

// Current device's SM count, error-word address and whole-SM cluster
// capacity (looked up once).
bool device_info(DeviceInfo& out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return false;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return false;
    d.num_sms = sms;
    d.error_word = static_cast<uint32_t*>(p);
    // host-side queries (no stream work); relaxed capture mode so that a
    // first call inside a stream capture leaves the capture intact
    cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
    const bool swapped = cudaThreadExchangeStreamCaptureMode(&mode) == cudaSuccess;
    for (int i = 0; i < 3; ++i) d.whole_sm_clusters[i] = query_whole_sm_clusters(2 << i);
    if (swapped) (void)cudaThreadExchangeStreamCaptureMode(&mode);
    d.ready = true;
  }
  out = d;
  return true;
}

// Clusters of `cluster` (2, 4 or 8) whole-SM CTAs the current device holds
// at once; -1 without a device.
int resident_whole_sm_clusters(int cluster) {
  DeviceInfo dev;
  if (!device_info(dev)) return -1;
  const int i = cluster == 2 ? 0 : cluster == 4 ? 1 : cluster == 8 ? 2 : -1;
  return i < 0 ? -1 : dev.whole_sm_clusters[i];
}

// The current device's SM count (the GB300 count without a device).
int current_sms() {
  DeviceInfo dev;
  return device_info(dev) ? dev.num_sms : kDefaultSms;
}

// ------------------------------------------------------------ catalogue
struct Variant {
  const char* name;
  GemmKernelConfig cfg;
  bool stream_k;   // false: whole tiles only (data parallel)
  int min_units;   // stream-K: at least this many units per CTA (fewer CTAs and
                   // fewer split tiles on small problems)
  double unit_us;  // measured time of one unit (128 weight rows x unit_groups groups)
                   // in steady state on GB300, for the selection rule
  double head_us = -1.0;   // launch-to-steady-state cost if not the common one
  double split_us = -1.0;  // split-tile fixup cost if not the common model's
  int csk = 0;             // > 1: cluster split-K with clusters of up to csk CTAs
};

const Variant kVariants[] = {
    {"tc_a16_grp_sk", {16, 2, true, 16}, true, 1, 0.44},
    {"tc_a32_grp_sk", {32, 2, true, 12}, true, 1, 0.57},
    {"tc_a64_grp_sk", {64, 2, true, 8}, true, 1, 1.30},
    {"tc_a64_deq_sk", {64, 1, false, 8}, true, 1, 0.60},
    {"tc_a128_deq_sk", {128, 1, false, 5}, true, 1, 0.57},
    {"tc_a256_deq_sk", {256, 1, false, 3}, true, 1, 0.63},
    {"tc_a16_grp_dp", {16, 2, true, 16}, false, 1, 0.38},
    {"tc_a64_grp_dp", {64, 2, true, 8}, false, 1, 1.10},
    {"tc_a128_deq_dp", {128, 1, false, 5}, false, 1, 0.68},
    {"tc_a256_deq_dp", {256, 1, false, 3}, false, 1, 0.95},
    {"tc_a16_grp_sk4", {16, 2, true, 16}, true, 4, 0.43},
    {"tc_a16_grp_sk8", {16, 2, true, 16}, true, 8, 0.39},
    {"tc_a32_grp_sk4", {32, 2, true, 12}, true, 4, 0.55},
    {"tc_a64_grp_sk4", {64, 2, true, 8}, true, 4, 1.27},
    {"tc_a64_grp_sk8", {64, 2, true, 8}, true, 8, 1.06},
    {"tc_a16_deq2_sk", {16, 2, false, 16}, true, 1, 0.48},
    {"tc_a32_deq2_sk", {32, 2, false, 12}, true, 1, 0.48},
    {"tc_a64_deq2_sk", {64, 2, false, 8}, true, 1, 0.50},
    {"tc_a128_deq2_sk", {128, 2, false, 4}, true, 1, 0.65},
    {"tc_a16_deq2_dp", {16, 2, false, 16}, false, 1, 0.45},
    {"tc_a64_deq2_dp", {64, 2, false, 8}, false, 1, 0.47},
    {"tc_a128_deq2_dp", {128, 2, false, 4}, false, 1, 0.70},
    // units of two groups (one 16 KiB copy of codes per unit)
    {"tc_a16_grp_sk_u2", {16, 2, true, 8, 2}, true, 1, 0.84},
    {"tc_a16_grp_sk8_u2", {16, 2, true, 8, 2}, true, 8, 0.73},
    {"tc_a16_grp_dp_u2", {16, 2, true, 8, 2}, false, 1, 0.76},
    {"tc_a16_deq2_sk_u2", {16, 2, false, 8, 2}, true, 1, 0.92},
    {"tc_a16_deq2_dp_u2", {16, 2, false, 8, 2}, false, 1, 0.86},
    {"tc_a32_deq2_sk_u2", {32, 2, false, 6, 2}, true, 1, 1.01},
    {"tc_a64_deq2_sk_u2", {64, 2, false, 4, 2}, true, 1, 1.08},
    {"tc_a64_deq2_dp_u2", {64, 2, false, 4, 2}, false, 1, 0.98},
    // cluster split-K: a tile's K range over the CTAs of one cluster (at
    // most 8), partials summed through distributed shared memory; for few
    // tiles of long K
    {"tc_a16_grp_csk", {16, 2, true, 16}, false, 1, 0.44, -1.0, 0.3, 8},
    {"tc_a16_grp_csk_u2", {16, 2, true, 8, 2}, false, 1, 0.80, -1.0, 0.3, 8},
    {"tc_a32_deq2_csk", {32, 2, false, 12}, false, 1, 0.48, -1.0, 0.3, 8},
    {"tc_a64_deq2_csk", {64, 2, false, 8}, false, 1, 0.50, -1.0, 0.35, 8},
    {"tc_a128_deq2_csk", {128, 2, false, 4}, false, 1, 0.65, -1.0, 0.5, 8},
    // row-block warp-MMA kernel for M <= 1, 2, 4, 8, 16: unit_us is the time
    // of one (row block, group) item per warp on a full SM (rb_cost)
    {"rb_m1", {1, 1, true, 0, 1, kFmtInt4, true, true}, false, 1, 1.07, 1.85, 0.0},
    {"rb_m2", {2, 1, true, 0, 1, kFmtInt4, true, true}, false, 1, 1.20, 1.85, 0.0},
    {"rb_m4", {4, 1, true, 0, 1, kFmtInt4, true, true}, false, 1, 1.33, 1.85, 0.0},
    {"rb_m8", {8, 1, true, 0, 1, kFmtInt4, true, true}, false, 1, 1.45, 1.85, 0.0},
    {"rb_m16", {16, 1, true, 0, 1, kFmtInt4, true, true}, false, 1, 2.30, 1.85, 0.0},
    // CUDA-core streaming kernel for M <= 1, 2, 4, 8: unit_us is the time of
    // one unit on one worker (a warp; many warps share an SM)
    {"simt_m1_sk", {1, 1, true, 2, 1, kFmtInt4, true}, true, 1, 6.0, 2.0, 0.8},
    {"simt_m2_sk", {2, 1, true, 2, 1, kFmtInt4, true}, true, 1, 5.2, 2.0, 0.8},
    {"simt_m4_sk", {4, 1, true, 2, 1, kFmtInt4, true}, true, 1, 7.0, 2.0, 0.8},
    {"simt_m8_sk", {8, 1, true, 2, 1, kFmtInt4, true}, true, 1, 10.2, 2.0, 0.8},
};
constexpr int kNumVariants = static_cast<int>(sizeof(kVariants) / sizeof(kVariants[0]));

// INT8 weights (W8A16), bf16 activations.
const Variant kVariants8[] = {
    {"w8_tc_a16_grp_sk", {16, 2, true, 10, 1, 8}, true, 1, 0.50},
    {"w8_tc_a16_grp_sk8", {16, 2, true, 10, 1, 8}, true, 8, 0.49},
    {"w8_tc_a16_grp_dp", {16, 2, true, 10, 1, 8}, false, 1, 0.48},
    {"w8_tc_a32_grp_sk", {32, 2, true, 8, 1, 8}, true, 1, 0.63},
    {"w8_tc_a64_deq2_sk", {64, 2, false, 6, 1, 8}, true, 1, 0.73},
    {"w8_tc_a64_deq2_dp", {64, 2, false, 6, 1, 8}, false, 1, 0.70},
    {"w8_tc_a128_deq_sk", {128, 1, false, 4, 1, 8}, true, 1, 0.77},
    {"w8_tc_a128_deq_dp", {128, 1, false, 4, 1, 8}, false, 1, 0.78},
    {"w8_tc_a256_deq_sk", {256, 1, false, 2, 1, 8}, true, 1, 1.36},
    {"w8_tc_a256_deq_dp", {256, 1, false, 2, 1, 8}, false, 1, 1.49},
    // split rings (stages = 2 activation stages + 32 x 4 code stages)
    {"w8_tc_a256_deq_w4_sk", {256, 1, false, 130, 1, 8}, true, 1, 1.3},
};
constexpr int kNumVariants8 = static_cast<int>(sizeof(kVariants8) / sizeof(kVariants8[0]));

// FP4 weights (MXFP4 or NVFP4: the format is set per call), bf16
// activations, dequant mode.
const Variant kVariantsF4[] = {
    {"fp4_tc_a16_deq2_sk", {16, 2, false, 16, 1, kFmtMxfp4}, true, 1, 0.47},
    {"fp4_tc_a16_deq2_dp", {16, 2, false, 16, 1, kFmtMxfp4}, false, 1, 0.47},
    {"fp4_tc_a32_deq2_sk", {32, 2, false, 12, 1, kFmtMxfp4}, true, 1, 0.47},
    {"fp4_tc_a64_deq2_sk", {64, 2, false, 8, 1, kFmtMxfp4}, true, 1, 0.48},
    {"fp4_tc_a64_deq2_dp", {64, 2, false, 8, 1, kFmtMxfp4}, false, 1, 0.48},
    {"fp4_tc_a128_deq_sk", {128, 1, false, 5, 1, kFmtMxfp4}, true, 1, 0.65},
    {"fp4_tc_a128_deq_dp", {128, 1, false, 5, 1, kFmtMxfp4}, false, 1, 0.65},
    {"fp4_tc_a256_deq_sk", {256, 1, false, 3, 1, kFmtMxfp4}, true, 1, 0.84},
    {"fp4_tc_a256_deq_dp", {256, 1, false, 3, 1, kFmtMxfp4}, false, 1, 0.92},
    {"fp4_tc_a16_deq2_sk_u2", {16, 2, false, 8, 2, kFmtMxfp4}, true, 1, 0.89},
    {"fp4_tc_a16_deq2_dp_u2", {16, 2, false, 8, 2, kFmtMxfp4}, false, 1, 0.88},
};
constexpr int kNumVariantsF4 = static_cast<int>(sizeof(kVariantsF4) / sizeof(kVariantsF4[0]));

// Public format codes (FP4A16_MXFP4, FP4A16_NVFP4) to the kernels' ones; 0
// for anything else.
int fp4_format(int public_format) {
  return public_format == FP4A16_MXFP4 ? kFmtMxfp4 : public_format == FP4A16_NVFP4 ? kFmtNvfp4 : 0;
}

Variant variant_f4(int id, int fmt) {
  Variant v = kVariantsF4[id];
  v.cfg.weight_format = fmt;
  return v;
}

int variant_by_name(const std::string& n) {
  for (int i = 0; i < kNumVariants; ++i)
    if (n == kVariants[i].name) return i;
  return -1;
}

bool shape_ok(int64_t M, int64_t N, int64_t K) {
  return M >= 1 && N >= 8 && K >= 128 && (K % kGroup) == 0 && (N % 8) == 0 &&
         M < (1ll << 31) && N < (1ll << 31) && K < (1ll << 31) && M * N < (1ll << 40) &&
         N * K < (1ll << 40);
}

// Row-block kernel: the cost of schedule s in units of one group-item's time
// on a full SM (two CTAs of 8 warps; one for M <= 16, whose CTA takes an SM),
// fitted to GB300 measurements.
// Persistent form: CTA c runs on SM c mod num_sms; an SM with two busy CTAs
// works through 16 group-items per unit of time, one with a single busy CTA
// through 8 / 0.65 (measured: 8 / 0.62); the cost is the busiest SM's.
// Cluster form: waves of the resident CTAs, each wave's warps running their
// share of a row block's K range, plus the cluster's own cost (barriers, the
// distributed shared-memory sum), about 1.3 items a wave.  Clusters that put
// two CTAs on an SM run each item at 1.4 (measured: 2048 x 16384 at M = 1
// and 4, a split of 4 on 256 CTAs 6-7% slower than a split of 2 on 128);
// with one CTA an SM the CTAs beyond the SMs form further waves instead.
double rb_cost(const GemmSchedule& s, int64_t blocks, int64_t KB, int64_t slots, int num_sms) {
  if (s.cluster > 1) {
    const int64_t waves = (blocks * s.cluster + slots - 1) / slots;
    const int64_t per = static_cast<int64_t>(s.cluster) * kRbWarpsPerCta;
    const double load = s.grid <= num_sms || slots <= num_sms ? 0.65 : 1.4;
    return static_cast<double>(waves * ((KB + per - 1) / per)) * load + 1.3 * static_cast<double>(waves);
  }
  const double thr1 = kRbWarpsPerCta / 0.65, thr2 = 2.0 * kRbWarpsPerCta;
  std::vector<double> load(static_cast<size_t>(num_sms), 0.0);
  std::vector<int> busy(static_cast<size_t>(num_sms), 0);
  const int tpc = kRbWarpsPerCta / s.team;
  const int64_t TT = static_cast<int64_t>(s.grid) * tpc;
  for (int c = 0; c < s.grid; ++c) {
    bool any = false;
    for (int j = 0; j < tpc; ++j) {
      const int64_t t = static_cast<int64_t>(c) * tpc + j;
      if (t >= blocks) break;
      load[static_cast<size_t>(c % num_sms)] += static_cast<double>(((blocks - 1 - t) / TT + 1) * KB);
      any = true;
    }
    if (any) ++busy[static_cast<size_t>(c % num_sms)];
  }
  double worst = 0.0;
  for (int i = 0; i < num_sms; ++i)
    if (busy[static_cast<size_t>(i)] > 0)
      worst = std::max(worst, load[static_cast<size_t>(i)] / (busy[static_cast<size_t>(i)] >= 2 ? thr2 : thr1));
  return worst;
}

// single: the problem has the launch to itself (false: one problem of a
// grouped launch, where the row-block kernel's cluster form, one cluster size
// per launch, is not open).
GemmSchedule make_schedule(const Variant& v, int64_t M, int64_t N, int64_t K, int num_sms,
                           bool single = true) {
  GemmSchedule s{};
  if (v.cfg.rb) {
    // Items are (row block, group) pairs.  Persistent: the resident CTAs
    // (fewer when there are fewer teams' worth of row blocks), teams of WK
    // warps, row blocks dealt round-robin to the teams.  Cluster split: one
    // CTA-wide team per row block and cluster rank, in waves of the resident
    // CTAs.  The smallest cost (rb_cost) wins; ties go to the persistent
    // form, then to smaller teams.
    const int64_t blocks = (N + gemv_rb_rows(v.cfg.act_tile) - 1) / gemv_rb_rows(v.cfg.act_tile);
    const int64_t KB = K / kGroup;
    const int64_t slots = static_cast<int64_t>(num_sms) * gemv_rb_ctas_per_sm(v.cfg.act_tile);
    double best = -1.0;
    GemmSchedule c{};
    c.dp_tiles = 0;
    c.sk_units = 0;
    for (int wk = 1; wk <= kRbWarpsPerCta && KB >= wk; wk *= 2) {
      const int64_t tpc = kRbWarpsPerCta / wk;
      c.grid = static_cast<int>(std::min(slots, (blocks + tpc - 1) / tpc));
      c.team = wk;
      c.cluster = 1;
      const double cost = rb_cost(c, blocks, KB, slots, num_sms);
      if (best < 0.0 || cost < best) {
        best = cost;
        s = c;
      }
    }
    for (int S = 2; single && S <= 8 && KB >= S * kRbWarpsPerCta; S *= 2) {
      c.grid = static_cast<int>(blocks * S);
      c.team = kRbWarpsPerCta;
      c.cluster = S;
      const double cost = rb_cost(c, blocks, KB, slots, num_sms);
      if (cost < best) {
        best = cost;
        s = c;
      }
    }
    return s;
  }
  if (v.cfg.simt) {
    // workers (warps) of the CUDA-core streaming kernel: every resident slot
    // (the warps of an SM share its issue slots, so units balance per SM,
    // and a warp left with fewer units frees slots for its neighbours);
    // whole tiles only when there are more split tiles than counters
    const int64_t tiles = gemm_tiles(v.cfg, M, N);
    const int64_t units = tiles * (K / kGroup);
    const int64_t cap = static_cast<int64_t>(num_sms) * gemv_workers_per_sm(v.cfg.act_tile);
    if (tiles > kCountersPerProblem) {
      s.grid = static_cast<int>(tiles < cap ? tiles : cap);
      s.dp_tiles = static_cast<int>(tiles);
      s.sk_units = 0;
      return s;
    }
    s.grid = static_cast<int>(units < cap ? units : cap);
    s.dp_tiles = 0;
    s.sk_units = units;
    return s;
  }
  if (num_sms > kMaxGrid) num_sms = kMaxGrid;
  const int64_t tiles = gemm_tiles(v.cfg, M, N);
  const int64_t KB = K / kGroup / v.cfg.unit_groups;   // units per tile
  const int64_t units = tiles * KB;
  if (v.csk > 1) {
    // the largest power-of-two cluster (<= v.csk, <= KB) such that every
    // tile's cluster is resident at once: tiles * cluster <= SMs and, on a
    // device, tiles <= the clusters of that size it holds at once (a
    // cluster's CTAs share one GPC: on GB300 16 tiles in clusters of 8 ran
    // in two waves, 2048 x 16384 at M = 16 in 21.8 us against 11.1 us for
    // 1024 x 16384); grid 0 when no cluster of 2 or more fits
    const auto resident = [&](int S2) {
      const int r = resident_whole_sm_clusters(S2);
      return r < 0 || tiles <= r;
    };
    int S = 1;
    while (2 * S <= v.csk && 2 * S <= KB && tiles * 2 * S <= num_sms && resident(2 * S)) S *= 2;
    s.cluster = S;
    s.grid = S > 1 ? static_cast<int>(tiles * S) : 0;
    s.dp_tiles = 0;
    s.sk_units = 0;
    return s;
  }
  if (!v.stream_k) {
    s.grid = static_cast<int>(tiles < num_sms ? tiles : num_sms);
    s.dp_tiles = static_cast<int>(tiles);
    s.sk_units = 0;
    return s;
  }
  if (tiles >= num_sms) {
    s.grid = num_sms;
    const int64_t rem = tiles % num_sms;
    if (rem != 0 && rem * KB >= num_sms) {
      s.dp_tiles = static_cast<int>(tiles - rem);
      s.sk_units = rem * KB;
    } else {
      s.dp_tiles = static_cast<int>(tiles);
      s.sk_units = 0;
    }
  } else {
    const int64_t want = (units + v.min_units - 1) / v.min_units;
    s.grid = static_cast<int>(want < num_sms ? want : num_sms);
    s.dp_tiles = 0;
    s.sk_units = units;
  }
  // one arrival counter per split tile
  if (s.sk_units / KB > kCountersPerProblem) {
    s.grid = static_cast<int>(tiles < num_sms ? tiles : num_sms);
    s.dp_tiles = static_cast<int>(tiles);
    s.sk_units = 0;
  }
  return s;
}

int current_sms();

bool variant_ok(const Variant& v, int64_t M, int64_t N, int64_t K) {
  if (!shape_ok(M, N, K)) return false;
  if (v.cfg.simt && M > v.cfg.act_tile) return false;
  if (!gemm_config_available(v.cfg)) return false;
  const int64_t tiles = gemm_tiles(v.cfg, M, N);
  if (tiles * (K / kGroup) >= (1ll << 31)) return false;
  if ((K / kGroup) % v.cfg.unit_groups != 0) return false;
  if (v.csk > 1 && make_schedule(v, M, N, K, current_sms()).cluster < 2) return false;
  return true;
}

bool variant_eligible(int id, int64_t M, int64_t N, int64_t K) {
  return id >= 0 && id < kNumVariants && variant_ok(kVariants[id], M, N, K);
}

bool variant8_eligible(int id, int64_t M, int64_t N, int64_t K) {
  return id >= 0 && id < kNumVariants8 && variant_ok(kVariants8[id], M, N, K);
}

// FP4: the scale rows are N bytes, a TMA stride, so N % 16 == 0.
bool variantf4_eligible(int id, int64_t M, int64_t N, int64_t K) {
  return id >= 0 && id < kNumVariantsF4 && N % 16 == 0 &&
         variant_ok(variant_f4(id, kFmtMxfp4), M, N, K);
}

// Rule for shapes without a table entry: a cost model fitted to GB300
// measurements.  A launch pays a fixed head (launch, set-up, pipeline fill);
// each CTA then runs its units at the variant's per-unit time; a schedule
// that splits tiles over CTAs adds the split-tile fixup (arrival count and
// the last contributor's sum of the partials; more for wider activation
// tiles).  The variant with the smallest estimate wins.
constexpr double kHeadUs = 3.71;
constexpr double kSplitUs = 2.44;
constexpr double kSplitUsPerCol = 0.051;
// a split tile's last contributor sums the others' partials: each
// contributor beyond two lengthens that tail (fitted, with the unit times
// of the two-group and row-block variants, to 72 shapes at M = 1 .. 816:
// mean regret of the rule 1.65% -> 0.73%, worst 35% -> 12%)
constexpr double kSplitUsPerContributor = 0.2;

double estimate_sched(const Variant& v, const GemmSchedule& s, int64_t K, int64_t N = 0,
                      int num_sms = kDefaultSms) {
  const int64_t KB = K / kGroup / v.cfg.unit_groups;
  if (v.cfg.rb) {
    // unit_us: one (row block, group) item per warp on a full SM
    const int64_t rows = gemv_rb_rows(v.cfg.act_tile);
    const int64_t slots = static_cast<int64_t>(num_sms) * gemv_rb_ctas_per_sm(v.cfg.act_tile);
    return v.head_us + rb_cost(s, (N + rows - 1) / rows, K / kGroup, slots, num_sms) * v.unit_us;
  }
  if (s.cluster > 1)
    return (v.head_us >= 0.0 ? v.head_us : kHeadUs) +
           static_cast<double>((KB + s.cluster - 1) / s.cluster) * v.unit_us + v.split_us;
  const int64_t dp_per_cta = (s.dp_tiles + s.grid - 1) / s.grid;
  const int64_t sk_per_cta = (s.sk_units + s.grid - 1) / s.grid;
  double t = (v.head_us >= 0.0 ? v.head_us : kHeadUs) +
             static_cast<double>(dp_per_cta * KB + sk_per_cta) * v.unit_us;
  if (s.sk_units > 0) {
    t += v.split_us >= 0.0 ? v.split_us : kSplitUs + kSplitUsPerCol * v.cfg.act_tile;
    if (!v.cfg.simt && sk_per_cta > 0 && sk_per_cta < KB) {
      const int64_t contributors = (KB + sk_per_cta - 1) / sk_per_cta;
      if (contributors > 2) t += kSplitUsPerContributor * static_cast<double>(contributors - 2);
    }
  }
  return t;
}

double estimate_us(const Variant& v, int64_t M, int64_t N, int64_t K, int num_sms) {
  return estimate_sched(v, make_schedule(v, M, N, K, num_sms), K, N, num_sms);
}

int rule_variant(int64_t M, int64_t N, int64_t K, int num_sms) {
  int best = -1;
  double best_t = 0.0;
  for (int id = 0; id < kNumVariants; ++id) {
    if (!variant_eligible(id, M, N, K)) continue;
    const double t = estimate_us(kVariants[id], M, N, K, num_sms);
    if (best < 0 || t < best_t) {
      best = id;
      best_t = t;
    }
  }
  return best;
}

// ---------------------------------------------------------------- table
// Catalogues with a measured table: the INT4 GEMM, the INT4 GEMM with the
// SwiGLU epilogue (same variants, chosen separately: its best variant can
// differ), the INT8 GEMM and the FP4 GEMM (one catalogue for both formats).
enum Catalogue { kCatInt4 = 0, kCatSwiglu = 1, kCatInt8 = 2, kCatFp4 = 3, kNumCats = 4 };
const char* const kCatTag[kNumCats] = {"", "swiglu", "int8", "fp4"};

std::mutex g_table_mutex;
std::map<std::tuple<int, int64_t, int64_t, int64_t>, int> g_table;   // (catalogue, M, N, K)
bool g_table_env_loaded = false;

bool swiglu_ok(int id);

int cat_count(int cat) {
  return cat == kCatInt8 ? kNumVariants8 : cat == kCatFp4 ? kNumVariantsF4 : kNumVariants;
}

const char* cat_name(int cat, int id) {
  if (id < 0 || id >= cat_count(cat)) return nullptr;
  return cat == kCatInt8 ? kVariants8[id].name : cat == kCatFp4 ? kVariantsF4[id].name
                                                               : kVariants[id].name;
}

int cat_by_name(int cat, const std::string& n) {
  for (int i = 0; i < cat_count(cat); ++i)
    if (n == cat_name(cat, i)) return i;
  return -1;
}

bool cat_eligible(int cat, int id, int64_t M, int64_t N, int64_t K) {
  switch (cat) {
    case kCatInt4: return variant_eligible(id, M, N, K);
    case kCatSwiglu: return swiglu_ok(id) && N % 2 == 0 && variant_eligible(id, M, N, K);
    case kCatInt8: return variant8_eligible(id, M, N, K);
    case kCatFp4: return variantf4_eligible(id, M, N, K);
    default: return false;
  }
}

// Text lines "M N K variant" (INT4) or "tag M N K variant" (tag swiglu, int8
// or fp4).
int load_table_locked(const char* path) {
  std::ifstream f(path);
  if (!f) return W4A16_ERR_INVALID_ARG;
  std::string line;
  while (std::getline(f, line)) {
    if (line.empty() || line[0] == '#') continue;
    std::istringstream ss(line);
    int cat = kCatInt4;
    if (!std::isdigit(static_cast<unsigned char>(line[0]))) {
      std::string tag;
      ss >> tag;
      cat = -1;
      for (int c = 1; c < kNumCats; ++c)
        if (tag == kCatTag[c]) cat = c;
      if (cat < 0) return W4A16_ERR_INVALID_ARG;
    }
    int64_t M, N, K;
    std::string name;
    if (!(ss >> M >> N >> K >> name)) return W4A16_ERR_INVALID_ARG;
    const int id = cat_by_name(cat, name);
    if (id < 0 || !cat_eligible(cat, id, M, N, K)) return W4A16_ERR_NO_VARIANT;
    g_table[{cat, M, N, K}] = id;
  }
  return W4A16_OK;
}

// The table's entry for a shape of a catalogue, or -1.
int table_get(int cat, int64_t M, int64_t N, int64_t K);

void maybe_load_env_table_locked() {
  if (g_table_env_loaded) return;
  g_table_env_loaded = true;
  const char* p = std::getenv("W4A16_VARIANT_TABLE");
  if (p != nullptr && p[0] != '\0') {
    const int st = load_table_locked(p);
    if (st != W4A16_OK) std::fprintf(stderr, "w4a16: could not load variant table %s (%d)\n", p, st);
  }
}

bool log_enabled() {
  static const bool on = [] {
    const char* p = std::getenv("W4A16_LOG");
    return p != nullptr && p[0] == '1';
  }();
  return on;
}

int table_get(int cat, int64_t M, int64_t N, int64_t K) {
  std::lock_guard<std::mutex> lock(g_table_mutex);
  maybe_load_env_table_locked();
  auto it = g_table.find({cat, M, N, K});
  return it != g_table.end() ? it->second : -1;
}

int table_put(int cat, int64_t M, int64_t N, int64_t K, int id) {
  if (!cat_eligible(cat, id, M, N, K)) return W4A16_ERR_NO_VARIANT;
  std::lock_guard<std::mutex> lock(g_table_mutex);
  maybe_load_env_table_locked();
  g_table[{cat, M, N, K}] = id;
  return W4A16_OK;
}

int select_variant(int64_t M, int64_t N, int64_t K) {
  int id = table_get(kCatInt4, M, N, K);
  if (id < 0) {
    DeviceInfo dev;
    const int sms = device_info(dev) ? dev.num_sms : kDefaultSms;
    id = rule_variant(M, N, K, sms);
  }
  if (!variant_eligible(id, M, N, K)) return -1;
  return id;
}

// SwiGLU epilogue: the variant select_variant gives for the shape, unless it
// is a CUDA-core streaming variant (whose epilogue does not pair rows); then
// the rule over the tcgen05 variants.
bool swiglu_ok(int id) {
  return id >= 0 && id < kNumVariants && !kVariants[id].cfg.simt && kVariants[id].csk == 0;
}

int select_variant_swiglu(int64_t M, int64_t N, int64_t K) {
  const int tuned = table_get(kCatSwiglu, M, N, K);
  if (tuned >= 0 && cat_eligible(kCatSwiglu, tuned, M, N, K)) return tuned;
  const int id = select_variant(M, N, K);
  if (id < 0 || swiglu_ok(id)) return id;
  DeviceInfo dev;
  const int sms = device_info(dev) ? dev.num_sms : kDefaultSms;
  int best = -1;
  double best_t = 0.0;
  for (int v = 0; v < kNumVariants; ++v) {
    if (!swiglu_ok(v) || !variant_eligible(v, M, N, K)) continue;
    const double t = estimate_us(kVariants[v], M, N, K, sms);
    if (best < 0 || t < best_t) {
      best = v;
      best_t = t;
    }
  }
  return best;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_gemm_args(const void* A, int64_t M, int64_t N, int64_t K, const void* packed,
                    const void* scales, int group, const void* bias, void* Y) {
  if (A == nullptr || packed == nullptr || scales == nullptr || Y == nullptr)
    return W4A16_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || K < 1) return W4A16_ERR_INVALID_ARG;
  if (group != kGroup) return W4A16_ERR_UNSUPPORTED;
  if (!shape_ok(M, N, K)) return W4A16_ERR_UNSUPPORTED;
  if (!aligned16(A) || !aligned16(packed) || !aligned16(scales) || !aligned16(Y) ||
      (bias != nullptr && !aligned16(bias)))
    return W4A16_ERR_ALIGNMENT;
  return W4A16_OK;
}

int run_gemm_v(const Variant& v, const void* A, int64_t M, int64_t N, int64_t K,
               const void* packed, const void* scales, const void* bias, void* Y, void* ws,
               size_t ws_bytes, cudaStream_t stream, bool act_f16,
               const float* tensor_scale = nullptr, bool swiglu = false) {
  DeviceInfo dev;
  if (!device_info(dev)) return W4A16_ERR_CUDA;
  const GemmSchedule s = make_schedule(v, M, N, K, dev.num_sms);
  const size_t need = gemm_workspace_bytes(v.cfg, s, M, N, K);
  if (need > 0) {
    if (ws == nullptr || ws_bytes < need) return W4A16_ERR_WORKSPACE;
    if (!aligned16(ws)) return W4A16_ERR_ALIGNMENT;
  }
  GemmProblem p{};
  p.A = A;
  p.packed = packed;
  p.scales = scales;
  p.bias = bias;
  p.Y = Y;
  p.M = M;
  p.N = N;
  p.K = K;
  p.workspace = ws;
  p.workspace_bytes = ws_bytes;
  p.error_word = dev.error_word;
  p.timeout_ns = g_timeout_ns.load();
  p.act_f16 = act_f16;
  p.tensor_scale = tensor_scale;
  p.swiglu = swiglu;
  p.weights_static = g_weights_static.load() != 0;
  if (log_enabled())
    std::fprintf(stderr, "w4a16: gemm M=%lld N=%lld K=%lld variant=%s grid=%d dp_tiles=%d sk_units=%lld\n",
                 static_cast<long long>(M), static_cast<long long>(N), static_cast<long long>(K),
                 v.name, s.grid, s.dp_tiles, static_cast<long long>(s.sk_units));
  const cudaError_t e = launch_gemm_tc(v.cfg, s, p, /*use_pdl=*/true, stream);
  if (e != cudaSuccess) return cuda_failure(e, v.name);
  g_launches.fetch_add(1);
  return W4A16_OK;
}

int run_gemm(int id, const void* A, int64_t M, int64_t N, int64_t K, const void* packed,
             const void* scales, const void* bias, void* Y, void* ws, size_t ws_bytes,
             cudaStream_t stream, bool act_f16 = false) {
  return run_gemm_v(kVariants[id], A, M, N, K, packed, scales, bias, Y, ws, ws_bytes, stream,
                    act_f16);
}

// INT8: the rule over the INT8 catalogue (no measured table).
int select_variant8(int64_t M, int64_t N, int64_t K) {
  const int tuned = table_get(kCatInt8, M, N, K);
  if (tuned >= 0 && variant8_eligible(tuned, M, N, K)) return tuned;
  DeviceInfo dev;
  const int sms = device_info(dev) ? dev.num_sms : kDefaultSms;
  int best = -1;
  double best_t = 0.0;
  for (int id = 0; id < kNumVariants8; ++id) {
    if (!variant8_eligible(id, M, N, K)) continue;
    const double t = estimate_us(kVariants8[id], M, N, K, sms);
    if (best < 0 || t < best_t) {
      best = id;
      best_t = t;
    }
  }
  return best;
}

// FP4: the rule over the FP4 catalogue.
int select_variantf4(int64_t M, int64_t N, int64_t K) {
  const int tuned = table_get(kCatFp4, M, N, K);
  if (tuned >= 0 && variantf4_eligible(tuned, M, N, K)) return tuned;
  DeviceInfo dev;
  const int sms = device_info(dev) ? dev.num_sms : kDefaultSms;
  int best = -1;
  double best_t = 0.0;
  for (int id = 0; id < kNumVariantsF4; ++id) {
    if (!variantf4_eligible(id, M, N, K)) continue;
    const double t = estimate_us(kVariantsF4[id], M, N, K, sms);
    if (best < 0 || t < best_t) {
      best = id;
      best_t = t;
    }
  }
  return best;
}

size_t variantf4_ws(int id, int64_t M, int64_t N, int64_t K) {
  DeviceInfo dev;
  int sms = kDefaultSms;
  if (device_info(dev)) sms = dev.num_sms;
  const Variant& v = kVariantsF4[id];
  return gemm_workspace_bytes(v.cfg, make_schedule(v, M, N, K, sms), M, N, K);
}

size_t variant8_ws(int id, int64_t M, int64_t N, int64_t K) {
  DeviceInfo dev;
  int sms = kDefaultSms;
  if (device_info(dev)) sms = dev.num_sms;
  const Variant& v = kVariants8[id];
  return gemm_workspace_bytes(v.cfg, make_schedule(v, M, N, K, sms), M, N, K);
}

// ------------------------------------------------------------ groups
// A group of independent GEMMs runs in one launch, problem i on its own
// sub-grid of CTAs.  Planning picks one variant for the group: CTAs are
// shared out in proportion to each problem's units (at least one each, no
// more than the SMs in total, so every sub-grid is resident at once), each
// problem gets that variant's schedule on its share, and the variant whose
// slowest problem has the smallest estimate wins.  Workspace: the fixed
// counter region (problem i's grid-barrier words at 2 i, 2 i + 1), then each
// split problem's partial slots.
struct GroupPlan {
  int variant = -1;
  GemmSchedule s[kMaxGemmGroup];
  size_t partial_off[kMaxGemmGroup];
  size_t ws_bytes = 0;
  double est_us = 0.0;
};

// The schedule of one problem of a grouped launch on `ctas` CTAs: the
// variant's own, or (when the variant is not forced) for a stream-K variant
// whole tiles only when that is estimated faster (every split tile pays the
// fixup).
GemmSchedule group_schedule(const Variant& v, const w4a16_gemm_problem& p, int ctas, double& est,
                            bool own_only, bool single) {
  GemmSchedule s = make_schedule(v, p.M, p.N, p.K, ctas, single);
  est = estimate_sched(v, s, p.K, p.N, ctas);
  if (!own_only && v.stream_k && s.sk_units > 0) {
    const int64_t tiles = gemm_tiles(v.cfg, p.M, p.N);
    GemmSchedule d{};
    d.grid = static_cast<int>(tiles < ctas ? tiles : ctas);
    d.dp_tiles = static_cast<int>(tiles);
    d.sk_units = 0;
    const double ed = estimate_sched(v, d, p.K, p.N, ctas);
    if (ed < est) {
      s = d;
      est = ed;
    }
  }
  return s;
}

// CTAs of a grouped launch: a single problem gets every SM (exactly the
// single-call schedule when the variant is forced); several start with one
// CTA each and take the rest one at a time, to the problem with the largest
// estimate while that estimate improves.
bool plan_for_variant(int id, const w4a16_gemm_problem* pr, int count, int sms, GroupPlan& plan,
                      bool forced) {
  const Variant& v = kVariants[id];
  // single problems only: the CUDA-core workers and the cluster split-K
  // variants (the row-block kernel groups problems in its persistent form;
  // a share of `ctas` SMs runs up to two of its CTAs each)
  if (((v.cfg.simt && !v.cfg.rb) || v.csk > 1) && count > 1) return false;
  for (int i = 0; i < count; ++i) {
    if (!variant_eligible(id, pr[i].M, pr[i].N, pr[i].K)) return false;
    if (pr[i].epilogue == W4A16_EPILOGUE_SWIGLU && !swiglu_ok(id)) return false;
  }
  if (count > sms) return false;
  int ctas[kMaxGemmGroup];
  double est[kMaxGemmGroup];
  for (int i = 0; i < count; ++i) {
    ctas[i] = count == 1 ? sms : 1;
    (void)group_schedule(v, pr[i], ctas[i], est[i], forced, count == 1);
  }
  // units per CTA fall in steps, so a problem may need several more CTAs
  // before its estimate improves: look ahead to the next improving count
  int used = count;
  while (count > 1 && used < sms) {
    int pick = -1, pick_k = 0;
    double pick_est = 0.0;
    for (int i = 0; i < count; ++i) {
      if (pick >= 0 && est[i] <= est[pick]) continue;
      for (int k = 1; used + k <= sms; ++k) {
        double e1;
        (void)group_schedule(v, pr[i], ctas[i] + k, e1, forced, count == 1);
        if (e1 < est[i]) {
          pick = i;
          pick_k = k;
          pick_est = e1;
          break;
        }
      }
    }
    if (pick < 0) break;
    ctas[pick] += pick_k;
    used += pick_k;
    est[pick] = pick_est;
  }
  plan.variant = id;
  plan.est_us = 0.0;
  size_t off = 0;
  bool split = false;
  for (int i = 0; i < count; ++i) {
    double e;
    plan.s[i] = group_schedule(v, pr[i], ctas[i], e, forced, count == 1);
    plan.est_us = std::max(plan.est_us, e);
    plan.partial_off[i] = off;
    if (plan.s[i].sk_units > 0) {
      split = true;
      off += (gemm_workspace_bytes(v.cfg, plan.s[i], pr[i].M, pr[i].N, pr[i].K) - kCounterBytes +
              255) / 256 * 256;
    }
  }
  plan.ws_bytes = split ? kCounterBytes + off : 0;
  return true;
}

// Plans are memoized per (variant, problem shapes): the selection work runs
// once per set of shapes, not on every call.
struct GroupKey {
  int variant, count, sms;
  int64_t mnk[kMaxGemmGroup][4];   // M, N, K, epilogue
  bool operator<(const GroupKey& o) const {
    if (sms != o.sms) return sms < o.sms;
    if (variant != o.variant) return variant < o.variant;
    if (count != o.count) return count < o.count;
    for (int i = 0; i < count; ++i)
      for (int j = 0; j < 4; ++j)
        if (mnk[i][j] != o.mnk[i][j]) return mnk[i][j] < o.mnk[i][j];
    return false;
  }
};
std::map<GroupKey, GroupPlan> g_group_plans;
std::mutex g_group_mutex;

GroupKey group_key(int variant, const w4a16_gemm_problem* pr, int count, int sms) {
  GroupKey key{};
  key.variant = variant < 0 ? -1 : variant;
  key.count = count;
  key.sms = sms;
  for (int i = 0; i < count; ++i) {
    key.mnk[i][0] = pr[i].M;
    key.mnk[i][1] = pr[i].N;
    key.mnk[i][2] = pr[i].K;
    key.mnk[i][3] = pr[i].epilogue;
  }
  return key;
}

int plan_group(const w4a16_gemm_problem* pr, int count, int variant, GroupPlan& plan) {
  DeviceInfo dev;
  const int sms = std::min(device_info(dev) ? dev.num_sms : kDefaultSms, kMaxGrid);
  if (variant >= kNumVariants) return W4A16_ERR_UNSUPPORTED;
  const GroupKey key = group_key(variant, pr, count, sms);
  {
    std::lock_guard<std::mutex> lock(g_group_mutex);
    auto it = g_group_plans.find(key);
    if (it != g_group_plans.end()) {
      plan = it->second;
      return W4A16_OK;
    }
  }
  bool found = false;
  if (variant >= 0) {
    found = plan_for_variant(variant, pr, count, sms, plan, true);
  } else {
    for (int id = 0; id < kNumVariants; ++id) {
      GroupPlan cand;
      if (!plan_for_variant(id, pr, count, sms, cand, false)) continue;
      if (!found || cand.est_us < plan.est_us) {
        plan = cand;
        found = true;
      }
    }
  }
  if (!found) return W4A16_ERR_NO_VARIANT;
  std::lock_guard<std::mutex> lock(g_group_mutex);
  g_group_plans[key] = plan;
  return W4A16_OK;
}

int check_group_args(const w4a16_gemm_problem* pr, int count, int group) {
  if (pr == nullptr || count < 1) return W4A16_ERR_INVALID_ARG;
  if (count > kMaxGemmGroup) return W4A16_ERR_UNSUPPORTED;
  for (int i = 0; i < count; ++i) {
    const int st = check_gemm_args(pr[i].A, pr[i].M, pr[i].N, pr[i].K, pr[i].packed, pr[i].scales,
                                   group, pr[i].bias_or_null, pr[i].Y);
    if (st != W4A16_OK) return st;
    if (pr[i].epilogue != W4A16_EPILOGUE_NONE && pr[i].epilogue != W4A16_EPILOGUE_SWIGLU)
      return W4A16_ERR_UNSUPPORTED;
    if (pr[i].epilogue == W4A16_EPILOGUE_SWIGLU && pr[i].N % 2 != 0) return W4A16_ERR_UNSUPPORTED;
  }
  return W4A16_OK;
}

bool group_has_swiglu(const w4a16_gemm_problem* pr, int count) {
  for (int i = 0; i < count; ++i)
    if (pr[i].epilogue == W4A16_EPILOGUE_SWIGLU) return true;
  return false;
}

size_t variant_ws(int id, int64_t M, int64_t N, int64_t K) {
  DeviceInfo dev;
  int sms = kDefaultSms;
  if (device_info(dev)) sms = dev.num_sms;
  const Variant& v = kVariants[id];
  return gemm_workspace_bytes(v.cfg, make_schedule(v, M, N, K, sms), M, N, K);
}

}  // namespace

// ------------------------------------------------------------------ TMA
namespace {
PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}
}  // namespace

CUresult encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                        uint64_t inner, uint64_t outer, uint64_t outer_stride_bytes,
                        uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle) {
  const auto fn = tmap_encoder();
  if (fn == nullptr) return CUDA_ERROR_NOT_FOUND;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {outer_stride_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

CUresult encode_tmap_3d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                        uint64_t d0, uint64_t d1, uint64_t d2, uint64_t stride1_bytes,
                        uint64_t stride2_bytes, uint32_t box0, uint32_t box1, uint32_t box2,
                        CUtensorMapSwizzle swizzle) {
  const auto fn = tmap_encoder();
  if (fn == nullptr) return CUDA_ERROR_NOT_FOUND;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
  const cuuint32_t box[3] = {box0, box1, box2};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, dtype, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace w4a16

namespace w4a16 {
namespace {

// Scratch for w4a16_gemm_noalloc: a file-scope device array, so that callers
// that must not allocate device memory can still run the stream-K GEMM.  Every
// GPU that loads this library holds it until the process exits.
constexpr size_t kNoAllocScratchBytes = 16u << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// with cudaGetSymbolAddress, once per device, with that device current.
int noalloc_scratch(void** out) {
  int dev = 0;
  const cudaError_t e0 = cudaGetDevice(&dev);
  if (e0 != cudaSuccess) return cuda_failure(e0, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return W4A16_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_failure(e, "cudaGetSymbolAddress(noalloc scratch)");
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return W4A16_OK;
}

}  // namespace
}  // namespace w4a16

using namespace w4a16;

extern "C" {

const char* w4a16_status_string(int status) {
  switch (status) {
    case W4A16_OK: return "W4A16_OK";
    case W4A16_ERR_INVALID_ARG: return "W4A16_ERR_INVALID_ARG: null pointer or size out of range";
    case W4A16_ERR_UNSUPPORTED: return "W4A16_ERR_UNSUPPORTED: group must be 128, K % 128 == 0, N % 8 == 0";
    case W4A16_ERR_ALIGNMENT: return "W4A16_ERR_ALIGNMENT: pointers must be 16-byte aligned";
    case W4A16_ERR_WORKSPACE: return "W4A16_ERR_WORKSPACE: workspace missing or too small";
    case W4A16_ERR_NO_VARIANT: return "W4A16_ERR_NO_VARIANT: no GEMM variant is usable for this shape";
    case W4A16_ERR_CUDA: return "W4A16_ERR_CUDA: a CUDA call failed";
    case W4A16_ERR_TIMEOUT: return "W4A16_ERR_TIMEOUT: a device-side bounded wait expired";
    default: return "W4A16: unknown status";
  }
}

size_t w4a16_packed_bytes(int64_t N, int64_t K) {
  if (N < 0 || K < 0) return 0;
  const int64_t n_pad = (N + kTileW - 1) / kTileW * kTileW;
  return static_cast<size_t>(n_pad) * static_cast<size_t>(K) / 2;
}

size_t w4a16_scales_bytes(int64_t N, int64_t K, int group) {
  if (group != kGroup || N < 0 || K < 0) return 0;
  return static_cast<size_t>(K / group) * static_cast<size_t>(N) * 2;
}

namespace {
int quantize_impl(const void* W_bf16, int64_t N, int64_t K, int group, const uint64_t* sr_seed,
                  void* packed_out, void* scales_out, void* stream, bool int8 = false) {
  if (W_bf16 == nullptr || packed_out == nullptr || scales_out == nullptr)
    return W4A16_ERR_INVALID_ARG;
  if (N < 1 || K < 1) return W4A16_ERR_INVALID_ARG;
  if (group != kGroup) return W4A16_ERR_UNSUPPORTED;
  if (K % kGroup != 0 || N % 8 != 0) return W4A16_ERR_UNSUPPORTED;
  if (N >= (1ll << 31) || K >= (1ll << 31) || N * K >= (1ll << 40)) return W4A16_ERR_UNSUPPORTED;
  if (!aligned16(W_bf16) || !aligned16(packed_out) || !aligned16(scales_out))
    return W4A16_ERR_ALIGNMENT;
  DeviceInfo dev;
  if (!device_info(dev)) return W4A16_ERR_CUDA;
  const cudaError_t e =
      launch_rtn_quantize(W_bf16, N, K, packed_out, scales_out, dev.num_sms, dev.error_word,
                          g_timeout_ns.load(), static_cast<cudaStream_t>(stream), sr_seed, int8);
  if (e != cudaSuccess)
    return cuda_failure(e, int8 ? "rtn_quantize (int8)"
                                : sr_seed ? "rtn_quantize (stochastic)" : "rtn_quantize");
  g_launches.fetch_add(1);
  return W4A16_OK;
}
}  // namespace

int w4a16_quantize(const void* W_bf16, int64_t N, int64_t K, int group, void* packed_out,
                   void* scales_out, void* stream) {
  return quantize_impl(W_bf16, N, K, group, nullptr, packed_out, scales_out, stream);
}

int w4a16_quantize_sr(const void* W_bf16, int64_t N, int64_t K, int group, uint64_t seed,
                      void* packed_out, void* scales_out, void* stream) {
  return quantize_impl(W_bf16, N, K, group, &seed, packed_out, scales_out, stream);
}

// ------------------------------------------------------- INT8 (W8A16)
size_t w8a16_packed_bytes(int64_t N, int64_t K) {
  if (N < 1 || K < 1) return 0;
  return static_cast<size_t>((N + kTileW - 1) / kTileW) * kTileW * static_cast<size_t>(K);
}

int w8a16_quantize(const void* W_bf16, int64_t N, int64_t K, int group, void* packed_out,
                   void* scales_out, void* stream) {
  return quantize_impl(W_bf16, N, K, group, nullptr, packed_out, scales_out, stream, true);
}

size_t w8a16_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  const int id = select_variant8(M, N, K);
  return id < 0 ? 0 : variant8_ws(id, M, N, K);
}

int w8a16_gemm(const void* A_bf16, int64_t M, int64_t N, int64_t K, const void* packed,
               const void* scales, int group, const void* bias_bf16_or_null, void* Y_bf16,
               void* workspace, size_t workspace_bytes, void* stream) {
  const int st = check_gemm_args(A_bf16, M, N, K, packed, scales, group, bias_bf16_or_null, Y_bf16);
  if (st != W4A16_OK) return st;
  const int id = select_variant8(M, N, K);
  if (id < 0) return W4A16_ERR_NO_VARIANT;
  return run_gemm_v(kVariants8[id], A_bf16, M, N, K, packed, scales, bias_bf16_or_null, Y_bf16,
                    workspace, workspace_bytes, static_cast<cudaStream_t>(stream), false);
}

int w8a16_variant_count(void) { return kNumVariants8; }

const char* w8a16_variant_name(int variant) {
  if (variant < 0 || variant >= kNumVariants8) return nullptr;
  return kVariants8[variant].name;
}

int w8a16_variant_eligible(int variant, int64_t M, int64_t N, int64_t K) {
  return variant8_eligible(variant, M, N, K) ? 1 : 0;
}

size_t w8a16_variant_workspace_bytes(int variant, int64_t M, int64_t N, int64_t K) {
  if (!variant8_eligible(variant, M, N, K)) return 0;
  return variant8_ws(variant, M, N, K);
}

int w8a16_select_variant(int64_t M, int64_t N, int64_t K) { return select_variant8(M, N, K); }

int w8a16_gemm_variant(int variant, const void* A_bf16, int64_t M, int64_t N, int64_t K,
                       const void* packed, const void* scales, int group,
                       const void* bias_bf16_or_null, void* Y_bf16, void* workspace,
                       size_t workspace_bytes, void* stream) {
  const int st = check_gemm_args(A_bf16, M, N, K, packed, scales, group, bias_bf16_or_null, Y_bf16);
  if (st != W4A16_OK) return st;
  if (variant < 0 || variant >= kNumVariants8) return W4A16_ERR_UNSUPPORTED;
  if (!variant8_eligible(variant, M, N, K)) return W4A16_ERR_NO_VARIANT;
  return run_gemm_v(kVariants8[variant], A_bf16, M, N, K, packed, scales, bias_bf16_or_null,
                    Y_bf16, workspace, workspace_bytes, static_cast<cudaStream_t>(stream), false);
}

// ------------------------------------------- FP4 weights (MXFP4, NVFP4)
size_t fp4a16_packed_bytes(int64_t N, int64_t K) { return w4a16_packed_bytes(N, K); }

size_t fp4a16_scales_bytes(int format, int64_t N, int64_t K) {
  const int f = fp4_format(format);
  if (f == 0 || N < 0 || K < 0 || K % kGroup != 0) return 0;
  return static_cast<size_t>(K / (f == kFmtMxfp4 ? 32 : 16)) * static_cast<size_t>(N);
}

int fp4a16_quantize(int format, const void* W_bf16, int64_t N, int64_t K, void* packed_out,
                    void* scales_out, float* tensor_scale_out, void* stream) {
  const int f = fp4_format(format);
  if (f == 0) return W4A16_ERR_UNSUPPORTED;
  if (W_bf16 == nullptr || packed_out == nullptr || scales_out == nullptr ||
      (f == kFmtNvfp4 && tensor_scale_out == nullptr))
    return W4A16_ERR_INVALID_ARG;
  if (N < 1 || K < 1) return W4A16_ERR_INVALID_ARG;
  if (K % kGroup != 0 || N % 16 != 0) return W4A16_ERR_UNSUPPORTED;
  if (N >= (1ll << 31) || K >= (1ll << 31) || N * K >= (1ll << 40)) return W4A16_ERR_UNSUPPORTED;
  if (!aligned16(W_bf16) || !aligned16(packed_out) || !aligned16(scales_out) ||
      (tensor_scale_out != nullptr && (reinterpret_cast<uintptr_t>(tensor_scale_out) & 7u) != 0))
    return W4A16_ERR_ALIGNMENT;
  DeviceInfo dev;
  if (!device_info(dev)) return W4A16_ERR_CUDA;
  const cudaError_t e =
      launch_fp4_quantize(W_bf16, N, K, packed_out, scales_out, tensor_scale_out, f, dev.num_sms,
                          dev.error_word, g_timeout_ns.load(), static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_failure(e, f == kFmtMxfp4 ? "quantize (mxfp4)" : "quantize (nvfp4)");
  g_launches.fetch_add(f == kFmtMxfp4 ? 1 : 2);
  return W4A16_OK;
}

namespace {
int check_fp4_gemm_args(int f, const void* A, int64_t M, int64_t N, int64_t K, const void* packed,
                        const void* scales, const float* tensor_scale, const void* bias,
                        void* Y) {
  if (f == 0) return W4A16_ERR_UNSUPPORTED;
  if (f == kFmtNvfp4 && tensor_scale == nullptr) return W4A16_ERR_INVALID_ARG;
  const int st = check_gemm_args(A, M, N, K, packed, scales, kGroup, bias, Y);
  if (st != W4A16_OK) return st;
  if (N % 16 != 0) return W4A16_ERR_UNSUPPORTED;
  if (tensor_scale != nullptr && (reinterpret_cast<uintptr_t>(tensor_scale) & 3u) != 0)
    return W4A16_ERR_ALIGNMENT;
  return W4A16_OK;
}
}  // namespace

size_t fp4a16_gemm_workspace_bytes(int format, int64_t M, int64_t N, int64_t K) {
  if (fp4_format(format) == 0) return 0;
  const int id = select_variantf4(M, N, K);
  return id < 0 ? 0 : variantf4_ws(id, M, N, K);
}

int fp4a16_gemm(int format, const void* A_bf16, int64_t M, int64_t N, int64_t K,
                const void* packed, const void* scales, const float* tensor_scale,
                const void* bias_bf16_or_null, void* Y_bf16, void* workspace,
                size_t workspace_bytes, void* stream) {
  const int f = fp4_format(format);
  const int st = check_fp4_gemm_args(f, A_bf16, M, N, K, packed, scales, tensor_scale,
                                     bias_bf16_or_null, Y_bf16);
  if (st != W4A16_OK) return st;
  const int id = select_variantf4(M, N, K);
  if (id < 0) return W4A16_ERR_NO_VARIANT;
  return run_gemm_v(variant_f4(id, f), A_bf16, M, N, K, packed, scales, bias_bf16_or_null,
                    Y_bf16, workspace, workspace_bytes, static_cast<cudaStream_t>(stream), false,
                    f == kFmtNvfp4 ? tensor_scale : nullptr);
}

int fp4a16_variant_count(void) { return kNumVariantsF4; }

const char* fp4a16_variant_name(int variant) {
  if (variant < 0 || variant >= kNumVariantsF4) return nullptr;
  return kVariantsF4[variant].name;
}

int fp4a16_variant_eligible(int variant, int64_t M, int64_t N, int64_t K) {
  return variantf4_eligible(variant, M, N, K) ? 1 : 0;
}

size_t fp4a16_variant_workspace_bytes(int variant, int64_t M, int64_t N, int64_t K) {
  if (!variantf4_eligible(variant, M, N, K)) return 0;
  return variantf4_ws(variant, M, N, K);
}

int fp4a16_select_variant(int64_t M, int64_t N, int64_t K) { return select_variantf4(M, N, K); }

int fp4a16_gemm_variant(int variant, int format, const void* A_bf16, int64_t M, int64_t N,
                        int64_t K, const void* packed, const void* scales,
                        const float* tensor_scale, const void* bias_bf16_or_null, void* Y_bf16,
                        void* workspace, size_t workspace_bytes, void* stream) {
  const int f = fp4_format(format);
  const int st = check_fp4_gemm_args(f, A_bf16, M, N, K, packed, scales, tensor_scale,
                                     bias_bf16_or_null, Y_bf16);
  if (st != W4A16_OK) return st;
  if (variant < 0 || variant >= kNumVariantsF4) return W4A16_ERR_UNSUPPORTED;
  if (!variantf4_eligible(variant, M, N, K)) return W4A16_ERR_NO_VARIANT;
  return run_gemm_v(variant_f4(variant, f), A_bf16, M, N, K, packed, scales, bias_bf16_or_null,
                    Y_bf16, workspace, workspace_bytes, static_cast<cudaStream_t>(stream), false,
                    f == kFmtNvfp4 ? tensor_scale : nullptr);
}

size_t w4a16_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  const int id = select_variant(M, N, K);
  if (id < 0) return 0;
  return variant_ws(id, M, N, K);
}

size_t w4a16_gemm_workspace_bytes_max(int64_t M, int64_t N, int64_t K) {
  size_t m = 0;
  for (int id = 0; id < kNumVariants; ++id) {
    if (!variant_eligible(id, M, N, K)) continue;
    const size_t b = variant_ws(id, M, N, K);
    if (b > m) m = b;
  }
  return m;
}

int w4a16_workspace_init(void* workspace, size_t bytes, void* stream) {
  if (bytes == 0) return W4A16_OK;
  if (workspace == nullptr) return W4A16_ERR_INVALID_ARG;
  if (cudaMemsetAsync(workspace, 0, bytes, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return W4A16_ERR_CUDA;
  return W4A16_OK;
}

int w4a16_gemm(const void* A_bf16, int64_t M, int64_t N, int64_t K, const void* packed,
               const void* scales, int group, const void* bias_bf16_or_null, void* Y_bf16,
               void* workspace, size_t workspace_bytes, void* stream) {
  const int st = check_gemm_args(A_bf16, M, N, K, packed, scales, group, bias_bf16_or_null, Y_bf16);
  if (st != W4A16_OK) return st;
  const int id = select_variant(M, N, K);
  if (id < 0) return W4A16_ERR_NO_VARIANT;
  return run_gemm(id, A_bf16, M, N, K, packed, scales, bias_bf16_or_null, Y_bf16, workspace,
                  workspace_bytes, static_cast<cudaStream_t>(stream));
}

size_t w4a16_gemm_swiglu_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  const int id = select_variant_swiglu(M, N, K);
  if (id < 0) return 0;
  return variant_ws(id, M, N, K);
}

int w4a16_gemm_swiglu_variant(int variant, const void* A_bf16, int64_t M, int64_t N, int64_t K,
                              const void* packed, const void* scales, int group,
                              const void* bias_bf16_or_null, void* Y_bf16, void* workspace,
                              size_t workspace_bytes, void* stream) {
  const int st = check_gemm_args(A_bf16, M, N, K, packed, scales, group, bias_bf16_or_null, Y_bf16);
  if (st != W4A16_OK) return st;
  if (!swiglu_ok(variant)) return W4A16_ERR_UNSUPPORTED;
  if (!variant_eligible(variant, M, N, K)) return W4A16_ERR_NO_VARIANT;
  return run_gemm_v(kVariants[variant], A_bf16, M, N, K, packed, scales, bias_bf16_or_null, Y_bf16,
                    workspace, workspace_bytes, static_cast<cudaStream_t>(stream),
                    /*act_f16=*/false, /*tensor_scale=*/nullptr, /*swiglu=*/true);
}

int w4a16_gemm_swiglu(const void* A_bf16, int64_t M, int64_t N, int64_t K, const void* packed,
                      const void* scales, int group, const void* bias_bf16_or_null, void* Y_bf16,
                      void* workspace, size_t workspace_bytes, void* stream) {
  const int st = check_gemm_args(A_bf16, M, N, K, packed, scales, group, bias_bf16_or_null, Y_bf16);
  if (st != W4A16_OK) return st;
  const int id = select_variant_swiglu(M, N, K);
  if (id < 0) return W4A16_ERR_NO_VARIANT;
  return w4a16_gemm_swiglu_variant(id, A_bf16, M, N, K, packed, scales, group, bias_bf16_or_null,
                                   Y_bf16, workspace, workspace_bytes, stream);
}

int w4a16_variant_count(void) { return kNumVariants; }

const char* w4a16_variant_name(int variant) {
  if (variant < 0 || variant >= kNumVariants) return nullptr;
  return kVariants[variant].name;
}

int w4a16_variant_eligible(int variant, int64_t M, int64_t N, int64_t K) {
  return variant_eligible(variant, M, N, K) ? 1 : 0;
}

size_t w4a16_variant_workspace_bytes(int variant, int64_t M, int64_t N, int64_t K) {
  if (!variant_eligible(variant, M, N, K)) return 0;
  return variant_ws(variant, M, N, K);
}

int w4a16_select_variant(int64_t M, int64_t N, int64_t K) { return select_variant(M, N, K); }

int w4a16_variant_schedule(int variant, int64_t M, int64_t N, int64_t K, int num_sms, int* out) {
  if (out == nullptr || num_sms < 0) return W4A16_ERR_INVALID_ARG;
  if (!variant_eligible(variant, M, N, K)) return W4A16_ERR_NO_VARIANT;
  const int sms = std::min(num_sms > 0 ? num_sms : current_sms(), kMaxGrid);
  const Variant& v = kVariants[variant];
  const GemmSchedule s = make_schedule(v, M, N, K, sms);
  out[0] = s.grid;
  out[1] = s.dp_tiles;
  out[2] = static_cast<int>(std::min<int64_t>(s.sk_units, 0x7FFFFFFF));
  out[3] = s.cluster;
  out[4] = v.cfg.rb ? s.team : 0;
  return W4A16_OK;
}

}  // extern "C"

namespace {
// One launch of a planned group (the caller checked the arguments and the
// workspace size).
int launch_group_plan(const GroupPlan& plan, const w4a16_gemm_problem* problems, int count,
                      int act_f16, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  DeviceInfo dev;
  if (!device_info(dev)) return W4A16_ERR_CUDA;
  const Variant& v = kVariants[plan.variant];
  GemmGroup grp;
  grp.count = count;
  for (int i = 0; i < count; ++i) {
    GemmProblem& p = grp.p[i];
    p.A = problems[i].A;
    p.packed = problems[i].packed;
    p.scales = problems[i].scales;
    p.bias = problems[i].bias_or_null;
    p.Y = problems[i].Y;
    p.M = problems[i].M;
    p.N = problems[i].N;
    p.K = problems[i].K;
    p.workspace = workspace;
    p.workspace_bytes = workspace_bytes;
    uint8_t* base = static_cast<uint8_t*>(workspace);
    p.counters = base ? reinterpret_cast<uint32_t*>(base) + kCountersPerProblem * i : nullptr;
    p.partials = base ? reinterpret_cast<float*>(base + kCounterBytes + plan.partial_off[i]) : nullptr;
    p.error_word = dev.error_word;
    p.timeout_ns = g_timeout_ns.load();
    p.act_f16 = act_f16 != 0;
    p.swiglu = problems[i].epilogue == W4A16_EPILOGUE_SWIGLU;
    p.weights_static = g_weights_static.load() != 0;
    grp.s[i] = plan.s[i];
  }
  if (log_enabled())
    std::fprintf(stderr, "w4a16: grouped gemm of %d, variant=%s, estimate %.1f us\n", count, v.name,
                 plan.est_us);
  const cudaError_t e = launch_gemm_tc_group(v.cfg, grp, /*use_pdl=*/true, stream);
  if (e != cudaSuccess) return cuda_failure(e, v.name);
  g_launches.fetch_add(1);
  return W4A16_OK;
}

}  // namespace

extern "C" {

size_t w4a16_gemm_grouped_workspace_bytes(const w4a16_gemm_problem* problems, int count,
                                          int variant) {
  if (check_group_args(problems, count, kGroup) != W4A16_OK) return 0;
  GroupPlan plan;
  if (plan_group(problems, count, variant, plan) != W4A16_OK) return 0;
  return plan.ws_bytes;
}

int w4a16_gemm_grouped(const w4a16_gemm_problem* problems, int count, int group, int act_f16,
                       int variant, void* workspace, size_t workspace_bytes, void* stream) {
  int st = check_group_args(problems, count, group);
  if (st != W4A16_OK) return st;
  if (act_f16 && group_has_swiglu(problems, count)) return W4A16_ERR_UNSUPPORTED;
  GroupPlan plan;
  st = plan_group(problems, count, variant, plan);
  if (st != W4A16_OK) return st;
  if (plan.ws_bytes > 0) {
    if (workspace == nullptr || workspace_bytes < plan.ws_bytes) return W4A16_ERR_WORKSPACE;
    if (!aligned16(workspace)) return W4A16_ERR_ALIGNMENT;
  }
  return launch_group_plan(plan, problems, count, act_f16, workspace, workspace_bytes,
                           static_cast<cudaStream_t>(stream));
}

int w4a16_tune_grouped(const w4a16_gemm_problem* problems, int count, int act_f16, void* stream_v,
                       int* out_variant) {
  int st = check_group_args(problems, count, kGroup);
  if (st != W4A16_OK) return st;
  if (act_f16 && group_has_swiglu(problems, count)) return W4A16_ERR_UNSUPPORTED;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone)
    return W4A16_ERR_INVALID_ARG;
  DeviceInfo dev;
  if (!device_info(dev)) return W4A16_ERR_CUDA;
  const int sms = std::min(dev.num_sms, kMaxGrid);

  // Synthetic operands of the problems' shapes; enough weight copies that
  // the timed launches stream them from HBM rather than L2.
  std::vector<void*> bufs;
  auto alloc = [&](size_t b) -> void* {
    void* p = nullptr;
    if (cudaMalloc(&p, b < 256 ? 256 : b) != cudaSuccess) return nullptr;
    bufs.push_back(p);
    return p;
  };
  auto release = [&]() {
    for (void* p : bufs) cudaFree(p);
    bufs.clear();
  };
  size_t per_copy = 0;
  for (int i = 0; i < count; ++i)
    per_copy += w4a16_packed_bytes(problems[i].N, problems[i].K) +
                w4a16_scales_bytes(problems[i].N, problems[i].K, kGroup);
  int copies = static_cast<int>((512ull << 20) / (per_copy + 1)) + 1;
  if (copies > 16) copies = 16;
  std::vector<std::vector<w4a16_gemm_problem>> sets(copies);
  bool ok = true;
  for (int c = 0; ok && c < copies; ++c) {
    sets[c].assign(problems, problems + count);
    for (int i = 0; ok && i < count; ++i) {
      w4a16_gemm_problem& q = sets[c][i];
      const size_t wb = w4a16_packed_bytes(q.N, q.K), sb = w4a16_scales_bytes(q.N, q.K, kGroup);
      void* w = alloc(wb);
      void* sc = alloc(sb);
      void* a = c == 0 ? alloc(static_cast<size_t>(q.M) * q.K * 2) : const_cast<void*>(sets[0][i].A);
      void* y = c == 0 ? alloc(static_cast<size_t>(q.M) * q.N * 2) : sets[0][i].Y;
      ok = w && sc && a && y;
      if (!ok) break;
      cudaMemsetAsync(w, 0x5A, wb, stream);
      cudaMemsetAsync(sc, 0x1C, sb, stream);
      if (c == 0) cudaMemsetAsync(a, 0x3C, static_cast<size_t>(q.M) * q.K * 2, stream);
      q.packed = w;
      q.scales = sc;
      q.A = a;
      q.Y = y;
      q.bias_or_null = nullptr;
    }
  }
  // every candidate plan: each variant with its per-problem schedules
  std::vector<GroupPlan> cands;
  size_t ws_max = 0;
  for (int id = 0; ok && id < kNumVariants; ++id) {
    GroupPlan cand;
    if (!plan_for_variant(id, problems, count, sms, cand, false)) continue;
    cands.push_back(cand);
    ws_max = std::max(ws_max, cand.ws_bytes);
  }
  void* ws = ok && ws_max ? alloc(ws_max) : nullptr;
  if (ok && ws_max) {
    ok = ws != nullptr;
    if (ok) cudaMemsetAsync(ws, 0, ws_max, stream);
  }
  if (!ok || cands.empty()) {
    release();
    return ok ? W4A16_ERR_NO_VARIANT : W4A16_ERR_CUDA;
  }

  cudaEvent_t e0, e1;
  cudaEventCreate(&e0);
  cudaEventCreate(&e1);
  cudaStream_t cs = nullptr;
  if (cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) != cudaSuccess) ok = false;
  if (ok && cudaStreamSynchronize(stream) != cudaSuccess) ok = false;
  constexpr int kIters = 20;
  int best = -1;
  float best_ms = 0.0f;
  for (size_t k = 0; ok && k < cands.size(); ++k) {
    const GroupPlan& pl = cands[k];
    bool fine = true;
    for (int it = 0; it < 2 && fine; ++it)
      fine = launch_group_plan(pl, sets[it % copies].data(), count, act_f16, ws, ws_max, cs) ==
             W4A16_OK;
    if (!fine) continue;
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
      ok = false;
      break;
    }
    for (int it = 0; it < kIters; ++it)
      launch_group_plan(pl, sets[it % copies].data(), count, act_f16, ws, ws_max, cs);
    if (cudaStreamEndCapture(cs, &graph) != cudaSuccess ||
        cudaGraphInstantiate(&exec, graph, 0) != cudaSuccess) {
      if (graph) cudaGraphDestroy(graph);
      ok = false;
      break;
    }
    cudaGraphLaunch(exec, cs);   // warm
    cudaEventRecord(e0, cs);
    cudaGraphLaunch(exec, cs);
    cudaEventRecord(e1, cs);
    const bool synced = cudaEventSynchronize(e1) == cudaSuccess;
    cudaGraphExecDestroy(exec);
    cudaGraphDestroy(graph);
    if (!synced) {
      ok = false;
      break;
    }
    float ms = 0.0f;
    cudaEventElapsedTime(&ms, e0, e1);
    if (log_enabled())
      std::fprintf(stderr, "w4a16: tune group of %d %s %.3f us (estimate %.1f)\n", count,
                   kVariants[pl.variant].name, 1000.0 * ms / kIters, pl.est_us);
    if (best < 0 || ms < best_ms) {
      best_ms = ms;
      best = static_cast<int>(k);
    }
  }
  if (cs) {
    cudaStreamSynchronize(cs);
    cudaStreamDestroy(cs);
  }
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  cudaGetLastError();
  const int dev_err = w4a16_get_device_error(stream);
  release();
  if (!ok) return cuda_failure(cudaErrorUnknown, "w4a16_tune_grouped: graph timing failed");
  if (dev_err != W4A16_OK) return dev_err;
  if (best < 0) return W4A16_ERR_NO_VARIANT;
  // memoize: later automatic grouped launches of these shapes use it
  const GroupKey key = group_key(-1, problems, count, sms);
  {
    std::lock_guard<std::mutex> lock(g_group_mutex);
    g_group_plans[key] = cands[best];
  }
  if (out_variant) *out_variant = cands[best].variant;
  return W4A16_OK;
}

int w4a16_set_grouped_variant(const w4a16_gemm_problem* problems, int count, int variant) {
  int st = check_group_args(problems, count, kGroup);
  if (st != W4A16_OK) return st;
  if (variant < 0 || variant >= kNumVariants) return W4A16_ERR_UNSUPPORTED;
  DeviceInfo dev;
  const int sms = std::min(device_info(dev) ? dev.num_sms : kDefaultSms, kMaxGrid);
  GroupPlan plan;
  if (!plan_for_variant(variant, problems, count, sms, plan, false)) return W4A16_ERR_NO_VARIANT;
  const GroupKey key = group_key(-1, problems, count, sms);
  std::lock_guard<std::mutex> lock(g_group_mutex);
  g_group_plans[key] = plan;
  return W4A16_OK;
}

int w4a16_quantize_grouped(const w4a16_quantize_problem* problems, int count, int group,
                           void* stream) {
  if (problems == nullptr || count < 1) return W4A16_ERR_INVALID_ARG;
  if (count > kMaxQuantizeGroup) return W4A16_ERR_UNSUPPORTED;
  if (group != kGroup) return W4A16_ERR_UNSUPPORTED;
  QuantizeProblem qp[kMaxQuantizeGroup];
  for (int i = 0; i < count; ++i) {
    const w4a16_quantize_problem& p = problems[i];
    if (p.W_bf16 == nullptr || p.packed_out == nullptr || p.scales_out == nullptr)
      return W4A16_ERR_INVALID_ARG;
    if (p.N < 1 || p.K < 1) return W4A16_ERR_INVALID_ARG;
    if (p.K % kGroup != 0 || p.N % 8 != 0) return W4A16_ERR_UNSUPPORTED;
    if (p.N >= (1ll << 31) || p.K >= (1ll << 31) || p.N * p.K >= (1ll << 40))
      return W4A16_ERR_UNSUPPORTED;
    if (!aligned16(p.W_bf16) || !aligned16(p.packed_out) || !aligned16(p.scales_out))
      return W4A16_ERR_ALIGNMENT;
    qp[i] = QuantizeProblem{p.W_bf16, p.N, p.K, p.packed_out, p.scales_out};
  }
  DeviceInfo dev;
  if (!device_info(dev)) return W4A16_ERR_CUDA;
  const cudaError_t e = launch_rtn_quantize_group(qp, count, dev.num_sms, dev.error_word,
                                                  g_timeout_ns.load(), static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_failure(e, "rtn_quantize (grouped)");
  g_launches.fetch_add(1);
  return W4A16_OK;
}

int w4a16_gemm_f16(const void* A_f16, int64_t M, int64_t N, int64_t K, const void* packed,
                   const void* scales, int group, const void* bias_f16_or_null, void* Y_f16,
                   void* workspace, size_t workspace_bytes, void* stream) {
  const int st = check_gemm_args(A_f16, M, N, K, packed, scales, group, bias_f16_or_null, Y_f16);
  if (st != W4A16_OK) return st;
  const int id = select_variant(M, N, K);
  if (id < 0) return W4A16_ERR_NO_VARIANT;
  return run_gemm(id, A_f16, M, N, K, packed, scales, bias_f16_or_null, Y_f16, workspace,
                  workspace_bytes, static_cast<cudaStream_t>(stream), /*act_f16=*/true);
}

int w4a16_gemm_variant_f16(int variant, const void* A_f16, int64_t M, int64_t N, int64_t K,
                           const void* packed, const void* scales, int group,
                           const void* bias_f16_or_null, void* Y_f16, void* workspace,
                           size_t workspace_bytes, void* stream) {
  const int st = check_gemm_args(A_f16, M, N, K, packed, scales, group, bias_f16_or_null, Y_f16);
  if (st != W4A16_OK) return st;
  if (variant < 0 || variant >= kNumVariants) return W4A16_ERR_UNSUPPORTED;
  if (!variant_eligible(variant, M, N, K)) return W4A16_ERR_NO_VARIANT;
  return run_gemm(variant, A_f16, M, N, K, packed, scales, bias_f16_or_null, Y_f16, workspace,
                  workspace_bytes, static_cast<cudaStream_t>(stream), /*act_f16=*/true);
}

int w4a16_gemm_variant(int variant, const void* A_bf16, int64_t M, int64_t N, int64_t K,
                       const void* packed, const void* scales, int group,
                       const void* bias_bf16_or_null, void* Y_bf16, void* workspace,
                       size_t workspace_bytes, void* stream) {
  const int st = check_gemm_args(A_bf16, M, N, K, packed, scales, group, bias_bf16_or_null, Y_bf16);
  if (st != W4A16_OK) return st;
  if (variant < 0 || variant >= kNumVariants) return W4A16_ERR_UNSUPPORTED;
  if (!variant_eligible(variant, M, N, K)) return W4A16_ERR_NO_VARIANT;
  return run_gemm(variant, A_bf16, M, N, K, packed, scales, bias_bf16_or_null, Y_bf16, workspace,
                  workspace_bytes, static_cast<cudaStream_t>(stream));
}

int w4a16_table_set(int64_t M, int64_t N, int64_t K, int variant) {
  return table_put(kCatInt4, M, N, K, variant);
}

int w4a16_swiglu_table_set(int64_t M, int64_t N, int64_t K, int variant) {
  return table_put(kCatSwiglu, M, N, K, variant);
}

int w8a16_table_set(int64_t M, int64_t N, int64_t K, int variant) {
  return table_put(kCatInt8, M, N, K, variant);
}

int fp4a16_table_set(int64_t M, int64_t N, int64_t K, int variant) {
  return table_put(kCatFp4, M, N, K, variant);
}

void w4a16_table_clear(void) {
  std::lock_guard<std::mutex> lock(g_table_mutex);
  g_table_env_loaded = true;
  g_table.clear();
}

int w4a16_table_save(const char* path) {
  if (path == nullptr) return W4A16_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_table_mutex);
  std::ofstream f(path);
  if (!f) return W4A16_ERR_INVALID_ARG;
  f << "# [catalogue] M N K variant  (no catalogue: INT4 GEMM; swiglu, int8, fp4)\n";
  for (const auto& kv : g_table) {
    const int cat = std::get<0>(kv.first);
    if (cat != kCatInt4) f << kCatTag[cat] << ' ';
    f << std::get<1>(kv.first) << ' ' << std::get<2>(kv.first) << ' ' << std::get<3>(kv.first)
      << ' ' << cat_name(cat, kv.second) << '\n';
  }
  return f ? W4A16_OK : W4A16_ERR_INVALID_ARG;
}

int w4a16_table_load(const char* path) {
  if (path == nullptr) return W4A16_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_table_mutex);
  g_table_env_loaded = true;
  return load_table_locked(path);
}

// Times every eligible variant of a catalogue on synthetic device buffers of
// the shape (each as one CUDA graph of back-to-back launches on weight copies
// rotating through more than the L2 size) and stores the fastest in the
// table.  fmt: the FP4 format (kFmtMxfp4 / kFmtNvfp4) for kCatFp4.
static int tune_impl(int cat, int fmt, int64_t M, int64_t N, int64_t K, void* stream_v,
                     int* out_variant) {
  if (!shape_ok(M, N, K)) return W4A16_ERR_UNSUPPORTED;
  if (cat == kCatFp4 && N % 16 != 0) return W4A16_ERR_UNSUPPORTED;
  if (cat == kCatSwiglu && N % 2 != 0) return W4A16_ERR_UNSUPPORTED;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone)
    return W4A16_ERR_INVALID_ARG;

  // Synthetic operands; enough weight copies that the timed launches stream
  // them from HBM rather than L2.
  const size_t wbytes = cat == kCatInt8 ? w8a16_packed_bytes(N, K) : w4a16_packed_bytes(N, K);
  const size_t sbytes = cat == kCatFp4 ? fp4a16_scales_bytes(fmt == kFmtNvfp4 ? FP4A16_NVFP4
                                                                                : FP4A16_MXFP4, N, K)
                                       : w4a16_scales_bytes(N, K, kGroup);
  const size_t abytes = static_cast<size_t>(M) * K * 2;
  const size_t ybytes = static_cast<size_t>(M) * (cat == kCatSwiglu ? N / 2 : N) * 2;
  size_t wsbytes = 0;
  for (int id = 0; id < cat_count(cat); ++id) {
    if (!cat_eligible(cat, id, M, N, K)) continue;
    const size_t w = cat == kCatInt8 ? variant8_ws(id, M, N, K)
                     : cat == kCatFp4 ? variantf4_ws(id, M, N, K)
                                      : variant_ws(id, M, N, K);
    wsbytes = std::max(wsbytes, w);
  }
  const size_t per_copy = wbytes + sbytes + 4096;
  int copies = static_cast<int>((512ull << 20) / per_copy) + 1;
  if (copies > 16) copies = 16;
  if (copies < 1) copies = 1;

  std::vector<void*> bufs;
  auto alloc = [&](size_t b) -> void* {
    void* p = nullptr;
    if (cudaMalloc(&p, b < 256 ? 256 : b) != cudaSuccess) return nullptr;
    bufs.push_back(p);
    return p;
  };
  auto release = [&]() {
    for (void* p : bufs) cudaFree(p);
    bufs.clear();
  };
  void* A = alloc(abytes);
  void* Y = alloc(ybytes);
  void* ws = wsbytes ? alloc(wsbytes) : nullptr;
  float* ts = cat == kCatFp4 ? static_cast<float*>(alloc(256)) : nullptr;
  std::vector<void*> Wp(copies), Sc(copies);
  bool ok = A && Y && (wsbytes == 0 || ws) && (cat != kCatFp4 || ts);
  for (int c = 0; ok && c < copies; ++c) {
    Wp[c] = alloc(wbytes);
    Sc[c] = alloc(sbytes);
    ok = Wp[c] && Sc[c];
  }
  if (!ok) {
    release();
    return W4A16_ERR_CUDA;
  }
  // finite operands: bf16 activations 0x3C3C, codes 0x5A, scales of a small
  // normal value (fp16 0x1C1C; E8M0 0x7A, i.e. 2^-5; E4M3 0x30, i.e. 0.5),
  // NVFP4 tensor scale 0x3C3C3C3C (about 0.0115)
  cudaMemsetAsync(A, 0x3C, abytes, stream);
  const int sfill = cat == kCatFp4 ? (fmt == kFmtNvfp4 ? 0x30 : 0x7A) : 0x1C;
  for (int c = 0; c < copies; ++c) {
    cudaMemsetAsync(Wp[c], 0x5A, wbytes, stream);
    cudaMemsetAsync(Sc[c], sfill, sbytes, stream);
  }
  if (ts) cudaMemsetAsync(ts, 0x3C, 256, stream);
  if (ws) cudaMemsetAsync(ws, 0, wsbytes, stream);

  auto launch = [&](int id, int c, cudaStream_t st) -> int {
    switch (cat) {
      case kCatSwiglu:
        return run_gemm_v(kVariants[id], A, M, N, K, Wp[c], Sc[c], nullptr, Y, ws, wsbytes, st,
                          false, nullptr, true);
      case kCatInt8:
        return run_gemm_v(kVariants8[id], A, M, N, K, Wp[c], Sc[c], nullptr, Y, ws, wsbytes, st,
                          false);
      case kCatFp4:
        return run_gemm_v(variant_f4(id, fmt), A, M, N, K, Wp[c], Sc[c], nullptr, Y, ws, wsbytes,
                          st, false, fmt == kFmtNvfp4 ? ts : nullptr);
      default:
        return run_gemm(id, A, M, N, K, Wp[c], Sc[c], nullptr, Y, ws, wsbytes, st);
    }
  };

  // Each variant is timed as one CUDA graph of kIters launches (so host
  // launch overhead does not hide short kernels), on a private stream.
  cudaEvent_t e0, e1;
  cudaEventCreate(&e0);
  cudaEventCreate(&e1);
  cudaStream_t cs = nullptr;
  if (cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) != cudaSuccess) ok = false;
  if (ok && cudaStreamSynchronize(stream) != cudaSuccess) ok = false;
  float best_ms = 0.0f;
  int best = -1;
  constexpr int kIters = 20;
  for (int id = 0; ok && id < cat_count(cat); ++id) {
    if (!cat_eligible(cat, id, M, N, K)) continue;
    bool fine = true;
    for (int it = 0; it < 3 && fine; ++it) fine = launch(id, it % copies, cs) == W4A16_OK;
    if (!fine) continue;
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
      ok = false;
      break;
    }
    for (int it = 0; it < kIters; ++it) launch(id, it % copies, cs);
    if (cudaStreamEndCapture(cs, &graph) != cudaSuccess ||
        cudaGraphInstantiate(&exec, graph, 0) != cudaSuccess) {
      if (graph) cudaGraphDestroy(graph);
      ok = false;
      break;
    }
    cudaGraphLaunch(exec, cs);   // warm
    cudaEventRecord(e0, cs);
    cudaGraphLaunch(exec, cs);
    cudaEventRecord(e1, cs);
    const bool synced = cudaEventSynchronize(e1) == cudaSuccess;
    cudaGraphExecDestroy(exec);
    cudaGraphDestroy(graph);
    if (!synced) {
      ok = false;
      break;
    }
    float ms = 0.0f;
    cudaEventElapsedTime(&ms, e0, e1);
    if (log_enabled())
      std::fprintf(stderr, "w4a16: tune %s M=%lld N=%lld K=%lld %s %.3f us\n", kCatTag[cat],
                   static_cast<long long>(M), static_cast<long long>(N), static_cast<long long>(K),
                   cat_name(cat, id), 1000.0 * ms / kIters);
    if (best < 0 || ms < best_ms) {
      best_ms = ms;
      best = id;
    }
  }
  if (cs) {
    cudaStreamSynchronize(cs);
    cudaStreamDestroy(cs);
  }
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  cudaGetLastError();   // a failed capture leaves no sticky error behind
  const int dev_err = w4a16_get_device_error(stream);
  release();
  if (!ok) return cuda_failure(cudaErrorUnknown, "tune: graph timing failed");
  if (dev_err != W4A16_OK) return dev_err;
  if (best < 0) return W4A16_ERR_NO_VARIANT;
  const int st = table_put(cat, M, N, K, best);
  if (st != W4A16_OK) return st;
  if (out_variant) *out_variant = best;
  if (log_enabled())
    std::fprintf(stderr, "w4a16: tuned %s M=%lld N=%lld K=%lld -> %s (%.3f us)\n", kCatTag[cat],
                 static_cast<long long>(M), static_cast<long long>(N), static_cast<long long>(K),
                 cat_name(cat, best), 1000.0 * best_ms / kIters);
  return W4A16_OK;
}

int w4a16_tune(int64_t M, int64_t N, int64_t K, void* stream, int* out_variant) {
  return tune_impl(kCatInt4, kFmtInt4, M, N, K, stream, out_variant);
}

int w4a16_tune_swiglu(int64_t M, int64_t N, int64_t K, void* stream, int* out_variant) {
  return tune_impl(kCatSwiglu, kFmtInt4, M, N, K, stream, out_variant);
}

int w8a16_tune(int64_t M, int64_t N, int64_t K, void* stream, int* out_variant) {
  return tune_impl(kCatInt8, kFmtInt8, M, N, K, stream, out_variant);
}

int fp4a16_tune(int format, int64_t M, int64_t N, int64_t K, void* stream, int* out_variant) {
  const int f = fp4_format(format);
  if (f == 0) return W4A16_ERR_UNSUPPORTED;
  return tune_impl(kCatFp4, f, M, N, K, stream, out_variant);
}

int w4a16_get_device_error(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return W4A16_ERR_CUDA;
  DeviceInfo dev;
  if (!device_info(dev)) return W4A16_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpy(&word, dev.error_word, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return W4A16_ERR_CUDA;
  if (word != 0) {
    const uint32_t zero = 0;
    if (cudaMemcpy(dev.error_word, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
      return W4A16_ERR_CUDA;
    return W4A16_ERR_TIMEOUT;
  }
  return W4A16_OK;
}

void w4a16_set_wait_timeout_ns(uint64_t ns) { g_timeout_ns.store(ns == 0 ? 1 : ns); }

void w4a16_set_weights_static(int enable) { g_weights_static.store(enable != 0 ? 1 : 0); }

int w4a16_weights_static(void) { return g_weights_static.load(); }

int w4a16_selftest_wait_timeout(uint64_t timeout_ns, void* stream) {
  DeviceInfo dev;
  if (!device_info(dev)) return W4A16_ERR_CUDA;
  const cudaError_t e =
      launch_wait_timeout_selftest(dev.error_word, timeout_ns, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_failure(e, "wait_timeout_selftest");
  g_launches.fetch_add(1);
  return W4A16_OK;
}

size_t w4a16_packed_rowmajor_bytes(int64_t N, int64_t K) {
  if (N < 0 || K < 0) return 0;
  return static_cast<size_t>(N) * static_cast<size_t>(K) / 2;
}

int w4a16_repack_rowmajor(const void* packed_rowmajor, int64_t N, int64_t K, void* packed_out,
                          void* stream) {
  if (packed_rowmajor == nullptr || packed_out == nullptr) return W4A16_ERR_INVALID_ARG;
  if (N < 1 || K < 1) return W4A16_ERR_INVALID_ARG;
  if (K % kGroup != 0 || N % 8 != 0) return W4A16_ERR_UNSUPPORTED;
  if (N >= (1ll << 31) || K >= (1ll << 31) || N * K >= (1ll << 40)) return W4A16_ERR_UNSUPPORTED;
  if (!aligned16(packed_rowmajor) || !aligned16(packed_out)) return W4A16_ERR_ALIGNMENT;
  DeviceInfo dev;
  if (!device_info(dev)) return W4A16_ERR_CUDA;
  const cudaError_t e = launch_repack_rowmajor(packed_rowmajor, N, K, packed_out, dev.num_sms,
                                               static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_failure(e, "repack_rowmajor");
  g_launches.fetch_add(1);
  return W4A16_OK;
}

int w4a16_selftest_quotient(int mode, unsigned long long* counts, void* stream) {
  if (counts == nullptr) return W4A16_ERR_INVALID_ARG;
  if (mode < 0 || mode > 2) return W4A16_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(counts) & 7u) != 0) return W4A16_ERR_ALIGNMENT;
  const cudaError_t e = launch_quotient_selftest(mode, counts, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_failure(e, "quotient_selftest");
  g_launches.fetch_add(1);
  return W4A16_OK;
}

uint64_t w4a16_launch_count(void) { return g_launches.load(); }

const char* w4a16_last_error_detail(void) { return g_error_detail; }

int w4a16_gemm_noalloc(const void* A_bf16, int64_t M, int64_t N, int64_t K, const void* packed,
                       const void* scales, int group, const void* bias_bf16_or_null, void* Y_bf16,
                       void* stream) {
  const int st = check_gemm_args(A_bf16, M, N, K, packed, scales, group, bias_bf16_or_null, Y_bf16);
  if (st != W4A16_OK) return st;
  const int id = select_variant(M, N, K);
  if (id < 0) return W4A16_ERR_NO_VARIANT;
  const size_t need = variant_ws(id, M, N, K);
  if (need > kNoAllocScratchBytes) {
    std::snprintf(g_error_detail, sizeof(g_error_detail),
                  "w4a16_gemm_noalloc: variant %s needs %zu scratch bytes, the static array holds %zu",
                  kVariants[id].name, need, kNoAllocScratchBytes);
    return W4A16_ERR_WORKSPACE;
  }
  void* scratch = nullptr;
  const int sst = noalloc_scratch(&scratch);
  if (sst != W4A16_OK) return sst;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (need > 0) {
    // the arrival counters must start at zero (a call that timed out could
    // have left them set); clearing them is a memset, not an allocation
    const cudaError_t e = cudaMemsetAsync(scratch, 0, kCounterBytes, s);
    if (e != cudaSuccess) return cuda_failure(e, "cudaMemsetAsync(noalloc counters)");
  }
  return run_gemm(id, A_bf16, M, N, K, packed, scales, bias_bf16_or_null, Y_bf16,
                  need > 0 ? scratch : nullptr, need > 0 ? kNoAllocScratchBytes : 0, s);
}

}  // extern "C"
