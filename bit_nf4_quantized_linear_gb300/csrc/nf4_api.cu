// nf4_api.cu -- the extern "C" entry points declared in include/nf4.h: argument
// validation on the host, tile planning, TMA tensor-map encoding and launches.
// No allocation, no synchronisation on the hot entry points.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <cstdlib>
#include <mutex>
#include <utility>
#include <vector>

#include "internal.h"
#include "nf4.h"

namespace {

std::atomic<uint64_t> g_counters[NF4_NUM_PATHS];
thread_local char g_last_error[512] = "no error";

// Records a failed CUDA call and maps it to NF4_ERR_CUDA.
nf4_status cuda_fail(cudaError_t e, const char* where) {
  if (e == cudaSuccess) e = cudaErrorUnknown;
  std::snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%s)", where, cudaGetErrorString(e),
                cudaGetErrorName(e));
  return NF4_ERR_CUDA;
}

// Device status word: kernels record NF4_ERR_TIMEOUT / NF4_ERR_BAD_OFFSETS here.
__device__ int g_device_status;

constexpr int kMaxDevices = 64;

struct DevInfo {
  bool ok = false;
  bool supported = false;
  int sms = 0;
  int* status = nullptr;
};

std::mutex g_mu;
DevInfo g_dev[kMaxDevices];

thread_local int t_bound_device = -1;

// The current device's cached properties.  The first call on a thread (and after
// a device switch) binds the device's primary context to the thread: driver calls
// such as cuTensorMapEncodeTiled need a current context, and threads the caller
// did not initialise (e.g. autograd's backward worker) have none yet.
bool current_device(DevInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  if (t_bound_device != dev) {
    if (cudaSetDevice(dev) != cudaSuccess) return false;
    t_bound_device = dev;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  DevInfo& d = g_dev[dev];
  if (!d.ok) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess)
      return false;
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    d.supported = (major == 10 && minor == 3);
    d.sms = sms;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return false;
    d.status = static_cast<int*>(p);
    d.ok = true;
  }
  *out = d;
  return true;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool encode_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner,
               uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
               CUtensorMapSwizzle sw) {
  auto fn = tensor_map_encoder();
  if (!fn) {
    std::snprintf(g_last_error, sizeof(g_last_error), "cuTensorMapEncodeTiled entry point not found");
    return false;
  }
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    std::snprintf(g_last_error, sizeof(g_last_error),
                  "cuTensorMapEncodeTiled failed (CUresult %d): base %p dims %llu x %llu stride %llu "
                  "box %u x %u",
                  static_cast<int>(r), base, static_cast<unsigned long long>(inner),
                  static_cast<unsigned long long>(outer), static_cast<unsigned long long>(row_bytes),
                  box_inner, box_outer);
  return r == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Tensor map of the codes for one contraction step: the forward reads 128 weight
// rows x 64 values, the input gradient 64 rows x 128 values.  4-bit codes: 32-byte
// rows (32B swizzle) / 64-byte rows (64B swizzle); 8-bit codes: 64-byte rows (64B
// swizzle) / 128-byte rows (128B swizzle).  The swizzles keep the decoders'
// 16-byte loads bank-conflict free.
bool encode_codes(CUtensorMap* m, const nf4_weight* w, int mode) {
  const int bits = w->bits == 8 ? 8 : 4;
  const uint64_t row_bytes = static_cast<uint64_t>(w->K) * bits / 8;
  if (mode == 0)
    return encode_2d(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, w->packed, row_bytes, w->N, row_bytes,
                     nf4::kTileK * bits / 8, nf4::kTileW,
                     bits == 8 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
  return encode_2d(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, w->packed, row_bytes, w->N, row_bytes,
                   nf4::kTileW * bits / 8, nf4::kTileK,
                   bits == 8 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
}

void count(int path) {
  g_counters[path].fetch_add(1, std::memory_order_relaxed);
  g_counters[NF4_PATH_TOTAL].fetch_add(1, std::memory_order_relaxed);
}

nf4_status check_weight(const nf4_weight* w) {
  if (!w || !w->packed || !w->code4) return NF4_ERR_INVALID_ARG;
  if (w->bits != 0 && w->bits != 4 && w->bits != 8) return NF4_ERR_INVALID_ARG;
  if (w->N < 1 || w->K < 1) return NF4_ERR_INVALID_ARG;
  if (w->blocksize != 64) return NF4_ERR_UNSUPPORTED;
  if (w->double_quant != 0 && w->double_quant != 1) return NF4_ERR_INVALID_ARG;
  if (w->double_quant) {
    if (!w->absmax_q || !w->nested_absmax || !w->nested_offset || !w->code8)
      return NF4_ERR_INVALID_ARG;
    if (w->nested_blocksize != nf4::kNestedBlock) return NF4_ERR_UNSUPPORTED;
  } else if (!w->absmax) {
    return NF4_ERR_INVALID_ARG;
  }
  return NF4_OK;
}

int choose_bt(int64_t M) {
  if (M <= 16) return 16;
  if (M <= 32) return 32;
  if (M <= 64) return 64;
  if (M <= 128) return 128;
  return 256;
}

struct Plan {
  int bt, wtiles, ttiles, splits, ksteps;
  int64_t items;
  size_t ws_bytes;
  bool gemv = false;  // small M: SIMT GEMV kernels
  bool skinny = false;  // small M: tensor-core (mma.sync) kernels
  nf4::SkinnyPlan sk;
  bool stream_k = false;  // fused kernel with the stream-K schedule
  int sk_ctas = 0;
  int cs = 0;  // cluster split: CTAs per tile (one cluster), 0 for none
  // Token split: the last `tail` tokens run as a second launch with tail_bt-token
  // single-CTA tiles (the plan's other fields describe the first M - tail tokens).
  int64_t tail = 0;
  int tail_bt = 0;
};

Plan make_plan(int64_t M, int64_t ncols, int64_t contract, int bt, int splits) {
  Plan p;
  p.bt = bt;
  const int64_t tw = bt == 512 ? 2 * nf4::kTileW : nf4::kTileW;  // CTA pairs: 256-row weight tiles
  p.wtiles = static_cast<int>((ncols + tw - 1) / tw);
  p.ttiles = static_cast<int>((M + bt - 1) / bt);
  p.ksteps = static_cast<int>((contract + nf4::kTileK - 1) / nf4::kTileK);
  p.splits = splits;
  p.items = static_cast<int64_t>(p.wtiles) * p.ttiles * splits;
  p.ws_bytes = splits > 1 ? static_cast<size_t>(splits) * M * ncols * sizeof(float) : 0;
  return p;
}

// Whether the small-M kernels may read the weight before the grid dependency on
// the previous kernel resolves (nf4_set_weight_prefetch).
std::atomic<int> g_weight_prefetch{0};

// Kernels for M <= 16 (nf4_set_small_m_path).
std::atomic<int> g_small_m_path{NF4_SMALL_M_AUTO};

// One-shot failure-path test hooks (nf4_inject_stream_k_timeout,
// nf4_inject_bounds_failure).
std::atomic<int> g_inject_sk_timeout{0};
std::atomic<int> g_inject_bounds{0};

// Stream-K schedule of the fused kernel (nf4_set_stream_k).
std::atomic<int> g_stream_k{NF4_STREAM_K_AUTO};

// Cluster split of the fused kernel (nf4_set_cluster_split).
std::atomic<int> g_cluster_split{NF4_CLUSTER_SPLIT_AUTO};

// Fixed token tile of the fused kernel, 0 for the planner's choice (nf4_set_token_tile).
std::atomic<int> g_token_tile{0};

// Clusters of cs CTAs that can be resident at once: the device's answer when one is
// current, else the SM count's bound (host-only plan queries).
int cluster_capacity(int mode, int bt, int cs, int sms, bool query_device) {
  if (query_device) {
    const int n = nf4::gemm_cluster_capacity(mode, bt, cs);
    if (n > 0) return n;
  }
  return sms / cs;
}

// Epoch a stream-K launch publishes in its ready flags: unique per launch of the
// process, never 0.  The flags live in the caller's workspace and the CTA that
// finishes a tile clears them, so a launch replayed from a CUDA graph (same epoch)
// finds them cleared by its previous replay.
std::atomic<uint64_t> g_sk_epoch{0};

uint64_t next_sk_epoch() {
  uint64_t e = g_sk_epoch.fetch_add(1, std::memory_order_relaxed) + 1;
  while (e == 0) e = g_sk_epoch.fetch_add(1, std::memory_order_relaxed) + 1;
  return e ^ 0x5a17c0de00000000ull;  // unlikely to match what a fresh buffer holds
}

// Cycles of one 64-deep contraction step of a tile (per SM), as measured on
// GB300 with the timeline probes: about 0.40 us for tiles of up to 128 tokens
// (bound by the MMA issuer's barrier round trips), about 0.46 us for 256 tokens
// (MMA time plus activation-ring stalls).
// CTA pairs (512-token tiles): two MMAs of M = 256, N = 256 per step on one decoded
// weight tile per CTA.
double step_cycles(int bt) {
  if (bt >= 512) return 1650.0;
  if (bt >= 256) return 950.0;
  return 830.0;
}

// Tile plan of a dense product: a deterministic function of the shape and the SM
// count.  Small M: the narrowest token tile and, when the weight tiles cannot fill
// the SMs, a split of the contraction while its fp32 partials stay small next to
// the packed weight.  Larger M: token tile and split chosen by a cost
// model in SM clocks -- waves of items times contraction steps, plus the split
// partials' round trip through memory.
Plan plan_dense(int mode, int64_t M, int64_t N, int64_t K, int sms, bool allow_sk = true,
                int bits = 4, bool f16 = false, bool allow_cs = true, bool query_device = false,
                int force_bt = 0) {
  const int64_t ncols = mode == 0 ? N : K;
  const int64_t contract = mode == 0 ? K : N;
  const int small = g_small_m_path.load(std::memory_order_relaxed);
  nf4::SkinnyPlan sk;
  // 8-bit codes (tiles of <= 128 tokens) run the fused tcgen05 kernel at every M;
  // small M with 4-bit codes takes the warp-MMA kernels (bf16 or fp16 operands),
  // or the SIMT GEMV (bf16 only).
  const bool skinny_ok = bits == 4;
  const bool gemv_ok = bits == 4 && !f16;
  if (skinny_ok && M > 0 && small == NF4_SMALL_M_AUTO && nf4::skinny_plan(mode, M, N, K, sms, &sk, f16)) {
    Plan p = make_plan(M, ncols, contract, 16, 1);
    p.skinny = true;
    p.sk = sk;
    p.items = 0;
    p.ws_bytes = 0;
    return p;
  }
  if (gemv_ok && M > 0 && small != NF4_SMALL_M_TILES &&
      M <= (mode == 0 ? nf4::kGemvMaxMFwd : nf4::kGemvMaxMDgrad)) {
    Plan p = make_plan(M, ncols, contract, 16, 1);
    p.gemv = true;
    p.items = 0;
    const int64_t groups = mode == 0 ? 1 : nf4::gemv_dgrad_row_groups(N);
    p.ws_bytes = groups > 1 ? static_cast<size_t>(groups) * M * K * sizeof(float) : 0;
    return p;
  }
  const int64_t ksteps = (contract + nf4::kTileK - 1) / nf4::kTileK;
  const int64_t wtiles = (ncols + nf4::kTileW - 1) / nf4::kTileW;
  if (M <= 32) {
    const int bt = choose_bt(M);
    int64_t s = 1;
    if (M > 0 && wtiles < sms) {
      s = sms / wtiles;  // one wave: a second, partial wave would double the time
      s = s < ksteps / 4 ? s : ksteps / 4;
      const int64_t traffic_cap = contract / (16 * M);
      s = s < traffic_cap ? s : traffic_cap;
      s = s < 32 ? s : 32;
      s = s < 1 ? 1 : s;
    }
    return make_plan(M, ncols, contract, bt, static_cast<int>(s));
  }
  // A fixed tile (nf4_set_token_tile) is the only candidate.  512-token tiles are
  // CTA-pair tiles (4-bit codes, from M = 1024).
  const int fixed_bt = force_bt > 0 ? force_bt : g_token_tile.load(std::memory_order_relaxed);
  int bt_max = bits == 8 && choose_bt(M) > 128 ? 128 : (bits == 4 && M >= 1024 ? 512 : choose_bt(M));
  if (fixed_bt > 0) bt_max = bits == 8 && fixed_bt > 128 ? 128 : fixed_bt;
  const int bt_min = fixed_bt > 0 ? bt_max : 0;
  const int cand_bt[4] = {512, 256, 128, 64};
  const int sp[7] = {1, 2, 3, 4, 5, 6, 8};
  const int skm = allow_sk ? g_stream_k.load(std::memory_order_relaxed) : NF4_STREAM_K_OFF;
  double best_t = 1e300, sk_t = 1e300;
  Plan best = make_plan(M, ncols, contract, bt_max, 1);
  Plan sk_best = best;
  for (int ci = 0; ci < 4; ++ci) {
    const int bt = cand_bt[ci];
    if (bt > bt_max || bt < bt_min) continue;
    const bool pair = bt == 512;
    const int64_t ttiles = (M + bt - 1) / bt;
    const int64_t tw = pair ? 2 * nf4::kTileW : nf4::kTileW;
    const int64_t wt = (ncols + tw - 1) / tw;
    // pairs: the clusters of two that can be resident at once
    const int64_t units = pair ? cluster_capacity(mode, bt, 2, sms, query_device) : sms;
    if (units < 1) continue;
    for (int si = 0; si < 7; ++si) {
      const int S = sp[si];
      if (S > 1 && ksteps / S < 8) break;
      if (S > 1 && force_bt > 0) break;  // the parts of a token split: whole contractions, no workspace
      const int64_t items = wt * ttiles * S;
      const int64_t waves = (items + units - 1) / units;
      const int64_t kps = (ksteps + S - 1) / S;
      // per wave: the steps and the epilogue (pairs: one accumulator, so the next
      // tile's MMAs wait for it)
      double t = static_cast<double>(waves) * (kps * step_cycles(bt) + (pair ? 6000.0 : 3000.0));
      if (S > 1) t += static_cast<double>(S) * M * ncols * 8.0 / 3500.0;  // write + read partials
      if (t < best_t * 0.999) {
        best_t = t;
        best = make_plan(M, ncols, contract, bt, S);
      }
    }
    if (skm != NF4_STREAM_K_OFF && sms <= nf4::kSkMaxCtas && !pair) {
      // Stream-K: equal runs of the items' contraction steps, one per CTA (each at
      // least one step), whose steps measured about 2% slower than those of whole
      // tiles, plus a fixed cost for the split tiles' partials (the CTA finishing a
      // split tile brings the next CTA's partial into shared memory with one bulk
      // copy; measured on GB300: about 19000 cycles at 256-token tiles).
      const int64_t U = wt * ttiles * ksteps;
      const int64_t G = U < sms ? U : sms;
      const double t = static_cast<double>((U + G - 1) / G) * step_cycles(bt) * 1.02 + 5000.0 +
                       14000.0 * bt / 256.0;
      if (G >= 1 && t < sk_t * 0.999) {
        sk_t = t;
        sk_best = make_plan(M, ncols, contract, bt, 1);
        sk_best.stream_k = true;
        sk_best.sk_ctas = static_cast<int>(G);
        sk_best.ws_bytes = nf4::stream_k_ws_bytes(static_cast<int>(G), bt);
      }
    }
  }
  // Cluster split: when every tile, cut into cs contraction slices (2..8, at least
  // 32 tokens of the tile per slice), fits the device in one wave of clusters, the
  // slices of a tile run on the cs CTAs of one cluster and meet in shared memory:
  // no fp32 partials in global memory and no reduction kernel.  Cost: the slice's
  // steps, plus a fixed cost and the exchange (each rank writes (cs - 1) / cs of
  // its partial tile through distributed shared memory).
  const int csm = allow_cs && bits == 4 ? g_cluster_split.load(std::memory_order_relaxed)
                                        : NF4_CLUSTER_SPLIT_OFF;
  Plan cs_best;
  double cs_t = 1e300;
  if (csm != NF4_CLUSTER_SPLIT_OFF) {
    const int cand_cs[3] = {2, 4, 8};
    for (int ci = 0; ci < 4; ++ci) {
      const int bt = cand_bt[ci];
      if (bt > bt_max || bt < bt_min || bt > 256) continue;
      const int64_t ttiles = (M + bt - 1) / bt;
      const int64_t tiles = ((ncols + nf4::kTileW - 1) / nf4::kTileW) * ttiles;
      for (int si = 0; si < 3; ++si) {
        const int cs = cand_cs[si];
        if (bt / cs < 32 || ksteps < cs) continue;
        // receive and outgoing blocks of the partials fit the idle rings
        const size_t xchg = 2 * static_cast<size_t>(cs - 1) * 4 * 32 * (bt / cs + 4) * 4;
        if (xchg > nf4::gemm_exchange_bytes(bt, 4)) continue;
        if (tiles > cluster_capacity(mode, bt, cs, sms, query_device)) continue;
        const double t = static_cast<double>((ksteps + cs - 1) / cs) * step_cycles(bt) + 3000.0 +
                         1500.0 + 8.0 * bt * (cs - 1) / cs;
        if (t < cs_t * 0.999) {
          cs_t = t;
          cs_best = make_plan(M, ncols, contract, bt, cs);
          cs_best.cs = cs;
          cs_best.ws_bytes = 0;
        }
      }
    }
  }
  double best_any = best_t;
  Plan chosen = best;
  // Token split of a CTA-pair plan: the first tA 512-token tiles on pairs, the rest
  // in one more launch of 256-token single-CTA tiles, when the pairs' last round
  // would be mostly empty (each round of pair tiles after the first also waits for
  // the previous accumulator's drain, in the 6000-cycle term).  Cost of a launch
  // beyond the first: about 20000 cycles of start-up and drain (measured at
  // M = 512).  Taken when 3% cheaper: at K = N = 4096 from M = 8192 (four pair
  // rounds become three plus one round of single tiles).
  if (chosen.bt == 512 && fixed_bt == 0 && bits == 4 && !f16 && skm != NF4_STREAM_K_FORCE) {
    const int64_t wt2 = (ncols + 2 * nf4::kTileW - 1) / (2 * nf4::kTileW);
    const int64_t pairs = cluster_capacity(mode, 512, 2, sms, query_device);
    if (pairs >= 1) {
      const int64_t ks = (contract + nf4::kTileK - 1) / nf4::kTileK;
      auto pair_cost = [&](int64_t m) {
        const int64_t items = wt2 * ((m + 511) / 512);
        return static_cast<double>((items + pairs - 1) / pairs) * (ks * step_cycles(512) + 6000.0);
      };
      auto single_cost = [&](int64_t m) {
        const int64_t items = wtiles * ((m + 255) / 256);
        return static_cast<double>((items + sms - 1) / sms) * (ks * step_cycles(256) + 3000.0);
      };
      const double launch = 20000.0;
      double split_t = pair_cost(M) + launch;
      int64_t split_a = 0;
      for (int64_t ta = 1; ta * 512 < M; ++ta) {
        const double t = pair_cost(ta * 512) + single_cost(M - ta * 512) + 2.0 * launch;
        if (t < split_t * 0.97) {
          split_t = t;
          split_a = ta * 512;
        }
      }
      if (split_a > 0) {
        chosen = make_plan(split_a, ncols, contract, 512, 1);
        chosen.tail = M - split_a;
        chosen.tail_bt = 256;
        return chosen;
      }
    }
  }
  if (sk_best.stream_k && (skm == NF4_STREAM_K_FORCE || sk_t < best_t * 0.97)) {
    chosen = sk_best;
    best_any = sk_t;
  }
  // The cluster split is taken unless the other schedules' estimate is more than
  // 15% below it: measured on GB300 (Llama-3.1-8B projections at M = 512) it beat
  // stream-K wherever it fits -- by 20% on the 4096-wide projections and by 5% on
  // the 224-step contractions (gate / up input gradient, down forward) whose
  // stream-K runs cut every tile between two or three CTAs -- while the model put
  // both within a few percent.
  if (cs_best.cs > 1 && (csm == NF4_CLUSTER_SPLIT_FORCE ||
                         (skm != NF4_STREAM_K_FORCE && cs_t < best_any * 1.15)))
    return cs_best;
  return chosen;
}

nf4_status run_dense(int mode, const void* act, int64_t M, int64_t ld_act, const nf4_weight* w,
                     void* out, int64_t ld_out, void* ws, size_t ws_bytes, void* stream,
                     bool allow_sk = true, bool f16 = false, int force_bt = 0) {
  nf4_status st = check_weight(w);
  if (st != NF4_OK) return st;
  const int64_t N = w->N, K = w->K;
  if (M < 0) return NF4_ERR_INVALID_ARG;
  if (K % 64 != 0) return NF4_ERR_UNSUPPORTED_SHAPE;
  const int64_t act_cols = mode == 0 ? K : N;
  const int64_t out_cols = mode == 0 ? N : K;
  if (ld_act < act_cols || ld_out < out_cols) return NF4_ERR_INVALID_ARG;
  if (M == 0) return NF4_OK;
  if (!act || !out) return NF4_ERR_INVALID_ARG;
  if (ld_act % 8 != 0 || !aligned16(act) || !aligned16(w->packed)) return NF4_ERR_ALIGNMENT;
  if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return NF4_ERR_UNSUPPORTED_SHAPE;
  DevInfo dev;
  if (!current_device(&dev)) return cuda_fail(cudaGetLastError(), "device query");
  if (!dev.supported) return NF4_ERR_UNSUPPORTED;
  const int bits = w->bits == 8 ? 8 : 4;
  if (f16 && bits == 8) return NF4_ERR_UNSUPPORTED;  // fp16 dtype: 4-bit codes
  // A cluster split stores its bf16 tile with bulk tensor stores, which need a
  // 16-byte aligned output and row pitch.
  const bool out_tma_ok = aligned16(out) && ld_out % 8 == 0;
  // (a forced tile -- the parts of a token split -- takes the classic schedule)
  const Plan p = plan_dense(mode, M, N, K, dev.sms, allow_sk && force_bt == 0, bits, f16,
                            out_tma_ok && force_bt == 0, true, force_bt);
  if (p.ws_bytes > 0 && (!ws || ws_bytes < p.ws_bytes)) return NF4_ERR_WORKSPACE;
  if (p.tail > 0) {
    // Token split: two launches over row slices of the activations and the output
    // (each row computed exactly as in one launch).
    const int64_t ma = M - p.tail;
    nf4_status st2 = run_dense(mode, act, ma, ld_act, w, out, ld_out, ws, ws_bytes, stream, false, f16, 512);
    if (st2 != NF4_OK) return st2;
    const uint8_t* act_b = static_cast<const uint8_t*>(act) + ma * ld_act * 2;
    uint8_t* out_b = static_cast<uint8_t*>(out) + ma * ld_out * 2;
    return run_dense(mode, act_b, p.tail, ld_act, w, out_b, ld_out, ws, ws_bytes, stream, false, f16, p.tail_bt);
  }

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (p.skinny) {
    nf4::SkinnyArgs k{};
    k.act = static_cast<const __nv_bfloat16*>(act);
    k.ld_act = ld_act;
    k.packed = w->packed;
    k.N = N;
    k.K = K;
    k.KB = K / 64;
    k.absmax = w->absmax;
    k.absmax_q = w->absmax_q;
    k.nested_absmax = w->nested_absmax;
    k.nested_offset = w->nested_offset;
    k.code4 = w->code4;
    k.code8 = w->code8;
    k.dq = w->double_quant;
    k.f16 = f16 ? 1 : 0;
    k.out = static_cast<__nv_bfloat16*>(out);
    k.ld_out = ld_out;
    k.M = M;
    k.S = p.sk.S;
    k.C = p.sk.C;
    k.T = p.sk.T;
    k.cc = p.sk.cc;
    k.prefetch = g_weight_prefetch.load(std::memory_order_relaxed);
    k.status = dev.status;
    // The packed codes as [N rows, K/2 bytes]: the forward copies 16 rows x 128
    // bytes per unit (128B swizzle), the input gradient 64 rows x 32 bytes (32B).
    CUtensorMap tmap_pk;
    if (!encode_2d(&tmap_pk, CU_TENSOR_MAP_DATA_TYPE_UINT8, w->packed, K / 2, N, K / 2,
                   mode == 0 ? 128 : 32, mode == 0 ? 16 : 64,
                   mode == 0 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_32B))
      return NF4_ERR_CUDA;
    cudaError_t le = nf4::launch_skinny(mode, k, p.sk, tmap_pk, s);
    if (le != cudaSuccess) return cuda_fail(le, "kernel launch");
    count(mode == 0 ? NF4_PATH_SKINNY_FWD : NF4_PATH_SKINNY_DGRAD);
    return NF4_OK;
  }
  if (p.gemv) {
    nf4::GemvArgs g{};
    g.act = static_cast<const __nv_bfloat16*>(act);
    g.ld_act = ld_act;
    g.packed = w->packed;
    g.N = N;
    g.K = K;
    g.KB = K / 64;
    g.absmax = w->absmax;
    g.absmax_q = w->absmax_q;
    g.nested_absmax = w->nested_absmax;
    g.nested_offset = w->nested_offset;
    g.code4 = w->code4;
    g.code8 = w->code8;
    g.dq = w->double_quant;
    g.out = static_cast<__nv_bfloat16*>(out);
    g.ld_out = ld_out;
    g.ws = static_cast<float*>(ws);
    g.M = M;
    g.m0 = 0;
    g.kseg = nf4::gemv_fwd_kseg(K);
    g.status = dev.status;
    cudaError_t le = mode == 0 ? nf4::launch_gemv_fwd(g, s) : nf4::launch_gemv_dgrad(g, s);
    if (le != cudaSuccess) return cuda_fail(le, "kernel launch");
    count(mode == 0 ? NF4_PATH_GEMV_FWD : NF4_PATH_GEMV_DGRAD);
    if (p.ws_bytes > 0) {
      le = nf4::launch_splitk_reduce(static_cast<const float*>(ws),
                                     static_cast<int>(nf4::gemv_dgrad_row_groups(N)), M, K,
                                     out, ld_out, false, s);
      if (le != cudaSuccess) return cuda_fail(le, "kernel launch");
      count(NF4_PATH_SPLITK_REDUCE);
    }
    return NF4_OK;
  }

  CUtensorMap tmap_act, tmap_pk;
  const CUtensorMapDataType dt16 = f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  // (CTA pairs: each CTA copies 128-token quarters of the 512-token tile)
  if (!encode_2d(&tmap_act, dt16, act, act_cols, M, ld_act * 2, 64,
                 p.bt == 512 ? 128 : p.bt, CU_TENSOR_MAP_SWIZZLE_128B))
    return NF4_ERR_CUDA;
  if (!encode_codes(&tmap_pk, w, mode)) return NF4_ERR_CUDA;
  nf4::GemmArgs a{};
  a.M = M;
  a.ncols = out_cols;
  a.N_total = N;
  a.K = K;
  a.KB = K / 64;
  a.N_e = N;
  a.ksteps = p.ksteps;
  a.wtiles = p.wtiles;
  a.ttiles = p.ttiles;
  a.splits = p.splits;
  a.total_items = p.items;
  a.grouped = 0;
  a.E = 1;
  a.offsets = nullptr;
  a.absmax = w->absmax;
  a.absmax_q = w->absmax_q;
  a.nested_absmax = w->nested_absmax;
  a.nested_offset = w->nested_offset;
  a.code4 = w->code4;
  a.code8 = w->code8;
  a.dq = w->double_quant;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.ld_out = ld_out;
  a.ws = static_cast<float*>(ws);
  a.status = dev.status;
  a.prefetch = g_weight_prefetch.load(std::memory_order_relaxed);
  const int64_t units = dev.sms;
  int grid = static_cast<int>(p.items < units ? p.items : units);
  if (p.bt == 512) {  // CTA pairs: two CTAs per item, as many pairs as can be resident
    const int64_t pairs = cluster_capacity(mode, 512, 2, dev.sms, true);
    grid = 2 * static_cast<int>(p.items < pairs ? p.items : pairs);
  }
  if (p.cs > 1) {
    a.cs = p.cs;  // items = tiles x cs, one per CTA, the clusters in one wave
    grid = static_cast<int>(p.items);
  }
  a.chk_inject = g_inject_bounds.exchange(0, std::memory_order_relaxed);
  if (p.stream_k) {
    a.sk = 1;
    a.sk_units = p.items * p.ksteps;
    a.sk_ctas = p.sk_ctas;
    a.sk_ws = static_cast<float*>(ws);
    a.sk_flags = reinterpret_cast<uint64_t*>(static_cast<uint8_t*>(ws) +
                                             static_cast<size_t>(p.sk_ctas) * nf4::kTileW * p.bt * sizeof(float));
    if ((reinterpret_cast<uintptr_t>(a.sk_flags) & 7u) != 0) return NF4_ERR_ALIGNMENT;
    a.sk_epoch = next_sk_epoch();
    if (g_inject_sk_timeout.exchange(0, std::memory_order_relaxed)) a.sk_wait_xor = 1ull << 62;
    grid = p.sk_ctas;
  }
  // The bf16 output goes out through bulk tensor stores when its base and row pitch
  // meet the 16-byte rule; otherwise through direct stores.
  CUtensorMap tmap_out;
  std::memset(&tmap_out, 0, sizeof(tmap_out));
  if ((p.splits == 1 || p.cs > 1) && out_tma_ok) {
    if (!encode_2d(&tmap_out, dt16, out, out_cols, M, ld_out * 2, 32, 32,
                   CU_TENSOR_MAP_SWIZZLE_NONE))
      return NF4_ERR_CUDA;
    a.tma_out = 1;
  }
  cudaError_t le = nf4::launch_gemm(mode, p.bt, bits, f16, a, tmap_act, tmap_pk, tmap_out, grid, s);
  if (le != cudaSuccess) return cuda_fail(le, "kernel launch");
  count(mode == 0 ? NF4_PATH_LINEAR_FWD : NF4_PATH_LINEAR_DGRAD);
  if (p.stream_k)  // a property of the launch just counted, not a launch of its own
    g_counters[NF4_PATH_STREAM_K].fetch_add(1, std::memory_order_relaxed);
  if (p.cs > 1) g_counters[NF4_PATH_CLUSTER_SPLIT].fetch_add(1, std::memory_order_relaxed);
  if (p.splits > 1 && p.cs == 0) {
    le = nf4::launch_splitk_reduce(static_cast<const float*>(ws), p.splits, M, out_cols, out,
                                   ld_out, f16, s);
    if (le != cudaSuccess) return cuda_fail(le, "kernel launch");
    count(NF4_PATH_SPLITK_REDUCE);
  }
  return NF4_OK;
}

// Backward of the SwiGLU epilogue (nf4_grouped_swiglu_bwd): the grouped forward
// kernel writes dg / du instead of h; `bwd` carries the upstream gradient and the
// routing-weight partials.
struct SwigluBwd {
  const void* dh;
  int64_t ld_dh;
  float* drw;  // [N_e / 64][T] partials, or null
};

// Workspace of nf4_grouped_swiglu_bwd: dg / du in bf16 [T, N_e] (the whole block
// padded to 256 bytes), then the routing-weight partials fp32 [N_e / 64][T].
size_t swiglu_bwd_dgu_bytes(int64_t T, int64_t N_e) {
  return (static_cast<size_t>(T) * N_e * 2 + 255) / 256 * 256;
}

nf4_status run_grouped(int mode, const void* act, const int32_t* offsets, int32_t E, int64_t T,
                       int64_t ld_act, const nf4_weight* w, int64_t N_e, void* out, int64_t ld_out,
                       void* stream, const nf4_epilogue* ep = nullptr,
                       const SwigluBwd* bwd = nullptr) {
  nf4_status st = check_weight(w);
  if (st != NF4_OK) return st;
  const int64_t K = w->K;
  if (E < 1 || E > nf4::kMaxExperts || T < 0 || N_e < 1 || !offsets) return NF4_ERR_INVALID_ARG;
  if (w->N != static_cast<int64_t>(E) * N_e) return NF4_ERR_INVALID_ARG;
  if (K % 64 != 0) return NF4_ERR_UNSUPPORTED_SHAPE;
  const bool swiglu = ep && ep->swiglu;
  if (ep && (ep->swiglu != 0 && ep->swiglu != 1)) return NF4_ERR_INVALID_ARG;
  if (swiglu && N_e % 128 != 0) return NF4_ERR_UNSUPPORTED_SHAPE;
  if (bwd && (mode != 0 || !swiglu)) return NF4_ERR_INVALID_ARG;
  const int64_t act_cols = mode == 0 ? K : N_e;
  const int64_t out_cols = mode == 0 ? N_e : K;
  const int64_t out_width = swiglu && !bwd ? N_e / 2 : out_cols;
  if (ld_act < act_cols || ld_out < out_width) return NF4_ERR_INVALID_ARG;
  if (T == 0) return NF4_OK;
  if (!act || !out) return NF4_ERR_INVALID_ARG;
  if (ld_act % 8 != 0 || !aligned16(act) || !aligned16(w->packed)) return NF4_ERR_ALIGNMENT;
  if (T > INT32_MAX || w->N > INT32_MAX || K > INT32_MAX) return NF4_ERR_UNSUPPORTED_SHAPE;
  DevInfo dev;
  if (!current_device(&dev)) return cuda_fail(cudaGetLastError(), "device query");
  if (!dev.supported) return NF4_ERR_UNSUPPORTED;
  // Tokens per tile: the tile that holds twice the mean rows per expert, so that
  // an expert near the mean takes one token tile, not a full one and a ragged one
  // (the steps of a tile cost about the same from 16 to 128 tokens: the weight
  // decode bounds them).
  int bt = choose_bt(2 * ((T + E - 1) / E));
  if (w->bits == 8 && bt > 128) bt = 128;  // 8-bit codes: tiles of <= 128 tokens
  CUtensorMap tmap_act, tmap_pk;
  if (!encode_2d(&tmap_act, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, act, act_cols, T, ld_act * 2, 64, bt,
                 CU_TENSOR_MAP_SWIZZLE_128B))
    return NF4_ERR_CUDA;
  if (!encode_codes(&tmap_pk, w, mode)) return NF4_ERR_CUDA;
  nf4::GemmArgs a{};
  a.M = T;
  a.ncols = out_cols;
  a.N_total = w->N;
  a.K = K;
  a.KB = K / 64;
  a.N_e = N_e;
  a.ksteps = static_cast<int>(mode == 0 ? K / 64 : (N_e + 63) / 64);
  a.wtiles = static_cast<int>((out_cols + nf4::kTileW - 1) / nf4::kTileW);
  a.ttiles = 0;
  a.splits = 1;
  a.total_items = 0;
  a.grouped = 1;
  a.E = E;
  a.offsets = offsets;
  a.absmax = w->absmax;
  a.absmax_q = w->absmax_q;
  a.nested_absmax = w->nested_absmax;
  a.nested_offset = w->nested_offset;
  a.code4 = w->code4;
  a.code8 = w->code8;
  a.dq = w->double_quant;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.ld_out = ld_out;
  a.ws = nullptr;
  a.status = dev.status;
  if (ep) {
    a.ep_bias = ep->bias;
    a.ep_scale = ep->row_scale;
    a.ep_swiglu = ep->swiglu;
  }
  if (bwd) {
    a.ep_bwd = 1;
    a.ep_dh = static_cast<const __nv_bfloat16*>(bwd->dh);
    a.ep_ld_dh = bwd->ld_dh;
    a.ep_drw = bwd->drw;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  CUtensorMap tmap_out;  // unused: expert row ranges end inside tiles (direct stores)
  std::memset(&tmap_out, 0, sizeof(tmap_out));
  a.tma_out = 0;
  cudaError_t le = nf4::launch_gemm(mode, bt, w->bits == 8 ? 8 : 4, false, a, tmap_act,
                                    tmap_pk, tmap_out, dev.sms, s);
  if (le != cudaSuccess) return cuda_fail(le, "kernel launch");
  count(mode == 0 ? NF4_PATH_GROUPED_FWD : NF4_PATH_GROUPED_DGRAD);
  return NF4_OK;
}

// Multi-product launch (nf4_linear_fwd_multi / nf4_linear_dgrad_multi).
nf4_status run_multi(int mode, int32_t nprod, const void* const* act, int64_t M, const int64_t* ld_act,
                     const nf4_weight* const* w, void* const* out, const int64_t* ld_out, void* stream) {
  if (nprod < 1 || nprod > nf4::kMaxProds || !act || !ld_act || !w || !out || !ld_out || M < 0)
    return NF4_ERR_INVALID_ARG;
  int64_t K = -1;
  for (int p = 0; p < nprod; ++p) {
    nf4_status st = check_weight(w[p]);
    if (st != NF4_OK) return st;
    if (w[p]->bits == 8) return NF4_ERR_UNSUPPORTED;
    if (p == 0) K = w[p]->K;
    if (w[p]->K != K || w[p]->double_quant != w[0]->double_quant || w[p]->code4 != w[0]->code4 ||
        (w[0]->double_quant && w[p]->code8 != w[0]->code8))
      return NF4_ERR_INVALID_ARG;
    const int64_t act_cols = mode == 0 ? K : w[p]->N;
    const int64_t out_cols = mode == 0 ? w[p]->N : K;
    if (ld_act[p] < act_cols || ld_out[p] < out_cols) return NF4_ERR_INVALID_ARG;
    if (w[p]->N > INT32_MAX) return NF4_ERR_UNSUPPORTED_SHAPE;
  }
  if (K % 64 != 0) return NF4_ERR_UNSUPPORTED_SHAPE;
  if (M == 0) return NF4_OK;
  for (int p = 0; p < nprod; ++p) {
    if (!act[p] || !out[p]) return NF4_ERR_INVALID_ARG;
    if (ld_act[p] % 8 != 0 || ld_out[p] % 8 != 0 || !aligned16(act[p]) || !aligned16(out[p]) ||
        !aligned16(w[p]->packed))
      return NF4_ERR_ALIGNMENT;
  }
  if (M > INT32_MAX || K > INT32_MAX) return NF4_ERR_UNSUPPORTED_SHAPE;
  DevInfo dev;
  if (!current_device(&dev)) return cuda_fail(cudaGetLastError(), "device query");
  if (!dev.supported) return NF4_ERR_UNSUPPORTED;
  // Products in order of decreasing contraction (longest items dealt first).
  int order[nf4::kMaxProds];
  for (int p = 0; p < nprod; ++p) order[p] = p;
  auto ksteps_of = [&](int p) { return mode == 0 ? K / 64 : (w[p]->N + 63) / 64; };
  auto wtiles_of = [&](int p) { return ((mode == 0 ? w[p]->N : K) + nf4::kTileW - 1) / nf4::kTileW; };
  for (int i = 1; i < nprod; ++i)
    for (int j = i; j > 0 && ksteps_of(order[j]) > ksteps_of(order[j - 1]); --j) std::swap(order[j], order[j - 1]);
  // Token tile: the busiest CTA of the classic round-robin deal, in SM clocks.
  int best_bt = 128;
  double best = 1e300;
  for (int bt : {256, 128}) {
    const int64_t ttiles = (M + bt - 1) / bt;
    int64_t total = 0;
    for (int i = 0; i < nprod; ++i) total += ttiles * wtiles_of(order[i]);
    const int64_t grid = total < dev.sms ? total : dev.sms;
    std::vector<int64_t> steps(static_cast<size_t>(grid), 0);
    int64_t idx = 0;
    for (int i = 0; i < nprod; ++i) {
      const int64_t n = ttiles * wtiles_of(order[i]);
      for (int64_t k = 0; k < n; ++k, ++idx) {  // the kernel's deal: odd rounds in reverse
        const int64_t r = idx / grid, pos = idx % grid;
        steps[static_cast<size_t>((r & 1) ? grid - 1 - pos : pos)] += ksteps_of(order[i]);
      }
    }
    int64_t busiest = 0;
    for (int64_t v : steps) busiest = v > busiest ? v : busiest;
    const double cost = static_cast<double>(busiest) * step_cycles(bt);
    if (cost < best * 0.999) {
      best = cost;
      best_bt = bt;
    }
  }
  const int bt = best_bt;
  const int64_t ttiles = (M + bt - 1) / bt;
  nf4::GemmArgs a{};
  nf4::MapSet<nf4::kMaxProds> maps;
  std::memset(&maps, 0, sizeof(maps));
  int64_t item0 = 0;
  for (int i = 0; i < nprod; ++i) {
    const int p = order[i];
    const nf4_weight* wp = w[p];
    nf4::ProdArgs& pa = a.prod[i];
    pa.absmax = wp->absmax;
    pa.absmax_q = wp->absmax_q;
    pa.nested_absmax = wp->nested_absmax;
    pa.nested_offset = wp->nested_offset;
    pa.out = static_cast<__nv_bfloat16*>(out[p]);
    pa.ld_out = ld_out[p];
    pa.N_total = wp->N;
    pa.ncols = mode == 0 ? wp->N : K;
    pa.ksteps = static_cast<int>(ksteps_of(p));
    pa.wtiles = static_cast<int>(wtiles_of(p));
    pa.item0 = item0;
    item0 += ttiles * pa.wtiles;
    const int64_t act_cols = mode == 0 ? K : wp->N;
    const int64_t out_cols = mode == 0 ? wp->N : K;
    if (!encode_2d(&maps.act[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, act[p], act_cols, M, ld_act[p] * 2, 64, bt,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_codes(&maps.pk[i], wp, mode) ||
        !encode_2d(&maps.out[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, out[p], out_cols, M, ld_out[p] * 2, 32, 32,
                   CU_TENSOR_MAP_SWIZZLE_NONE))
      return NF4_ERR_CUDA;
  }
  if (item0 > INT32_MAX) return NF4_ERR_UNSUPPORTED_SHAPE;
  a.M = M;
  a.K = K;
  a.KB = K / 64;
  a.ncols = a.prod[0].ncols;
  a.N_total = a.prod[0].N_total;
  a.N_e = a.prod[0].N_total;
  a.ksteps = a.prod[0].ksteps;
  a.wtiles = a.prod[0].wtiles;
  a.ttiles = static_cast<int>(ttiles);
  a.splits = 1;
  a.total_items = item0;
  a.grouped = 0;
  a.E = 1;
  a.absmax = a.prod[0].absmax;
  a.absmax_q = a.prod[0].absmax_q;
  a.nested_absmax = a.prod[0].nested_absmax;
  a.nested_offset = a.prod[0].nested_offset;
  a.code4 = w[0]->code4;
  a.code8 = w[0]->code8;
  a.dq = w[0]->double_quant;
  a.out = a.prod[0].out;
  a.ld_out = a.prod[0].ld_out;
  a.status = dev.status;
  a.prefetch = g_weight_prefetch.load(std::memory_order_relaxed);
  a.tma_out = 1;
  a.nprod = nprod;
  a.chk_inject = g_inject_bounds.exchange(0, std::memory_order_relaxed);
  const int grid = static_cast<int>(item0 < dev.sms ? item0 : dev.sms);
  cudaError_t le = nf4::launch_gemm_multi(mode, bt, a, maps, grid, static_cast<cudaStream_t>(stream));
  if (le != cudaSuccess) return cuda_fail(le, "kernel launch");
  count(NF4_PATH_MULTI);
  return NF4_OK;
}

// Top-k combine of the experts, or its backward (nf4_moe_combine / _bwd).
nf4_status run_moe(bool backward, const void* src, int64_t src_rows, int64_t ld_src,
                          const int32_t* token_rows, int64_t tokens, int32_t k, int64_t R, int64_t H, void* dst,
                          int64_t ld_dst, void* stream) {
  if (k < 1 || tokens < 0 || R < 0 || H < 0 || src_rows < 0) return NF4_ERR_INVALID_ARG;
  if (ld_src < H || ld_dst < H) return NF4_ERR_INVALID_ARG;
  if (H % 8 != 0) return NF4_ERR_UNSUPPORTED_SHAPE;
  if (tokens == 0 || H == 0) return NF4_OK;
  if (!src || !dst || !token_rows) return NF4_ERR_INVALID_ARG;
  if (!aligned16(src) || !aligned16(dst) || ld_src % 8 != 0 || ld_dst % 8 != 0) return NF4_ERR_ALIGNMENT;
  if (tokens > INT32_MAX || R > INT32_MAX || H > INT32_MAX) return NF4_ERR_UNSUPPORTED_SHAPE;
  DevInfo dev;
  if (!current_device(&dev)) return cuda_fail(cudaGetLastError(), "device query");
  nf4::MoeArgs a{};
  a.rows = static_cast<const __nv_bfloat16*>(src);
  a.ld_rows = ld_src;
  a.token_rows = token_rows;
  a.k = k;
  a.tokens = tokens;
  a.R = R;
  a.H = H;
  a.out = static_cast<__nv_bfloat16*>(dst);
  a.ld_out = ld_dst;
  a.status = dev.status;
  cudaError_t le = nf4::launch_moe(backward, a, static_cast<cudaStream_t>(stream));
  if (le != cudaSuccess) return cuda_fail(le, "kernel launch");
  count(NF4_PATH_MOE_COMBINE);
  return NF4_OK;
}

}  // namespace

extern "C" {

nf4_status nf4_quantize(const void* W, int32_t w_dtype, int64_t N, int64_t K, int32_t blocksize,
                        int32_t double_quant, int32_t nested_blocksize, const float* code4,
                        const float* code8, uint8_t* packed, float* absmax, uint8_t* absmax_q,
                        float* nested_absmax, float* nested_offset, void* ws, size_t ws_bytes,
                        void* stream) {
  if (!W || !code4 || !packed || !absmax || N < 1 || K < 1) return NF4_ERR_INVALID_ARG;
  if (w_dtype != NF4_DTYPE_F32 && w_dtype != NF4_DTYPE_BF16) return NF4_ERR_INVALID_ARG;
  if (blocksize != 64) return NF4_ERR_UNSUPPORTED;
  if (double_quant != 0 && double_quant != 1) return NF4_ERR_INVALID_ARG;
  const int64_t numel = N * K;
  const int64_t nblocks = (numel + 63) / 64;
  if (double_quant) {
    if (nested_blocksize != nf4::kNestedBlock) return NF4_ERR_UNSUPPORTED;
    if (!code8 || !absmax_q || !nested_absmax || !nested_offset) return NF4_ERR_INVALID_ARG;
    const size_t need = static_cast<size_t>((nblocks + nf4::kMeanChunk - 1) / nf4::kMeanChunk) * 8;
    if (!ws || ws_bytes < need) return NF4_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & 7u) != 0) return NF4_ERR_ALIGNMENT;
  }
  DevInfo dev;
  if (!current_device(&dev)) return cuda_fail(cudaGetLastError(), "device query");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t le = nf4::launch_quantize(W, w_dtype, numel, code4, packed, absmax, s);
  if (le != cudaSuccess) return cuda_fail(le, "kernel launch");
  count(NF4_PATH_QUANTIZE);
  if (double_quant) {
    le = nf4::launch_double_quant(absmax, nblocks, code8, absmax_q, nested_absmax, nested_offset,
                                  static_cast<double*>(ws), s);
    if (le != cudaSuccess) return cuda_fail(le, "kernel launch");
  }
  return NF4_OK;
}

nf4_status nf4_quantize_8bit(const void* W, int32_t w_dtype, int64_t N, int64_t K,
                             int32_t blocksize, int32_t double_quant, int32_t nested_blocksize,
                             const float* code, const float* code8, uint8_t* codes,
                             float* absmax, uint8_t* absmax_q, float* nested_absmax,
                             float* nested_offset, void* ws, size_t ws_bytes, void* stream) {
  if (!W || !code || !codes || !absmax || N < 1 || K < 1) return NF4_ERR_INVALID_ARG;
  if (w_dtype != NF4_DTYPE_F32 && w_dtype != NF4_DTYPE_BF16) return NF4_ERR_INVALID_ARG;
  if (blocksize != 64) return NF4_ERR_UNSUPPORTED;
  if (double_quant != 0 && double_quant != 1) return NF4_ERR_INVALID_ARG;
  const int64_t numel = N * K;
  const int64_t nblocks = (numel + 63) / 64;
  if (double_quant) {
    if (nested_blocksize != nf4::kNestedBlock) return NF4_ERR_UNSUPPORTED;
    if (!code8 || !absmax_q || !nested_absmax || !nested_offset) return NF4_ERR_INVALID_ARG;
    const size_t need = static_cast<size_t>((nblocks + nf4::kMeanChunk - 1) / nf4::kMeanChunk) * 8;
    if (!ws || ws_bytes < need) return NF4_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & 7u) != 0) return NF4_ERR_ALIGNMENT;
  }
  DevInfo dev;
  if (!current_device(&dev)) return cuda_fail(cudaGetLastError(), "device query");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t le = nf4::launch_quantize8(W, w_dtype, numel, code, codes, absmax, s);
  if (le != cudaSuccess) return cuda_fail(le, "kernel launch");
  count(NF4_PATH_QUANTIZE);
  if (double_quant) {
    le = nf4::launch_double_quant(absmax, nblocks, code8, absmax_q, nested_absmax, nested_offset,
                                  static_cast<double*>(ws), s);
    if (le != cudaSuccess) return cuda_fail(le, "kernel launch");
  }
  return NF4_OK;
}

nf4_status nf4_dequantize(const nf4_weight* w, void* out, int32_t out_dtype, void* stream) {
  nf4_status st = check_weight(w);
  if (st != NF4_OK) return st;
  if (!out) return NF4_ERR_INVALID_ARG;
  if (out_dtype != NF4_DTYPE_F32 && out_dtype != NF4_DTYPE_BF16) return NF4_ERR_INVALID_ARG;
  DevInfo dev;
  if (!current_device(&dev)) return cuda_fail(cudaGetLastError(), "device query");
  cudaError_t le = nf4::launch_dequantize(*w, out, out_dtype, static_cast<cudaStream_t>(stream));
  if (le != cudaSuccess) return cuda_fail(le, "kernel launch");
  count(NF4_PATH_DEQUANTIZE);
  return NF4_OK;
}

nf4_status nf4_linear_fwd(const void* x, int64_t M, int64_t ldx, const nf4_weight* w, void* y,
                          int64_t ldy, void* ws, size_t ws_bytes, void* stream) {
  return run_dense(0, x, M, ldx, w, y, ldy, ws, ws_bytes, stream);
}

nf4_status nf4_linear_dgrad(const void* gy, int64_t M, int64_t ldgy, const nf4_weight* w, void* gx,
                            int64_t ldgx, void* ws, size_t ws_bytes, void* stream) {
  return run_dense(1, gy, M, ldgy, w, gx, ldgx, ws, ws_bytes, stream);
}

nf4_status nf4_linear_fwd_f16(const void* x, int64_t M, int64_t ldx, const nf4_weight* w, void* y,
                              int64_t ldy, void* ws, size_t ws_bytes, void* stream) {
  return run_dense(0, x, M, ldx, w, y, ldy, ws, ws_bytes, stream, true, true);
}

nf4_status nf4_linear_dgrad_f16(const void* gy, int64_t M, int64_t ldgy, const nf4_weight* w,
                                void* gx, int64_t ldgx, void* ws, size_t ws_bytes, void* stream) {
  return run_dense(1, gy, M, ldgy, w, gx, ldgx, ws, ws_bytes, stream, true, true);
}

nf4_status nf4_grouped_fwd(const void* x, const int32_t* offsets, int32_t E, int64_t T, int64_t ldx,
                           const nf4_weight* w, int64_t N_e, void* y, int64_t ldy, void* stream) {
  return run_grouped(0, x, offsets, E, T, ldx, w, N_e, y, ldy, stream);
}

nf4_status nf4_grouped_fwd_ep(const void* x, const int32_t* offsets, int32_t E, int64_t T,
                              int64_t ldx, const nf4_weight* w, int64_t N_e, const nf4_epilogue* ep,
                              void* y, int64_t ldy, void* stream) {
  if (!ep) return NF4_ERR_INVALID_ARG;
  return run_grouped(0, x, offsets, E, T, ldx, w, N_e, y, ldy, stream, ep);
}

nf4_status nf4_grouped_dgrad(const void* gy, const int32_t* offsets, int32_t E, int64_t T,
                             int64_t ldgy, const nf4_weight* w, int64_t N_e, void* gx, int64_t ldgx,
                             void* stream) {
  return run_grouped(1, gy, offsets, E, T, ldgy, w, N_e, gx, ldgx, stream);
}

nf4_status nf4_grouped_swiglu_bwd(const void* x, const int32_t* offsets, int32_t E, int64_t T,
                                  int64_t ldx, const nf4_weight* w, int64_t N_e,
                                  const nf4_epilogue* ep, const void* gh, int64_t ldgh, void* gx,
                                  int64_t ldgx, float* grad_row_scale, void* ws, size_t ws_bytes,
                                  void* stream) {
  if (!ep || ep->swiglu != 1) return NF4_ERR_INVALID_ARG;
  if (grad_row_scale && !ep->row_scale) return NF4_ERR_INVALID_ARG;
  if (T < 0 || N_e < 1 || ldgh < N_e / 2) return NF4_ERR_INVALID_ARG;
  if (T == 0) return NF4_OK;
  if (!gh || !gx) return NF4_ERR_INVALID_ARG;
  if (ldgh % 8 != 0 || (reinterpret_cast<uintptr_t>(gh) & 15u) != 0) return NF4_ERR_ALIGNMENT;
  const size_t need = nf4_workspace_size(NF4_OP_GROUPED_SWIGLU_BWD, T, N_e, w ? w->K : 0, E);
  if (!ws || ws_bytes < need) return NF4_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return NF4_ERR_ALIGNMENT;
  uint8_t* base = static_cast<uint8_t*>(ws);
  void* dgu = base;  // bf16 [T, N_e]
  float* part = grad_row_scale ? reinterpret_cast<float*>(base + swiglu_bwd_dgu_bytes(T, N_e)) : nullptr;
  SwigluBwd b{gh, ldgh, part};
  nf4_status st = run_grouped(0, x, offsets, E, T, ldx, w, N_e, dgu, N_e, stream, ep, &b);
  if (st != NF4_OK) return st;
  st = run_grouped(1, dgu, offsets, E, T, N_e, w, N_e, gx, ldgx, stream);
  if (st != NF4_OK) return st;
  if (grad_row_scale) {
    cudaError_t le = nf4::launch_row_partial_sum(part, static_cast<int>(N_e / 64), T, offsets, E,
                                                 grad_row_scale, static_cast<cudaStream_t>(stream));
    if (le != cudaSuccess) return cuda_fail(le, "kernel launch");
    count(NF4_PATH_SPLITK_REDUCE);
  }
  return NF4_OK;
}

size_t nf4_workspace_size(int32_t op, int64_t M, int64_t N, int64_t K, int32_t E) {
  (void)E;
  if (op == NF4_OP_GROUPED_SWIGLU_BWD) {
    if (M <= 0 || N <= 0) return 0;
    return swiglu_bwd_dgu_bytes(M, N) + static_cast<size_t>(N / 64) * M * sizeof(float);
  }
  if (op == NF4_OP_QUANTIZE) {
    const int64_t nblocks = (N * K + 63) / 64;
    return static_cast<size_t>((nblocks + nf4::kMeanChunk - 1) / nf4::kMeanChunk) * 8;
  }
  if (op == NF4_OP_LINEAR_FWD || op == NF4_OP_LINEAR_DGRAD) {
    if (M <= 0 || N <= 0 || K <= 0) return 0;
    DevInfo dev;
    if (!current_device(&dev)) return 0;
    // Enough for either code width (the plan depends on it).
    const int mode = op == NF4_OP_LINEAR_FWD ? 0 : 1;
    size_t need = 0;
    for (int v = 0; v < 6; ++v) {  // 4-bit bf16, 8-bit bf16, 4-bit fp16; aligned output or not
      const size_t b = plan_dense(mode, M, N, K, dev.sms, true, v % 3 == 1 ? 8 : 4, v % 3 == 2, v < 3,
                                  true).ws_bytes;
      need = b > need ? b : need;
    }
    return need;
  }
  return 0;
}

const char* nf4_status_string(nf4_status s) {
  switch (s) {
    case NF4_OK: return "ok";
    case NF4_ERR_INVALID_ARG: return "invalid argument";
    case NF4_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case NF4_ERR_ALIGNMENT: return "pointer or leading dimension not 16-byte aligned";
    case NF4_ERR_WORKSPACE: return "workspace too small";
    case NF4_ERR_CUDA: return "CUDA error";
    case NF4_ERR_TIMEOUT: return "device wait timed out";
    case NF4_ERR_UNSUPPORTED: return "unsupported device or parameter";
    case NF4_ERR_BAD_OFFSETS: return "expert offsets out of contract";
    case NF4_ERR_BOUNDS: return "an in-kernel index check failed (checked build)";
  }
  return "unknown status";
}

int32_t nf4_checked_build(void) { return NF4_CHECKED ? 1 : 0; }

nf4_status nf4_moe_combine(const void* rows, int64_t R, int64_t ld_rows, const int32_t* token_rows,
                           int64_t tokens, int32_t k, int64_t H, void* out, int64_t ld_out, void* stream) {
  return run_moe(false, rows, R, ld_rows, token_rows, tokens, k, R, H, out, ld_out, stream);
}

nf4_status nf4_moe_combine_bwd(const void* grad_out, int64_t tokens, int64_t ld_grad_out,
                               const int32_t* token_rows, int32_t k, int64_t R, int64_t H, void* grad_rows,
                               int64_t ld_grad_rows, void* stream) {
  return run_moe(true, grad_out, tokens, ld_grad_out, token_rows, tokens, k, R, H, grad_rows, ld_grad_rows,
                 stream);
}

nf4_status nf4_linear_fwd_multi(int32_t nprod, const void* const* x, int64_t M, const int64_t* ldx,
                                const nf4_weight* const* w, void* const* y, const int64_t* ldy, void* stream) {
  return run_multi(0, nprod, x, M, ldx, w, y, ldy, stream);
}

nf4_status nf4_linear_dgrad_multi(int32_t nprod, const void* const* gy, int64_t M, const int64_t* ldgy,
                                  const nf4_weight* const* w, void* const* gx, const int64_t* ldgx,
                                  void* stream) {
  return run_multi(1, nprod, gy, M, ldgy, w, gx, ldgx, stream);
}

void nf4_get_path_counters(uint64_t* out) {
  if (!out) return;
  for (int i = 0; i < NF4_NUM_PATHS; ++i) out[i] = g_counters[i].load(std::memory_order_relaxed);
}

void nf4_reset_path_counters(void) {
  for (int i = 0; i < NF4_NUM_PATHS; ++i) g_counters[i].store(0, std::memory_order_relaxed);
}

nf4_status nf4_device_status(int32_t* out, int32_t clear) {
  if (!out) return NF4_ERR_INVALID_ARG;
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_device_status, sizeof(int));
  if (e != cudaSuccess) return cuda_fail(e, "device status copy");
  *out = v;
  if (clear) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "device status copy");
  }
  return NF4_OK;
}

const char* nf4_last_cuda_error(void) { return g_last_error; }

void nf4_set_small_m_path(int32_t path) {
  if (path >= NF4_SMALL_M_AUTO && path <= NF4_SMALL_M_TILES)
    g_small_m_path.store(path, std::memory_order_relaxed);
}

void nf4_set_stream_k(int32_t mode) {
  if (mode >= NF4_STREAM_K_OFF && mode <= NF4_STREAM_K_FORCE)
    g_stream_k.store(mode, std::memory_order_relaxed);
}

void nf4_set_cluster_split(int32_t mode) {
  if (mode >= NF4_CLUSTER_SPLIT_OFF && mode <= NF4_CLUSTER_SPLIT_FORCE)
    g_cluster_split.store(mode, std::memory_order_relaxed);
}

void nf4_set_token_tile(int32_t tokens) {
  if (tokens == 0 || tokens == 64 || tokens == 128 || tokens == 256 || tokens == 512)
    g_token_tile.store(tokens, std::memory_order_relaxed);
}

void nf4_inject_stream_k_timeout(void) { g_inject_sk_timeout.store(1, std::memory_order_relaxed); }

void nf4_inject_bounds_failure(void) { g_inject_bounds.store(1, std::memory_order_relaxed); }

nf4_status nf4_plan_query(int32_t op, int64_t M, int64_t N, int64_t K, int32_t sms, int32_t bits,
                          int32_t f16, nf4_plan_info* out) {
  if (!out || (op != NF4_OP_LINEAR_FWD && op != NF4_OP_LINEAR_DGRAD) || sms < 1 ||
      (bits != 4 && bits != 8) || (f16 && bits == 8) || M <= 0 || N <= 0 || K <= 0)
    return NF4_ERR_INVALID_ARG;
  const int mode = op == NF4_OP_LINEAR_FWD ? 0 : 1;
  const Plan p = plan_dense(mode, M, N, K, sms, true, bits, f16 != 0, true, true);
  nf4_plan_info r{};
  r.kernel = p.skinny ? NF4_PLAN_SMALL_M_MMA : p.gemv ? NF4_PLAN_SIMT_GEMV : NF4_PLAN_FUSED;
  r.token_tile = p.bt;
  r.splits = p.splits;
  r.stream_k = p.stream_k ? 1 : 0;
  if (p.skinny) {
    r.grid = p.sk.S * p.sk.C;
  } else if (!p.gemv) {
    const int64_t units = sms;
    r.grid = p.stream_k ? p.sk_ctas : static_cast<int32_t>(p.items < units ? p.items : units);
    if (p.bt == 512) {  // CTA pairs: two CTAs per item
      const int64_t pairs = cluster_capacity(op == NF4_OP_LINEAR_FWD ? 0 : 1, 512, 2, sms, true);
      r.grid = 2 * static_cast<int32_t>(p.items < pairs ? p.items : pairs);
    }
  }
  r.items = p.items;
  r.workspace_bytes = p.ws_bytes;
  r.cluster_split = p.cs;
  r.tail_tokens = static_cast<int32_t>(p.tail);
  r.tail_token_tile = p.tail_bt;
  *out = r;
  return NF4_OK;
}

void nf4_set_weight_prefetch(int32_t enabled) {
  g_weight_prefetch.store(enabled ? 1 : 0, std::memory_order_relaxed);
}

nf4_status nf4_device_check(int32_t* sm_count) {
  DevInfo dev;
  if (!current_device(&dev)) return cuda_fail(cudaGetLastError(), "device query");
  if (sm_count) *sm_count = dev.sms;
  return dev.supported ? NF4_OK : NF4_ERR_UNSUPPORTED;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free forward.
//
// For callers that cannot call cudaMalloc -- e.g. code running under an
// allocator that owns all device memory and forbids direct allocation, or a
// plugin that is handed only its input and output buffers -- this variant of
// nf4_linear_fwd takes no workspace.  Its split-contraction partials live in a
// fixed file-scope device array instead, so the call itself allocates nothing.
// ---------------------------------------------------------------------------
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[NF4_NOALLOC_SCRATCH_BYTES];

std::mutex g_noalloc_mu;
void* g_noalloc_addr[kMaxDevices];  // device address of the array, per device

// Device address of the scratch array on the current device.  Host code cannot
// use the symbol itself (on the host it names a stand-in, not device memory), so
// the address is looked up once per device, with that device current.
nf4_status noalloc_scratch(void** out) {
  DevInfo dev;
  if (!current_device(&dev)) return cuda_fail(cudaGetLastError(), "device query");
  int d = 0;
  cudaError_t e = cudaGetDevice(&d);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_addr[d]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) return cuda_fail(e, "cudaGetSymbolAddress(scratch)");
    g_noalloc_addr[d] = p;
  }
  *out = g_noalloc_addr[d];
  return NF4_OK;
}

}  // namespace

extern "C" nf4_status nf4_linear_fwd_noalloc(const void* x, int64_t M, int64_t ldx,
                                             const nf4_weight* w, void* y, int64_t ldy,
                                             void* stream) {
  nf4_status st = check_weight(w);
  if (st != NF4_OK) return st;
  if (M < 0 || ldx < w->K || ldy < w->N) return NF4_ERR_INVALID_ARG;
  if (w->K % 64 != 0) return NF4_ERR_UNSUPPORTED_SHAPE;
  if (M == 0) return NF4_OK;
  DevInfo dev;
  if (!current_device(&dev)) return cuda_fail(cudaGetLastError(), "device query");
  if (!dev.supported) return NF4_ERR_UNSUPPORTED;
  // The stream-K schedule is not used here (its partial tiles outgrow the array);
  // shapes whose split partials would not fit are rejected up front.
  if (plan_dense(0, M, w->N, w->K, dev.sms, false, w->bits == 8 ? 8 : 4, false,
                 aligned16(y) && ldy % 8 == 0, true).ws_bytes > NF4_NOALLOC_SCRATCH_BYTES)
    return NF4_ERR_WORKSPACE;
  void* scratch = nullptr;
  st = noalloc_scratch(&scratch);
  if (st != NF4_OK) return st;
  // Every partial the kernel later reads is written first in the same call, so
  // what a previous call left in the array is never read and needs no clearing.
  return run_dense(0, x, M, ldx, w, y, ldy, scratch, NF4_NOALLOC_SCRATCH_BYTES, stream, false);
}
