// nf4_gemm.cu -- fused NF4 dequantise-and-multiply on the 5th-generation tensor
// cores (tcgen05 + tensor memory) of sm_103a.
//
// Computes, straight from the packed 4-bit codes and the (nested) block
// statistics, with no dense weight ever written to global memory:
//   forward         y[t, n]  = sum_k x[t, k]  * Wb[n, k]
//   input gradient  gx[t, k] = sum_n gy[t, n] * Wb[n, k]
// where Wb = bf16(fp32(code4[q] * absmax')) is the dequantised weight
// (bitsandbytes issue "MatMul4Bit keeps B and quant_state on ctx ...", "Root
// cause": the backward is grad_output @ dequantize_4bit(B, state); Soup issue
// #842, "Design sketch": a fused forward and a transposed fused backward that
// never materialise W, with a deterministic reduction).
//
// Structure (one CTA per SM, persistent over its work; 19 warps):
//   warp 0      TMA producer of code tiles (a deep ring, far ahead);
//   warp 18     TMA producer of activation tiles [BT tokens x 64] (128B swizzle);
//   warps 6-17  decoders, three groups of four, group g taking contraction steps
//               j = g mod 3: each thread turns one 64-value block (one scale) into
//               the 16-bit operand -- 4-bit codes through a register codebook (byte
//               permutes), 8-bit codes through a per-lane shared codebook -- and
//               stores it in the UMMA canonical 128B-swizzled layout of the A
//               operand (K-major for the forward, MN-major for the input gradient);
//   warp 1      MMA issuer: tcgen05.mma M=128 (weight rows / in-features), N=BT
//               (tokens), K=16, fp32 accumulators in tensor memory, two
//               accumulator buffers so the epilogue overlaps the next item; one
//               barrier wait and one commit per contraction step;
//   warps 2-5   epilogue: tcgen05.ld of the accumulator, rounding, bulk tensor
//               stores through shared memory (or direct stores), the grouped
//               expert epilogue (bias, row scale, SwiGLU), stream-K partials.
// Every output element gets a fixed order of MMAs and, when its tile is split
// (small-M contraction split, or stream-K), partials added in a fixed order: by a
// second kernel, or by the CTA holding the tile's first steps.  No atomics.
// Every wait is bounded; on timeout the kernel records the error and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "internal.h"
#include "decode.cuh"
#include "sm100_ptx.cuh"

// Code width and operand type of the kernel instances this translation unit
// launches: 4-bit codes with bf16 operands here, 8-bit codes when nf4_gemm8.cu
// compiles this file again, fp16 operands when nf4_gemm_f16.cu does.
#ifndef NF4_GEMM_BITS
#define NF4_GEMM_BITS 4
#endif
#ifndef NF4_GEMM_F16
#define NF4_GEMM_F16 0
#endif
#define NF4_GEMM_MAIN_TU (NF4_GEMM_BITS == 4 && NF4_GEMM_F16 == 0)

namespace nf4 {
namespace {

using namespace nf4ptx;

constexpr int kDecGroups = 3;                    // decoder groups of four warps
constexpr int kNumDecWarps = 4 * kDecGroups;
constexpr int kWarpTma = 0;   // packed-code producer
constexpr int kWarpMma = 1;
constexpr int kWarpEpi0 = 2;
constexpr int kNumEpiWarps = 4;
constexpr int kWarpDec0 = 6;
constexpr int kWarpTmaX = kWarpDec0 + kNumDecWarps;  // activation producer
constexpr int kThreads = (kWarpTmaX + 1) * 32;
constexpr int kAStage = kTileW * kTileK * 2;  // 16 KB of bf16
constexpr int kMiscBase = 8192;  // codebooks, barriers, expert tables
constexpr int kOutWarpBytes = 32 * 32 * 2;        // epilogue staging: 32 tokens x 32 bf16 per warp
constexpr int kOutBytes = 4 * kOutWarpBytes;
constexpr uint64_t kTimeoutNs = 2000000000ull;  // bound of every wait (2 s)
constexpr uint32_t kSleepHintNs = 20000;         // a waiting thread sleeps up to 20 us per try

// BITS = 4: two codes per byte (packed nibbles, 16-level codebook in registers);
// BITS = 8: one code per byte (256-level codebook in shared memory after the base
// misc region, one copy per lane: entry e of lane l in word 32 e + l, so the
// lookups of a warp never share a bank).
//
// BT = 512 is the CTA-pair tile: the two CTAs of a cluster share each MMA of
// M = 256 weight rows (each decodes its own 128 rows) and N = 256 tokens (each
// holds 128 of them), two such MMAs per step for the tile's two 256-token halves,
// into one 512-column accumulator per CTA.  A decoded weight tile then serves 512
// tokens, and each CTA's activation stage is 256 token rows (two 128-row copies).
template <int BT, int BITS>
struct Geo {
  static constexpr bool kPair = BT == 512;
  static constexpr int kPkStage = kTileW * kTileK * BITS / 8;  // codes of one step: 4 or 8 KB
  static constexpr int kMiscBytes = kMiscBase + (BITS == 8 ? 256 * 32 * 4 : 0);
  static constexpr int kXRows = kPair ? BT / 2 : BT;  // token rows of a step's activation tile here
  static constexpr int kXStage = kXRows * 128;        // of 64 bf16 each
  static constexpr int kXParts = kPair ? 2 : 1;       // bulk tensor copies per stage
  static constexpr int kXPartRows = kXRows / kXParts;
  static constexpr int kMmaN = kPair ? 256 : BT;      // tokens per MMA
  static constexpr int kAccCols = kPair ? 512 : BT;   // accumulator columns of a tile
  static constexpr int kAccBufs = kPair ? 1 : 2;      // accumulators in tensor memory
  static constexpr int kBudget = 225 * 1024 - kMiscBytes - 1024;
  // Decoded operand tiles: one slot more than decoder groups, so a group never
  // waits on the MMAs of the step just before -- except at 256 tokens, where the
  // activation tiles take the room (pairs make room with a shallower code ring).
  static constexpr int kStagesA = BT == 256 ? kDecGroups : kDecGroups + 1;
  static constexpr int kStagesP = (BT <= 64 ? 16 : (kPair ? 4 : 8)) / (BITS / 4);  // code tiles, prefetched far ahead
  static constexpr int kStagesX0 =
      (kBudget - kStagesA * kAStage - kStagesP * kPkStage - kOutBytes) / kXStage;
  static constexpr int kStagesX = kStagesX0 > 8 ? 8 : kStagesX0;  // activation tiles
  static constexpr int kOffA = 0;
  static constexpr int kOffX = kOffA + kStagesA * kAStage;
  static constexpr int kOffPk = kOffX + kStagesX * kXStage;
  static constexpr int kOffOut = kOffPk + kStagesP * kPkStage;  // output staging
  static constexpr int kOffMisc = kOffOut + kOutBytes;
  static constexpr int kSmem = kOffMisc + kMiscBytes + 1024;
  static constexpr uint32_t kTmemCols =
      (kAccBufs * kAccCols < 32) ? 32u : static_cast<uint32_t>(kAccBufs * kAccCols);
  static_assert(kTmemCols <= 512, "tensor memory columns");
  static_assert(kStagesX >= 3, "pipeline too shallow");
  static_assert(kStagesA <= 8 && kStagesP <= 16 && kStagesX <= 8, "barrier slots");
  // A decoded slot waits on the "stage done" ring for the step kStagesA back; that
  // ring slot must not be able to complete again first.
  static_assert(kStagesX >= kStagesA, "stage-done ring shallower than the decoded ring");
  static_assert(kStagesA >= kDecGroups && kStagesP >= kDecGroups && kStagesX >= kDecGroups,
                "a decoder group advances every ring by kDecGroups slots per step");
  static_assert(kXStage % 1024 == 0, "activation stage must keep 1024-byte alignment");
  static_assert(BITS == 4 || (BITS == 8 && BT <= 128), "8-bit codes: tiles of <= 128 tokens");
  static_assert(kXPartRows <= 256, "a bulk tensor copy box is at most 256 rows");
};

// Barrier slots in the misc region.  Three rings advance one stage per
// contraction step: packed codes (pfull: TMA landed; pempty: decoders read it),
// activations (xfull: TMA landed; xempty: MMAs done, the "stage done" signal
// that also frees the decoded slot of the same step) and decoded operand tiles
// (afull: decoders wrote it).
constexpr int kBarPFull = 0;
constexpr int kBarPEmpty = 16;
constexpr int kBarXFull = 32;
constexpr int kBarXEmpty = 40;
constexpr int kBarAFull = 48;
constexpr int kBarAccFull = 56;
constexpr int kBarAccEmpty = 58;
constexpr int kBarDrain = 60;
constexpr int kBarEpFull = 61;   // SwiGLU epilogue: up values of a batch written (2 warp pairs)
constexpr int kBarEpEmpty = 63;  // ... and read by the gate warp
constexpr int kBarSkPart = 65;   // stream-K: a lower CTA's partial landed (one per epilogue warp)
constexpr int kBarCsFree = 69;   // cluster split: every other rank's ring is free (their arrivals)
constexpr int kBarCsRecv = 70;   // cluster split: the other ranks' partials of this rank's slice landed
constexpr int kNumBars = 71;
// Misc region: codebooks (16 + 256 fp32), barriers, four words (tensor-memory
// slot, abort flag, item count, dependency flag), three expert tables.
static_assert((16 + 256) * 4 + kNumBars * 8 + 16 + 3 * (kMaxExperts + 1) * 4 <= kMiscBase,
              "misc region overflow");

struct Item {
  int64_t idx;    // item (tile) index
  int64_t tok0, tok_end;
  int64_t wrow0;  // forward: first weight row of the tile; input gradient: first row of the expert
  int64_t col0;   // first output column of the tile
  int ks0, ks1;   // contraction steps of this segment of the item
  int split;
  int p;          // product of a multi-product launch (0 otherwise)
};

struct Shared {
  float* code4;
  float* code8;
  uint32_t bars;  // shared address of barrier 0
  uint32_t* tmem_slot;
  volatile int* abort_flag;
  int* starts;
  int* ends;
  int* pref;
  uint32_t rank;  // CTA pairs: rank in the cluster (0 otherwise)
};

__device__ __forceinline__ uint32_t bar_at(const Shared& sh, int i) { return sh.bars + 8u * i; }

// 0 until the grid dependency has resolved (set when the weight-side roles start
// early), then 1; the word after the tensor-memory slot, abort flag and item count.
__device__ __forceinline__ volatile int* dep_done(const Shared& sh) {
  return reinterpret_cast<volatile int*>(sh.tmem_slot + 3);
}

__device__ __forceinline__ void record_error(const GemmArgs& a, int code) {
  *reinterpret_cast<volatile int*>(a.status) = code;
}

// Barrier among `count` threads (a multiple of 32) of the CTA, id 1..15.
__device__ __forceinline__ void named_barrier_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Programmatic dependent launch: wait for the preceding grid on the stream
// (its results visible), and let the next grid launch early.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void allow_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Bounded wait, slow path: true once the phase completed; false on abort (another
// role gave up) or after kTimeoutNs, in which case the timeout is recorded.  The
// bound runs from the later of the wait's start and the resolution of the grid
// dependency: the roles that start early wait on phases that follow it.
__device__ __noinline__ bool wait_phase_slow(uint32_t bar, uint32_t parity, const Shared& sh,
                                             const GemmArgs& a) {
  uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait_sleep(bar, parity, kSleepHintNs)) return true;
    if (*sh.abort_flag) return false;
    const uint64_t now = globaltimer_ns();
    if (!*dep_done(sh)) {
      t0 = now;
    } else if (now - t0 > kTimeoutNs) {
      *sh.abort_flag = 1;
      record_error(a, kStatusTimeout);
      return false;
    }
  }
}

// Bounded wait: an inline non-blocking test first (the common case on a pipelined
// ring, where the phase has completed already), the sleeping slow path otherwise.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, const Shared& sh,
                                           const GemmArgs& a) {
  if (mbar_test_wait(bar, parity)) return true;
  return wait_phase_slow(bar, parity, sh, a);
}

// Bounded wait on a phase completed by arrivals of other CTAs of the cluster
// (acquire at cluster scope); as wait_phase otherwise.
__device__ __noinline__ bool wait_phase_cluster_slow(uint32_t bar, uint32_t parity, const Shared& sh,
                                                     const GemmArgs& a) {
  uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait_sleep_cluster(bar, parity, kSleepHintNs)) return true;
    if (*sh.abort_flag) return false;
    const uint64_t now = globaltimer_ns();
    if (!*dep_done(sh)) {
      t0 = now;
    } else if (now - t0 > kTimeoutNs) {
      *sh.abort_flag = 1;
      record_error(a, kStatusTimeout);
      return false;
    }
  }
}

__device__ __forceinline__ bool wait_phase_cluster(uint32_t bar, uint32_t parity, const Shared& sh,
                                                   const GemmArgs& a) {
  if (mbar_test_wait_cluster(bar, parity)) return true;
  return wait_phase_cluster_slow(bar, parity, sh, a);
}

// Wait used while draining on exit: bounded, ignores the abort flag.
__device__ __noinline__ void drain_phase(uint32_t bar, uint32_t parity, const GemmArgs& a) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait_sleep(bar, parity, kSleepHintNs)) {
    if (globaltimer_ns() - t0 > kTimeoutNs) {
      record_error(a, kStatusTimeout);
      return;
    }
  }
}

// Stream-K partial-tile flags: publish with release semantics after the partial's
// stores; wait (bounded) with acquire semantics before reading it.
__device__ __forceinline__ void flag_publish(uint64_t* f, uint64_t v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(f), "l"(v) : "memory");
}

__device__ __forceinline__ uint64_t flag_read(const uint64_t* f) {
  uint64_t v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(f) : "memory");
  return v;
}

__device__ __noinline__ bool flag_wait(const uint64_t* f, uint64_t v, const Shared& sh,
                                       const GemmArgs& a) {
  if (flag_read(f) == v) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    __nanosleep(64);
    if (flag_read(f) == v) return true;
    if (*sh.abort_flag) return false;
    if (globaltimer_ns() - t0 > kTimeoutNs) {
      *sh.abort_flag = 1;
      record_error(a, kStatusTimeout);
      return false;
    }
  }
}

template <int MODE, int BT, bool MULTI>
__device__ __forceinline__ Item get_item(int64_t idx, const GemmArgs& a, const Shared& sh) {
  Item it;
  it.idx = idx;
  it.p = 0;
  if constexpr (MULTI) {
    // Multi-product launch: the product holding item idx, then its (token tile,
    // weight tile); whole items (no splits), one 128-row weight tile each.
    int p = 0;
#pragma unroll
    for (int q = 1; q < kMaxProds; ++q)
      if (q < a.nprod && idx >= a.prod[q].item0) p = q;
    const int r = static_cast<int>(idx - a.prod[p].item0);  // (items of a launch fit in 32 bits)
    const int wtiles = a.prod[p].wtiles;
    const int wt = r % wtiles;
    const int tt = r / wtiles;
    it.p = p;
    it.tok0 = static_cast<int64_t>(tt) * BT;
    it.tok_end = min(a.M, it.tok0 + BT);
    it.ks0 = 0;
    it.ks1 = a.prod[p].ksteps;
    it.split = 0;
    it.col0 = static_cast<int64_t>(wt) * kTileW;
    it.wrow0 = (MODE == 0) ? it.col0 : 0;
    return it;
  }
  if (!a.grouped) {
    const int64_t s = idx % a.splits;
    const int64_t r = idx / a.splits;
    const int64_t wt = r % a.wtiles;
    const int64_t tt = r / a.wtiles;
    it.tok0 = tt * BT;
    it.tok_end = min(a.M, it.tok0 + BT);
    it.ks0 = static_cast<int>((s * a.ksteps) / a.splits);
    it.ks1 = static_cast<int>(((s + 1) * a.ksteps) / a.splits);
    it.split = static_cast<int>(s);
    // CTA pairs: a weight tile is 256 rows (or in-features), of which this CTA
    // holds the 128 of its rank.
    it.col0 = BT == 512 ? wt * 2 * kTileW + kTileW * static_cast<int64_t>(sh.rank) : wt * kTileW;
    it.wrow0 = (MODE == 0) ? it.col0 : 0;
  } else {
    const int64_t g = idx / a.wtiles;
    const int64_t wt = idx % a.wtiles;
    int lo = 0, hi = a.E;  // last e with pref[e] <= g
    while (hi - lo > 1) {
      int mid = (lo + hi) >> 1;
      if (sh.pref[mid] <= g) lo = mid; else hi = mid;
    }
    const int e = lo;
    const int64_t tt = g - sh.pref[e];
    it.tok0 = sh.starts[e] + tt * BT;
    it.tok_end = min(static_cast<int64_t>(sh.ends[e]), it.tok0 + BT);
    it.ks0 = 0;
    it.ks1 = a.ksteps;
    it.split = 0;
    it.col0 = wt * kTileW;
    it.wrow0 = (MODE == 0) ? static_cast<int64_t>(e) * a.N_e + it.col0
                           : static_cast<int64_t>(e) * a.N_e;
  }
  return it;
}

// The CTA's sequence of item segments.  Classic: whole items unit, unit + nunits,
// ... (their contraction split fixed by the plan).  Stream-K: the contiguous run
// of contraction steps [unit * U / G, (unit + 1) * U / G) over items in order, cut
// at item boundaries and walked from its last item back to its first (the steps
// of each segment still in increasing order): the segment a CTA contributes to a
// tile finished elsewhere (its run's last item) comes first, the segment it
// finishes itself (its run's first item, when cut) comes last.  Every role of the
// CTA walks the same sequence.
struct Cursor {
  int64_t pos, end;  // stream-K: the run's first step and the end of what is left
  int64_t unit;      // multi-product launches: this CTA (pos counts its rounds)
};

__device__ __forceinline__ int64_t sk_first_unit(const GemmArgs& a, int64_t cta) {
  return cta * a.sk_units / a.sk_ctas;
}

template <bool MULTI>
__device__ __forceinline__ Cursor cursor_begin(const GemmArgs& a, int64_t unit,
                                               int64_t total_items) {
  if (MULTI) return Cursor{0, total_items, unit};
  if (a.sk) return Cursor{sk_first_unit(a, unit), sk_first_unit(a, unit + 1), unit};
  return Cursor{unit, total_items, unit};
}

template <int MODE, int BT, bool MULTI>
__device__ __forceinline__ bool cursor_next(Cursor& c, const GemmArgs& a, const Shared& sh,
                                            int64_t nunits, Item& it) {
  if constexpr (MULTI) {
    // Multi-product launches deal whole items in rounds of nunits, odd rounds in
    // reverse CTA order (the items come longest first, so a CTA that took a long
    // item in one round takes a short one in the next).
    const int64_t idx = c.pos * nunits + ((c.pos & 1) ? nunits - 1 - c.unit : c.unit);
    if (idx >= c.end) return false;
    ++c.pos;
    it = get_item<MODE, BT, MULTI>(idx, a, sh);
    return true;
  }
  if (c.pos >= c.end) return false;
  if (!a.sk) {
    it = get_item<MODE, BT, MULTI>(c.pos, a, sh);
    c.pos += nunits;
    return true;
  }
  const int64_t idx = (c.end - 1) / a.ksteps;  // last item with steps left
  const int64_t tile0 = idx * a.ksteps;
  const int64_t seg0 = c.pos > tile0 ? c.pos : tile0;
  it = get_item<MODE, BT, MULTI>(idx, a, sh);
  it.ks0 = static_cast<int>(seg0 - tile0);
  it.ks1 = static_cast<int>(c.end - tile0);
  c.end = seg0;
  return true;
}

// Raw statistics of one block, fetched ahead of use: the fp32 absmax, or the
// 8-bit code and its nested absmax.  Out-of-range blocks read as scale 0.
struct RawScale {
  float v;     // absmax, or nested absmax under double quantisation
  uint32_t q;  // 8-bit code (double quantisation)
};

// Read-only global loads kept where the program puts them (volatile asm is not
// moved past the barrier waits around it), so that a fetch issued steps ahead of
// its use stays ahead instead of being scheduled next to the use.
__device__ __forceinline__ float ldg_keep_f32(const float* p) {
  float v;
  asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t ldg_keep_u8(const uint8_t* p) {
  uint16_t v;
  asm volatile("ld.global.nc.u8 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

// Multi-product launches: the statistics of product p, whose index travels in
// bits 8.. of q.
template <bool MULTI>
__device__ __forceinline__ RawScale fetch_scale(const GemmArgs& a, int p, int64_t n, int64_t kb) {
  RawScale r{0.0f, MULTI ? static_cast<uint32_t>(p) << 8 : 0u};
  const int64_t N_total = MULTI ? a.prod[p].N_total : a.N_total;
  if (n >= N_total || kb >= a.KB) return r;
  const int64_t b = n * a.KB + kb;
  if (!in_bounds(n >= 0 && kb >= 0 && !a.chk_inject, a.status)) return r;
  if (!a.dq) {
    r.v = ldg_keep_f32((MULTI ? a.prod[p].absmax : a.absmax) + b);
  } else {
    r.q |= ldg_keep_u8((MULTI ? a.prod[p].absmax_q : a.absmax_q) + b);
    r.v = ldg_keep_f32((MULTI ? a.prod[p].nested_absmax : a.nested_absmax) + (b >> 8));
  }
  return r;
}

// Decoded block scale: absmax, or fp32(fp32(code8[q] * nested) + offset), with the
// nested offset of the block's product (multi-product launches: offsets_s[p], in
// shared memory).
template <bool MULTI>
__device__ __forceinline__ float finish_scale(const GemmArgs& a, const float* code8_s,
                                              const RawScale& r, float offset, const float* offsets_s) {
  if (!a.dq) return r.v;
  if constexpr (MULTI) return __fadd_rn(__fmul_rn(code8_s[r.q & 255u], r.v), offsets_s[r.q >> 8]);
  return __fadd_rn(__fmul_rn(code8_s[r.q], r.v), offset);
}

// fp32 to the output / operand 16-bit type (bf16, or IEEE fp16 when F16), RNE.
template <bool F16>
__device__ __forceinline__ uint16_t to16(float f) {
  if constexpr (F16) return __half_as_ushort(__float2half_rn(f));
  else return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// Cluster-split epilogue of the CTA's tile (one epilogue warp per TMEM row
// quarter q).  The cs CTAs of this cluster hold one contraction slice each of the
// same tile, and rank p finishes token slice p (W = BT / cs tokens).  The CTA's
// rings [0, kOffOut) are idle once its single tile's MMAs are done; they hold a
// receive block and an outgoing block per (other rank, row quarter), each 32 rows
// x W tokens fp32 at a row pitch of W + 4 floats (so that the 16-byte row reads
// and writes are conflict-free).  Each warp stages its fp32 partial of every other
// slice in its outgoing blocks, and once every other rank's rings are idle one
// lane sends each block to its owner with one bulk copy (shared memory to the
// other CTA's shared memory), completing on the owner's receive barrier.  The owner
// then adds the partials of its own slice in rank order (its own from tensor
// memory) and stores bf16 through its 2 KB staging slice and bulk tensor stores
// (tokens past M are not written).
template <int BT, int BITS, bool F16>
__device__ __forceinline__ void cs_epilogue(const GemmArgs& a, const Shared& sh, uint8_t* smem, uint32_t sbase,
                                            const CUtensorMap* tmap_out, const Item& it, uint32_t taddr,
                                            int q, int ntok) {
  using G = Geo<BT, BITS>;
  const int lane = threadIdx.x & 31;
  const int S = a.cs;
  const int rank = static_cast<int>(cluster_ctarank());
  const int W = BT / S;
  const int pitch = W + 4;
  const int blk = 32 * pitch * 4;  // bytes of a block
  auto recv_off = [&](int slot, int qq) { return (slot * kNumEpiWarps + qq) * blk; };
  auto out_off = [&](int slot, int qq) { return ((S - 1 + slot) * kNumEpiWarps + qq) * blk; };
  bool cs_ok = 2 * (S - 1) * kNumEpiWarps * blk <= G::kOffOut && W % 32 == 0;
  if (!cs_ok) record_error(a, NF4_ERR_UNSUPPORTED_SHAPE);
  if (cs_ok) {
    // 1. The partials of the other slices into the outgoing blocks (block slot of
    // rank p: p, skipping this rank).
    for (int p = 0; p < S; ++p) {
      if (p == rank) continue;
      uint8_t* dst = smem + out_off(p < rank ? p : p - 1, q) + lane * pitch * 4;
      for (int c0 = 0; c0 < W && p * W + c0 < ntok; c0 += 16) {
        uint32_t v[16];
        tmem_ld_32x32b_x16(taddr + p * W + c0, v);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; j += 4)
          *reinterpret_cast<uint4*>(dst + (c0 + j) * 4) = make_uint4(v[j], v[j + 1], v[j + 2], v[j + 3]);
      }
    }
    fence_proxy_async_smem();  // the stores above, then the bulk copies that read them
    __syncwarp();
    // 2. This rank expects its receive blocks, then tells every other rank that its
    // rings are idle.
    if (q == 0 && lane == 0) {
      mbar_arrive_expect_tx(bar_at(sh, kBarCsRecv), static_cast<uint32_t>((S - 1) * kNumEpiWarps * blk));
      for (int p = 0; p < S; ++p)
        if (p != rank) mbar_arrive_cluster(mapa_shared(bar_at(sh, kBarCsFree), static_cast<uint32_t>(p)));
    }
    // 3. Once every other rank's rings are idle, send each its blocks (this rank's
    // block slot there: rank, skipping p).
    cs_ok = wait_phase_cluster(bar_at(sh, kBarCsFree), 0, sh, a);
    if (cs_ok && lane == 0)
      for (int p = 0; p < S; ++p) {
        if (p == rank) continue;
        bulk_copy_s2cluster(mapa_shared(sbase + recv_off(rank < p ? rank : rank - 1, q), static_cast<uint32_t>(p)),
                            sbase + out_off(p < rank ? p : p - 1, q), static_cast<uint32_t>(blk),
                            mapa_shared(bar_at(sh, kBarCsRecv), static_cast<uint32_t>(p)));
      }
  }
  // 4. This rank's slice: the ranks' partials added in rank order, to bf16.
  if (cs_ok) cs_ok = wait_phase_cluster(bar_at(sh, kBarCsRecv), 0, sh, a);
  if (cs_ok) {
    const int t0 = rank * W;
    uint16_t* stg = reinterpret_cast<uint16_t*>(smem + G::kOffOut + q * kOutWarpBytes);
    const uint32_t stg_addr = sbase + G::kOffOut + q * kOutWarpBytes;
#pragma unroll 1
    for (int c0 = 0; c0 < W && t0 + c0 < ntok; c0 += 32) {
      if (lane == 0) bulk_wait_read_all();  // the previous chunk has left the buffer
      __syncwarp();
#pragma unroll 1
      for (int h = 0; h < 32; h += 16) {  // two 16-token halves of the chunk
        uint32_t v[16];
        tmem_ld_32x32b_x16(taddr + t0 + c0 + h, v);
        tmem_wait_ld();
        float acc[16];
#pragma unroll 1
        for (int r = 0; r < S; ++r) {
          if (r == rank) {
#pragma unroll
            for (int j = 0; j < 16; ++j)
              acc[j] = r == 0 ? __uint_as_float(v[j]) : __fadd_rn(acc[j], __uint_as_float(v[j]));
          } else {
            const int slot = r < rank ? r : r - 1;
            const float* src = reinterpret_cast<const float*>(smem + recv_off(slot, q) + lane * pitch * 4) + c0 + h;
#pragma unroll
            for (int j = 0; j < 16; j += 4) {
              const float4 f = *reinterpret_cast<const float4*>(src + j);
              acc[j] = r == 0 ? f.x : __fadd_rn(acc[j], f.x);
              acc[j + 1] = r == 0 ? f.y : __fadd_rn(acc[j + 1], f.y);
              acc[j + 2] = r == 0 ? f.z : __fadd_rn(acc[j + 2], f.z);
              acc[j + 3] = r == 0 ? f.w : __fadd_rn(acc[j + 3], f.w);
            }
          }
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) stg[(h + j) * 32 + lane] = to16<F16>(acc[j]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(tmap_out, stg_addr, static_cast<int32_t>(it.col0 + 32 * q),
                     static_cast<int32_t>(it.tok0 + t0 + c0));
        bulk_commit_group();
      }
    }
  }
}

// MULTI: a multi-product launch (tensor maps and statistics per product).
template <int MODE, int BT, int BITS, bool F16, bool MULTI = false>
__global__ void __launch_bounds__(kThreads, 1)
    nf4_gemm_kernel(const __grid_constant__ MapSet<MULTI ? kMaxProds : 1> tm, const GemmArgs a) {
  using G = Geo<BT, BITS>;
  static_assert(!MULTI || (BT <= 256 && BITS == 4), "multi-product launches: single-CTA tiles, 4-bit codes");
  const CUtensorMap& tmap_act = tm.act[0];
  const CUtensorMap& tmap_pk = tm.pk[0];
  const CUtensorMap& tmap_out = tm.out[0];
  constexpr int kPkStage = G::kPkStage;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  const uint32_t pad = (1024u - (raw_addr & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw_addr + pad;

  Shared sh;
  constexpr bool kPair = G::kPair;
  sh.rank = kPair ? cluster_ctarank() : 0u;
  // Work items are per CTA, or per CTA pair (both CTAs of a cluster walk the same
  // items).
  const int64_t unit = kPair ? blockIdx.x / 2 : blockIdx.x;
  const int64_t nunits = kPair ? gridDim.x / 2 : gridDim.x;
  sh.code4 = reinterpret_cast<float*>(smem + G::kOffMisc);
  sh.code8 = sh.code4 + 16;
  uint64_t* bars_ptr = reinterpret_cast<uint64_t*>(sh.code8 + 256);
  sh.bars = smem_addr(bars_ptr);
  sh.tmem_slot = reinterpret_cast<uint32_t*>(bars_ptr + kNumBars);
  sh.abort_flag = reinterpret_cast<volatile int*>(sh.tmem_slot + 1);
  int* item_count = reinterpret_cast<int*>(sh.tmem_slot + 2);
  sh.starts = reinterpret_cast<int*>(sh.tmem_slot + 4);
  sh.ends = sh.starts + (kMaxExperts + 1);
  sh.pref = sh.ends + (kMaxExperts + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---------------------------------------------------------------- prologue --
  // Local setup first (barriers, tensor memory, tensor-map prefetch): with
  // programmatic dependent launch it overlaps the previous kernel's tail.  Global
  // memory is touched only after the grid dependency has resolved -- except, for a
  // dense product whose weight the caller declared frozen (`early`), by the
  // weight-side roles: the code producer and the decoders then stream and decode
  // the first steps while the previous kernel drains, and only the activation
  // producer and the epilogue (the readers of activations, the writers of
  // outputs and partials) wait.
  const bool early = a.prefetch != 0 && !a.grouped;
  if (threadIdx.x == 0) {
    for (int i = 0; i < G::kStagesP; ++i) {
      mbar_init(bar_at(sh, kBarPFull + i), 1);
      mbar_init(bar_at(sh, kBarPEmpty + i), 4);  // the four warps of the owning group
    }
    for (int i = 0; i < G::kStagesX; ++i) {
      mbar_init(bar_at(sh, kBarXFull + i), 1);
      mbar_init(bar_at(sh, kBarXEmpty + i), 1);
    }
    // Pairs: the leader's full / accumulator-empty barriers also count the peer's
    // four decoder / epilogue warps (remote arrivals); the leader's MMA commits
    // arrive on the empty and accumulator-full barriers of both CTAs.
    for (int i = 0; i < G::kStagesA; ++i)
      mbar_init(bar_at(sh, kBarAFull + i), kPair ? 8 : 4);  // the decoder warps of the step's group
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_at(sh, kBarAccFull + i), 1);
      mbar_init(bar_at(sh, kBarAccEmpty + i), kPair ? 2 * kNumEpiWarps : kNumEpiWarps);
    }
    mbar_init(bar_at(sh, kBarDrain), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_at(sh, kBarEpFull + i), 1);
      mbar_init(bar_at(sh, kBarEpEmpty + i), 1);
    }
    for (int i = 0; i < kNumEpiWarps; ++i) mbar_init(bar_at(sh, kBarSkPart + i), 1);
    const int cs_peers = a.cs > 1 ? a.cs - 1 : 1;
    mbar_init(bar_at(sh, kBarCsFree), cs_peers);                  // one arrival per other rank
    mbar_init(bar_at(sh, kBarCsRecv), 1);  // this rank's expect-tx (the blocks complete it)
    *sh.abort_flag = 0;
    *dep_done(sh) = early ? 0 : 1;
    fence_mbar_init();
  }
  if (warp == kWarpTma && lane == 0)
    for (int p = 0; p < (MULTI ? a.nprod : 1); ++p) prefetch_tensormap(&tm.pk[p]);
  if (warp == kWarpTmaX && lane == 0)
    for (int p = 0; p < (MULTI ? a.nprod : 1); ++p) prefetch_tensormap(&tm.act[p]);
  if (warp == kWarpMma) {
    if (kPair) {
      tmem_alloc_pair(smem_addr(sh.tmem_slot), G::kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_addr(sh.tmem_slot), G::kTmemCols);
      tmem_relinquish();
    }
    tc_fence_before();
  }
  if (!early) grid_dependency_wait();
  allow_dependents();
  // The codebooks are loaded by the decoders alone (below), so the producers start
  // their first copies without waiting on those loads.
  if (a.grouped && threadIdx.x == kWarpEpi0 * 32) {
    // Per-expert token tiles and their prefix; offsets outside the contract are
    // reported and that expert is skipped.
    int acc = 0;
    bool bad = false;
    sh.pref[0] = 0;
    for (int e = 0; e < a.E; ++e) {
      const int s0 = a.offsets[e], s1 = a.offsets[e + 1];
      const bool ok = s0 >= 0 && s1 >= s0 && static_cast<int64_t>(s1) <= a.M;
      bad |= !ok;
      sh.starts[e] = ok ? s0 : 0;
      sh.ends[e] = ok ? s1 : 0;
      acc += ok ? (s1 - s0 + BT - 1) / BT : 0;
      sh.pref[e + 1] = acc;
    }
    *item_count = acc;
    if (bad) record_error(a, kStatusBadOffsets);
  }
  __syncthreads();
  if (a.cs > 1 || kPair) cluster_sync();  // every rank's barriers exist before any remote arrival
  tc_fence_after();
  const uint32_t tmem_base = *sh.tmem_slot;
  const int64_t total_items =
      a.grouped ? static_cast<int64_t>(*item_count) * a.wtiles : a.total_items;

  if (warp == kWarpTma || warp == kWarpTmaX) {
    // ----------------------------------------------------------- producers --
    // Warp 0 streams packed-code tiles (deep ring, far ahead of the decoders);
    // warp 18 streams activation tiles for the MMAs.
    if (early && warp == kWarpTmaX) {
      grid_dependency_wait();
      if (lane == 0) *dep_done(sh) = 1;
    }
    if (lane == 0) {
      const bool is_pk = warp == kWarpTma;
      const int nst = is_pk ? G::kStagesP : G::kStagesX;
      const int bar_full = is_pk ? kBarPFull : kBarXFull;
      const int bar_empty = is_pk ? kBarPEmpty : kBarXEmpty;
      const uint32_t bytes = is_pk ? kPkStage : G::kXStage;
      uint32_t st = 0, ph = 0, issued = 0, par = 0;
      bool ok = true;
      Cursor cur = cursor_begin<MULTI>(a, unit, total_items);
      Item it;
      while (ok && cursor_next<MODE, BT, MULTI>(cur, a, sh, nunits, it)) {
        for (int ks = it.ks0; ks < it.ks1; ++ks) {
          if (!wait_phase(bar_at(sh, bar_empty + st), ph ^ 1u, sh, a)) { ok = false; break; }
          const uint32_t full = bar_at(sh, bar_full + st);
          mbar_arrive_expect_tx(full, bytes);
          if (!is_pk) {
            // Pairs: this CTA's 128 tokens of each 256-token half of the tile.
#pragma unroll
            for (int h = 0; h < G::kXParts; ++h)
              tma_load_2d(sbase + G::kOffX + st * G::kXStage + h * (G::kXStage / G::kXParts), &tm.act[MULTI ? it.p : 0],
                          full, ks * kTileK,
                          static_cast<int32_t>(it.tok0 + (kPair ? 256 * h + 128 * static_cast<int>(sh.rank) : 0)));
          } else if (MODE == 0)
            tma_load_2d(sbase + G::kOffPk + st * kPkStage, &tm.pk[MULTI ? it.p : 0], full, ks * (kTileK * BITS / 8),
                        static_cast<int32_t>(it.wrow0));
          else
            tma_load_2d(sbase + G::kOffPk + st * kPkStage, &tm.pk[MULTI ? it.p : 0], full,
                        static_cast<int32_t>(it.col0 * BITS / 8),
                        static_cast<int32_t>(it.wrow0 + static_cast<int64_t>(ks) * kTileK));
          issued |= 1u << st;
          par = (par & ~(1u << st)) | (ph << st);
          if (++st == static_cast<uint32_t>(nst)) { st = 0; ph ^= 1u; }
        }
      }
      // Every load issued must have landed before the CTA may exit.
      for (int q = 0; q < nst; ++q)
        if (issued & (1u << q)) drain_phase(bar_at(sh, bar_full + q), (par >> q) & 1u, a);
    }
  } else if (warp == kWarpMma) {
    // ---------------------------------------------------------- MMA issuer --
    // Pairs: rank 0 issues the pair's MMAs (M = 256) and commits them to the
    // barriers of both CTAs; rank 1's issuer warp has nothing to do.
    if (lane == 0 && sh.rank == 0) {
      constexpr int kMmaM = kPair ? 2 * kTileW : kTileW;
      constexpr uint32_t idesc = F16 ? idesc_f16_f32(kMmaM, G::kMmaN, MODE == 1, false)
                                     : idesc_bf16_f32(kMmaM, G::kMmaN, MODE == 1, false);
      // Constant fields of the operand descriptors (address field zero).
      const uint64_t a_desc_hi = (MODE == 0) ? smem_desc_sw128(0, 16, 1024) : smem_desc_sw128(0, 8192, 1024);
      const uint64_t b_desc_hi = smem_desc_sw128(0, 16, 1024);
      // A commit that frees a slot: the barrier in this CTA, or in both CTAs of a pair.
      auto commit_both = [&](int bar) {
        if (kPair) {
          mma_commit_pair(mapa_shared(bar_at(sh, bar), 0u));
          mma_commit_pair(mapa_shared(bar_at(sh, bar), 1u));
        } else {
          mma_commit(bar_at(sh, bar));
        }
      };
      // Waits on barriers that remote arrivals complete (pairs) acquire at cluster scope.
      auto wait_in = [&](int bar, uint32_t parity) {
        return kPair ? wait_phase_cluster(bar_at(sh, bar), parity, sh, a) : wait_phase(bar_at(sh, bar), parity, sh, a);
      };
      uint32_t sx = 0, phx = 0, sa = 0, pha = 0;
      int acc_i = 0;
      bool ok = true;
      Cursor cur = cursor_begin<MULTI>(a, unit, total_items);
      Item it;
      for (; ok && cursor_next<MODE, BT, MULTI>(cur, a, sh, nunits, it); ++acc_i) {
        const int ab = acc_i % G::kAccBufs;
        const uint32_t acc_ph = (acc_i / G::kAccBufs) & 1;
        if (!wait_in(kBarAccEmpty + ab, acc_ph ^ 1u)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(ab * G::kAccCols);
        for (int ks = it.ks0; ks < it.ks1; ++ks) {
          // The decoders signal a stage only after its activation tile landed, so
          // one wait per step covers both operands (every barrier operation of this
          // thread is serialised with its MMA issue).
          if (!wait_in(kBarAFull + sa, pha)) { ok = false; break; }
          tc_fence_after();
          // Descriptors differ only in the start-address field (bits 0-13, address >> 4).
          // Only the CTA-local offset goes there: in a cluster launch the shared
          // addresses of ranks above 0 carry the rank in higher bits, which would
          // otherwise spill into the leading-byte-offset field (used by the
          // MN-major operand of the input gradient).
          const uint64_t adesc0 = a_desc_hi | (((sbase + G::kOffA + sa * kAStage) & 0x3FFFFu) >> 4);
#pragma unroll
          for (int h = 0; h < G::kXParts; ++h) {  // pairs: the tile's two 256-token halves
            const uint32_t xoff = G::kOffX + sx * G::kXStage + h * (G::kXStage / G::kXParts);
            const uint64_t bdesc0 = b_desc_hi | (((sbase + xoff) & 0x3FFFFu) >> 4);
#pragma unroll
            for (int kk = 0; kk < kTileK / 16; ++kk) {
              const uint64_t adesc = adesc0 + static_cast<uint64_t>(kk * (MODE == 0 ? 32 : 2048) >> 4);
              const uint64_t bdesc = bdesc0 + static_cast<uint64_t>(kk * 32 >> 4);
              const uint32_t acc = (ks > it.ks0 || kk > 0) ? 1u : 0u;
              if (kPair)
                mma_bf16_ss_pair(d_tmem + static_cast<uint32_t>(h * G::kMmaN), adesc, bdesc, idesc, acc);
              else
                mma_bf16_ss(d_tmem, adesc, bdesc, idesc, acc);
            }
          }
          // one "stage done" ring frees the activation and decoded slots
          commit_both(kBarXEmpty + sx);
          if (++sa == G::kStagesA) { sa = 0; pha ^= 1u; }
          if (++sx == G::kStagesX) { sx = 0; phx ^= 1u; }
        }
        if (!ok) break;
        commit_both(kBarAccFull + ab);
      }
      // All MMAs issued must be complete before tensor memory is released.
      if (kPair)
        mma_commit_pair(mapa_shared(bar_at(sh, kBarDrain), 0u));
      else
        mma_commit(bar_at(sh, kBarDrain));
      drain_phase(bar_at(sh, kBarDrain), 0, a);
    }
    __syncwarp();
  } else if (warp < kWarpDec0) {
    // ------------------------------------------------------------ epilogue --
    if (early) grid_dependency_wait();
    const int q = warp & 3;  // tensor-memory lane quarter this warp may access
    const int row = 32 * q + lane;
    int acc_i = 0;
    uint32_t xb = 0;    // SwiGLU exchange batches so far (barrier phases)
    bool ep_ok = true;  // false once an exchange wait gave up
    Cursor cur = cursor_begin<MULTI>(a, unit, total_items);
    Item it;
    for (; ep_ok && cursor_next<MODE, BT, MULTI>(cur, a, sh, nunits, it); ++acc_i) {
      const int ab = acc_i % G::kAccBufs;
      const uint32_t acc_ph = (acc_i / G::kAccBufs) & 1;
      if (kPair ? !wait_phase_cluster(bar_at(sh, kBarAccFull + ab), acc_ph, sh, a)
                : !wait_phase(bar_at(sh, kBarAccFull + ab), acc_ph, sh, a))
        break;
      tc_fence_after();
      const int64_t col = it.col0 + row;
      const bool col_ok = col < (MULTI ? a.prod[it.p].ncols : a.ncols);
      const int ntok = static_cast<int>(it.tok_end - it.tok0);  // tokens in this tile (<= BT)
      // Stream-K: a segment that stops before the tile's last step publishes its
      // fp32 partial (this warp's quarter of the rows, lane-contiguous per token) in
      // this CTA's slot; the segment holding the last steps of a tile cut between
      // CTAs (always the highest-index CTA on it) adds the partials of the lower
      // CTAs, from the nearest down, before rounding.  Waits only go to lower CTAs,
      // which are dispatched first, so the grid needs no co-residency.
      // (checked build: the CTAs whose partial slots and flags this one touches,
      // own_first .. unit with own_first >= 0, are CTAs of the launch)
      const bool sk_in = !a.sk || in_bounds(unit >= 0 && unit < a.sk_ctas, a.status);
      const bool sk_part = a.sk && sk_in && it.ks1 < a.ksteps;
      const bool sk_own = a.sk && sk_in && it.ks1 == a.ksteps && it.ks0 > 0;
      int64_t own_first = unit;  // lowest CTA holding steps of an owned split tile
      if (sk_own) {
        const int64_t tile0 = it.idx * a.ksteps;
        while (own_first > 0 && sk_first_unit(a, own_first) > tile0) --own_first;
        for (int64_t c = unit - 1; c >= own_first; --c)
          if (!flag_wait(a.sk_flags + c * 4 + q, a.sk_epoch ^ a.sk_wait_xor, sh, a)) break;
      }
      auto sk_slot = [&](int64_t c) {  // partial of CTA c, this quarter, token 0, this lane
        return a.sk_ws + ((c * 4 + q) * BT) * 32 + lane;
      };
      // The owned segment is the CTA's last item, so when its accumulator is full
      // the activation ring is idle (every tile loaded into it has been consumed by
      // the MMAs).  The previous CTA's partial of this warp's quarter (ntok x 128
      // bytes) then comes into the warp's part of that ring with one bulk copy, and
      // the chunks below read it from shared memory instead of waiting on L2 per
      // chunk; further CTAs' partials (tiles cut three or more ways) are read from
      // global memory.  The sum order is the same either way.
      const float* p_first = nullptr;  // partial of CTA unit - 1 in shared memory
      // (Stream-K does not run on CTA pairs, whose 512-token partials would not fit.)
      constexpr bool kPartFits = G::kStagesX * G::kXStage >= kNumEpiWarps * BT * 128;
      static_assert(kPartFits || kPair, "stream-K partials of the four row quarters fit in the activation ring");
      if (kPartFits && sk_own && own_first < unit &&
          (reinterpret_cast<uintptr_t>(a.sk_ws) & 15u) == 0) {
        float* land = reinterpret_cast<float*>(smem + G::kOffX) + q * (BT * 32);
        const uint32_t bar = bar_at(sh, kBarSkPart + q);
        if (lane == 0) {
          fence_proxy_async_global();  // the flag acquired above, then the async-proxy read
          mbar_arrive_expect_tx(bar, static_cast<uint32_t>(ntok) * 128u);
          bulk_load_g2s(smem_addr(land), sk_slot(unit - 1) - lane, static_cast<uint32_t>(ntok) * 128u, bar);
        }
        __syncwarp();
        // Completes once (the owned tile is the last item).  Waited for even after
        // another role gave up: the copy must land before the CTA may exit.
        drain_phase(bar, 0, a);
        p_first = land + lane;
      }
      auto part_src = [&](int64_t c, int c0) -> const float* {
        return (c == unit - 1 && p_first) ? p_first + c0 * 32 : sk_slot(c) + c0 * 32;
      };
      const uint32_t taddr =
          tmem_base + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(ab * G::kAccCols);
      // Tensor-memory loads are issued kWide columns (tokens) at a time with one wait:
      // the load latency, not the stores, bounds a narrow batch.
      constexpr int kBatch = 16;
      constexpr int kWide = BT < 32 ? BT : 32;
      auto load_wide = [&](int c0, uint32_t (&v)[kWide]) {
#pragma unroll
        for (int b = 0; b < kWide / 16; ++b)
          tmem_ld_32x32b_x16(taddr + c0 + 16 * b, *reinterpret_cast<uint32_t(*)[16]>(v + 16 * b));
        tmem_wait_ld();
      };
      // Adds the lower CTAs' partials (stream-K owner) to kWide tokens from c0.
      auto add_partials = [&](int c0, uint32_t (&v)[kWide]) {
        for (int64_t c = unit - 1; c >= own_first; --c)
#pragma unroll
          for (int sb = 0; sb < kWide; sb += 16) {
            const float* src = part_src(c, c0 + sb);
            float p[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) p[j] = src[j * 32];
#pragma unroll
            for (int j = 0; j < 16; ++j)
              v[sb + j] = __float_as_uint(__fadd_rn(__uint_as_float(v[sb + j]), p[j]));
          }
      };
      if (a.cs > 1) {
        cs_epilogue<BT, BITS, F16>(a, sh, smem, sbase, &tmap_out, it, taddr, q, ntok);
      } else if (sk_part) {
        float* dst = sk_slot(unit);
#pragma unroll 1
        for (int c0 = 0; c0 < ntok; c0 += kWide) {
          uint32_t v[kWide];
          load_wide(c0, v);
#pragma unroll
          for (int j = 0; j < kWide; ++j)
            if (c0 + j < ntok) dst[(c0 + j) * 32] = __uint_as_float(v[j]);
        }
        fence_proxy_async_global();  // the owner may read the partial with a bulk copy
        __threadfence();  // every lane's partial stores, then the quarter's flag
        __syncwarp();
        if (lane == 0) flag_publish(a.sk_flags + unit * 4 + q, a.sk_epoch);
      } else if (a.tma_out && a.splits == 1) {
        // bf16 tile through shared memory: per 32-token chunk this warp writes its
        // 32 columns x 32 tokens and one lane stores them with a bulk tensor copy
        // (rows past M and columns past the output width are not written).  A chunk
        // is one tensor-memory wait, and its partial loads (stream-K) are all in
        // flight together.
        uint16_t* stg = reinterpret_cast<uint16_t*>(smem + G::kOffOut + q * kOutWarpBytes);
        const uint32_t stg_addr = sbase + G::kOffOut + q * kOutWarpBytes;
        uint32_t v[32];
        auto load_chunk = [&](int c0) {
          tmem_ld_32x32b_x16(taddr + c0, *reinterpret_cast<uint32_t(*)[16]>(v));
          if (BT > 16) tmem_ld_32x32b_x16(taddr + c0 + 16, *reinterpret_cast<uint32_t(*)[16]>(v + 16));
        };
        load_chunk(0);
#pragma unroll 1
        for (int c0 = 0; c0 < ntok; c0 += 32) {
          tmem_wait_ld();
          if (sk_own)
            for (int64_t c = unit - 1; c >= own_first; --c) {
              const float* src = part_src(c, c0);
              float p[32];
#pragma unroll
              for (int j = 0; j < 32; ++j) p[j] = (BT > 16 || j < 16) ? src[j * 32] : 0.0f;
#pragma unroll
              for (int j = 0; j < 32; ++j)
                v[j] = __float_as_uint(__fadd_rn(__uint_as_float(v[j]), p[j]));
            }
          if (lane == 0) bulk_wait_read_all();  // the previous chunk has left the buffer
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (BT > 16 || j < 16)
              stg[j * 32 + lane] = to16<F16>(__uint_as_float(v[j]));
          // The next chunk's loads go out now, in flight during this chunk's store.
          if (c0 + 32 < ntok) load_chunk(c0 + 32);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tm.out[MULTI ? it.p : 0], stg_addr, static_cast<int32_t>(it.col0 + 32 * q),
                         static_cast<int32_t>(it.tok0 + c0));
            bulk_commit_group();
          }
        }
      } else if (MODE == 0 && a.ep_swiglu) {
        // Grouped SwiGLU: the tile's rows 0-63 are gate rows and rows 64-127 the up
        // rows of the same 64 output columns, held by other TMEM lane quarters, so the
        // up warp (quarter p + 2) passes each 16-token batch to the gate warp
        // (quarter p) through shared memory (32 rows x 16 fp32, conflict-free), with
        // a full / empty barrier pair per warp pair.  Biases are added to g and u
        // first.  Forward: h = silu(g) * u, times the row scale.  Backward (ep_bwd):
        // with d = dh * r, dg = d u silu'(g) and du = d silu(g) go to the gate and up
        // rows' columns, and the warp's 32 values of silu(g) u dh per token are summed
        // (fixed butterfly) into its routing-weight partial.
        const int p = q & 1;
        float* xch = reinterpret_cast<float*>(smem + G::kOffOut) + p * (32 * kBatch);
        const float bias = a.ep_bias ? __ldg(a.ep_bias + it.wrow0 + row) : 0.0f;
        const bool bwd = a.ep_bwd != 0;
        uint16_t* op = reinterpret_cast<uint16_t*>(a.out) + it.tok0 * a.ld_out +
                       (bwd ? it.col0 + row : it.col0 / 2 + row);
        const uint16_t* dhp = bwd ? reinterpret_cast<const uint16_t*>(a.ep_dh) + it.tok0 * a.ep_ld_dh +
                                        it.col0 / 2 + row
                                  : nullptr;
        float* drw = (bwd && a.ep_drw) ? a.ep_drw + ((it.col0 >> 7) * 2 + q) * a.M + it.tok0 : nullptr;
        // (checked build: the item's tokens and this lane's output columns inside
        // the output, and the routing-weight partial row inside its array)
        const bool gate_ok =
            q < 2 && it.col0 / 2 + row < a.ncols / 2 &&
            in_bounds(it.tok0 >= 0 && it.tok_end <= a.M &&
                          (bwd ? it.col0 + row + 64 < a.ld_out : it.col0 / 2 + row < a.ld_out) &&
                          (!drw || ((it.col0 >> 7) * 2 + q) * 64 < a.N_e),
                      a.status);
#pragma unroll 1
        for (int c0 = 0; c0 < ntok && ep_ok; c0 += kBatch, ++xb) {
          uint32_t v[kBatch];
          tmem_ld_32x32b_x16(taddr + c0, v);
          tmem_wait_ld();
          if (q >= 2) {  // up rows: hand the batch to the gate warp
            if (!wait_phase(bar_at(sh, kBarEpEmpty + p), (xb & 1u) ^ 1u, sh, a)) { ep_ok = false; break; }
#pragma unroll
            for (int j = 0; j < kBatch; ++j)
              xch[j * 32 + lane] = __fadd_rn(__uint_as_float(v[j]), bias);
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_at(sh, kBarEpFull + p));
          } else {
            if (!wait_phase(bar_at(sh, kBarEpFull + p), xb & 1u, sh, a)) { ep_ok = false; break; }
            const int nj = ntok - c0;
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
              const float g = __fadd_rn(__uint_as_float(v[j]), bias);
              const float u = xch[j * 32 + lane];
              const bool tok_ok = j < nj;
              const float r = (a.ep_scale && tok_ok) ? __ldg(a.ep_scale + it.tok0 + c0 + j) : 1.0f;
              if (!bwd) {
                float h = __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, expf(-g))), u);
                if (a.ep_scale) h = __fmul_rn(h, r);
                if (gate_ok && tok_ok) op[static_cast<int64_t>(c0 + j) * a.ld_out] = to16<F16>(h);
              } else {
                const int64_t tj = static_cast<int64_t>(c0 + j);
                const float dh = (gate_ok && tok_ok)
                                     ? __uint_as_float(static_cast<uint32_t>(dhp[tj * a.ep_ld_dh]) << 16)
                                     : 0.0f;
                const float sg = __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-g)));  // sigmoid(g)
                const float silu = __fmul_rn(g, sg);
                const float d = __fmul_rn(dh, r);
                // silu'(g) = s (1 + g (1 - s))
                const float dsilu = __fmul_rn(sg, __fadd_rn(1.0f, __fmul_rn(g, __fsub_rn(1.0f, sg))));
                const float dg = __fmul_rn(__fmul_rn(d, u), dsilu);
                const float du = __fmul_rn(d, silu);
                if (gate_ok && tok_ok) {
                  op[tj * a.ld_out] = to16<F16>(dg);
                  op[tj * a.ld_out + 64] = to16<F16>(du);
                }
                if (drw) {  // routing-weight partial over this warp's 32 gate columns
                  float t = __fmul_rn(__fmul_rn(silu, u), dh);
#pragma unroll
                  for (int o = 16; o > 0; o >>= 1) t = __fadd_rn(t, __shfl_xor_sync(0xffffffffu, t, o));
                  if (lane == 0 && tok_ok) drw[tj] = t;
                }
              }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_at(sh, kBarEpEmpty + p));
          }
        }
      } else {
        // Direct stores, one token row per element: y / gx in bf16, or this split's
        // fp32 partials.  Grouped forward epilogue: bias per weight row, scale per
        // output row.
        const int64_t ld_out = MULTI ? a.prod[it.p].ld_out : a.ld_out;
        uint16_t* op = reinterpret_cast<uint16_t*>(MULTI ? a.prod[it.p].out : a.out) + it.tok0 * ld_out + col;
        float* wp = a.ws + (static_cast<int64_t>(it.split) * a.M + it.tok0) * a.ncols + col;
        const float bias = MODE == 0 && a.ep_bias && col_ok ? __ldg(a.ep_bias + it.wrow0 + row) : 0.0f;
#pragma unroll 1
        for (int c0 = 0; c0 < ntok; c0 += kWide) {
          uint32_t v[kWide];
          load_wide(c0, v);
          if (sk_own) add_partials(c0, v);
          if (MODE == 0 && (a.ep_bias || a.ep_scale)) {
#pragma unroll
            for (int j = 0; j < kWide; ++j) {
              float f = __fadd_rn(__uint_as_float(v[j]), bias);
              if (a.ep_scale && c0 + j < ntok) f = __fmul_rn(f, __ldg(a.ep_scale + it.tok0 + c0 + j));
              v[j] = __float_as_uint(f);
            }
          }
          const int nj = ntok - c0;  // valid tokens in this batch when fewer than kWide
          const int64_t tok_hi = it.tok0 + c0 + (nj < kWide ? nj : kWide);  // one past the batch's last token
          if (col_ok && in_bounds(it.tok0 >= 0 && tok_hi <= a.M && col >= 0 &&
                                      (a.splits > 1 ? it.split < a.splits : col < ld_out),
                                  a.status)) {
            if (a.splits > 1) {
#pragma unroll
              for (int j = 0; j < kWide; ++j)
                if (j < nj) wp[static_cast<int64_t>(c0 + j) * a.ncols] = __uint_as_float(v[j]);
            } else {
#pragma unroll
              for (int j = 0; j < kWide; ++j)
                if (j < nj) op[static_cast<int64_t>(c0 + j) * ld_out] = to16<F16>(__uint_as_float(v[j]));
            }
          }
        }
      }
      if (sk_own) {  // the partials are consumed: clear their flags for the next launch
        __syncwarp();
        if (lane == 0)
          for (int64_t c = unit - 1; c >= own_first; --c) a.sk_flags[c * 4 + q] = 0ull;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {  // pairs: on the leader's barrier
        if (kPair && sh.rank != 0)
          mbar_arrive_cluster(mapa_shared(bar_at(sh, kBarAccEmpty + ab), 0u));
        else
          mbar_arrive(bar_at(sh, kBarAccEmpty + ab));
      }
    }
    // The output tiles' bulk stores have read their staging before the CTA exits (the
    // writes complete with the grid, before any dependent grid reads them).
    if (lane == 0) bulk_wait_read_all();
    __syncwarp();
  } else {
    // ------------------------------------------------------------ decoders --
    // kDecGroups groups of four warps: group g decodes the CTA's contraction steps
    // j = g, g + kDecGroups, g + 2 kDecGroups, ... (j counts the steps of the CTA's
    // items in order); each thread turns one whole 64-value block (one scale) into
    // bf16.  The ring slots of step j are j mod (ring depth), kept incrementally.
    const int dw = warp - kWarpDec0;
    const int grp = dw >> 2;
    const int rb = ((dw & 3) << 5) | lane;     // row-block 0..127
    const float offset = (a.dq && !MULTI) ? __ldg(a.nested_offset) : 0.0f;
    uint64_t code2[8];
    if (BITS == 4) {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        code2[i] = (static_cast<uint64_t>(__float_as_uint(__ldg(a.code4 + 2 * i + 1))) << 32) |
                   __float_as_uint(__ldg(a.code4 + 2 * i));
    }
    // The 8-bit map of the block statistics (and, for 8-bit codes, the 256-level
    // value codebook) go to shared memory for the random lookups; the decoder
    // warps alone synchronise on them (named barrier 1).
    float* valtab = reinterpret_cast<float*>(smem + G::kOffMisc + kMiscBase);
    const int dtid = dw * 32 + lane;
    if (a.dq && dtid < 256) sh.code8[dtid] = __ldg(a.code8 + dtid);
    // Multi-product launches: the products' nested offsets in shared memory (the
    // expert table's words, unused by these launches).
    float* offsets_s = reinterpret_cast<float*>(sh.starts);
    if (MULTI && a.dq && dtid < a.nprod) offsets_s[dtid] = __ldg(a.prod[dtid].nested_offset);
    if (BITS == 8)
      for (int i = dtid; i < 256 * 32; i += kNumDecWarps * 32) valtab[i] = __ldg(a.code4 + (i >> 5));
    const float* vt = valtab + lane;  // this lane's copy: entry e at vt[32 e]
    static_assert(kNumDecWarps * 32 >= 256, "one code8 entry per decoder thread");
    // Geometry of this thread's 128-byte line in the A tile and of its two 16-byte
    // chunks of packed codes.  The packed tile arrives with a TMA swizzle (32-byte
    // rows: 32B mode; 64-byte rows: 64B mode) so that a quarter-warp's chunk loads
    // fall in distinct banks.
    // 8-bit codes: 64-byte rows (64B swizzle) in the forward, 128-byte rows (128B
    // swizzle) in the input gradient; four 16-byte chunks per thread.
    int line_off, key, pk0, pk1, pkc[4];
    if (MODE == 0) {
      line_off = (rb >> 3) * 1024 + (rb & 7) * 128;
      key = rb & 7;
      const int x = (rb >> 2) & 1;  // 32B swizzle: chunk bit 0 ^= row bit 2
      pk0 = rb * 32 + ((0 ^ x) << 4);
      pk1 = rb * 32 + ((1 ^ x) << 4);
#pragma unroll
      for (int c = 0; c < 4; ++c) pkc[c] = rb * 64 + ((c ^ ((rb >> 1) & 3)) << 4);
    } else {
      const int nl = rb & 63, j = rb >> 6;
      line_off = j * 8192 + (nl >> 3) * 1024 + (nl & 7) * 128;
      key = nl & 7;
      const int x = (nl >> 1) & 3;  // 64B swizzle: chunk bits 0-1 ^= row bits 1-2
      pk0 = nl * 64 + (((2 * j) ^ x) << 4);
      pk1 = nl * 64 + (((2 * j + 1) ^ x) << 4);
#pragma unroll
      for (int c = 0; c < 4; ++c) pkc[c] = nl * 128 + (((4 * j + c) ^ (nl & 7)) << 4);
    }
    // Checked build: this thread's fixed offsets stay inside one decoded stage and
    // one code stage (a failing thread skips its loads and stores).
    const bool dec_in = in_bounds(
        line_off >= 0 && line_off + 128 <= kAStage &&
            (BITS == 4 ? (pk0 >= 0 && pk0 + 16 <= kPkStage && pk1 >= 0 && pk1 + 16 <= kPkStage)
                       : (pkc[0] >= 0 && pkc[0] + 16 <= kPkStage && pkc[1] >= 0 && pkc[1] + 16 <= kPkStage &&
                          pkc[2] >= 0 && pkc[2] + 16 <= kPkStage && pkc[3] >= 0 && pkc[3] + 16 <= kPkStage)),
        a.status);
    // The statistics of this group's steps are fetched kAhead owned steps ahead
    // into a register ring (global-memory latency hides behind the decodes in
    // between).  A walker over (item, step) supplies them; q == kNoStep marks the
    // end of the CTA's sequence.
    constexpr uint32_t kNoStep = 0xffffffffu;
    constexpr int kAhead = 3;
    Cursor fcur = cursor_begin<MULTI>(a, unit, total_items);
    Item fit{};
    bool fvalid = cursor_next<MODE, BT, MULTI>(fcur, a, sh, nunits, fit);
    int fks = fit.ks0;
    auto walk = [&](int n) {  // advance the walker n steps
      fks += n;
      while (fvalid && fks >= fit.ks1) {
        const int over = fks - fit.ks1;
        fvalid = cursor_next<MODE, BT, MULTI>(fcur, a, sh, nunits, fit);
        if (fvalid) fks = fit.ks0 + over;
      }
    };
    auto fetch_next = [&]() {
      RawScale r{0.0f, kNoStep};
      if (fvalid) {
        int64_t n, kb;
        if (MODE == 0) {
          n = fit.wrow0 + rb;
          kb = fks;
        } else {
          n = fit.wrow0 + static_cast<int64_t>(fks) * kTileK + (rb & 63);
          kb = (fit.col0 >> 6) + (rb >> 6);
        }
        r = fetch_scale<MULTI>(a, fit.p, n, kb);
        walk(kDecGroups);
      }
      return r;
    };
    walk(grp);
    RawScale ring[kAhead];
#pragma unroll
    for (int i = 0; i < kAhead; ++i) ring[i] = fetch_next();
    named_barrier_sync(1, kNumDecWarps * 32);  // code8 in shared memory
    uint32_t sp = grp, php = 0, sa = grp, pha = 0, sx = grp, phx = 0;
    // Decoded slot j mod kStagesA is free once the MMAs of step
    // m = j - kStagesA are done, which the "stage done" ring (depth kStagesX)
    // records in slot ms with phase parity mph.
    int m = grp - G::kStagesA;
    uint32_t ms = 0, mph = 0;
    while (ring[0].q != kNoStep) {
      const float s = finish_scale<MULTI>(a, sh.code8, ring[0], offset, offsets_s);
#pragma unroll
      for (int i = 0; i + 1 < kAhead; ++i) ring[i] = ring[i + 1];
      ring[kAhead - 1] = fetch_next();
      if (!wait_phase(bar_at(sh, kBarPFull + sp), php, sh, a)) break;
      if (!in_bounds(sp < static_cast<uint32_t>(G::kStagesP) && sa < static_cast<uint32_t>(G::kStagesA) &&
                         sx < static_cast<uint32_t>(G::kStagesX) && ms < static_cast<uint32_t>(G::kStagesX),
                     a.status))
        break;
      const uint8_t* pk = smem + G::kOffPk + sp * kPkStage;
      uint4 wc[4] = {};
      Lut L;
      if (BITS == 4) {
        if (dec_in) {
          wc[0] = *reinterpret_cast<const uint4*>(pk + pk0);
          wc[1] = *reinterpret_cast<const uint4*>(pk + pk1);
        }
        L = make_lut<F16>(code2, s);
      } else if (dec_in) {
#pragma unroll
        for (int c = 0; c < 4; ++c) wc[c] = *reinterpret_cast<const uint4*>(pk + pkc[c]);
      }
      if (m >= 0) {  // pairs: the leader's commit arrives from the other CTA
        if (kPair ? !wait_phase_cluster(bar_at(sh, kBarXEmpty + ms), mph, sh, a)
                  : !wait_phase(bar_at(sh, kBarXEmpty + ms), mph, sh, a))
          break;
      }
      uint8_t* A = smem + G::kOffA + sa * kAStage + line_off;
      if (!dec_in) {
        // (checked build: offsets outside the stage; nothing is written)
      } else if (BITS == 4) {
        const uint32_t wv[8] = {wc[0].x, wc[0].y, wc[0].z, wc[0].w, wc[1].x, wc[1].y, wc[1].z, wc[1].w};
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4*>(A + ((c ^ key) << 4)) = decode8(wv[c], L);
      } else {
        // One code per byte: value = bf16(fp32(code[q] * s)) from the shared table.
        const uint64_t s2 = (static_cast<uint64_t>(__float_as_uint(s)) << 32) | __float_as_uint(s);
#pragma unroll
        for (int c = 0; c < 8; ++c) {  // eight codes -> one 16-byte chunk of the A line
          const uint4 w = wc[c >> 1];
          const uint32_t lo = (c & 1) ? w.z : w.x, hi = (c & 1) ? w.w : w.y;
          uint32_t o[4];
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            const uint32_t word = p < 2 ? lo : hi;
            const int sft = (p & 1) * 16;
            const float f0 = vt[((word >> sft) & 0xffu) * 32];
            const float f1 = vt[((word >> (sft + 8)) & 0xffu) * 32];
            const uint64_t m = mul_f32x2(
                (static_cast<uint64_t>(__float_as_uint(f1)) << 32) | __float_as_uint(f0), s2);
            o[p] = pack16x2<F16>(__uint_as_float(static_cast<uint32_t>(m)),
                                 __uint_as_float(static_cast<uint32_t>(m >> 32)));
          }
          *reinterpret_cast<uint4*>(A + ((c ^ key) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
      // The stage's activation tile must have landed
      // before the MMA issuer is told the stage is ready; the decode above does not
      // need it, so it may run before the activations exist.
      if (!wait_phase(bar_at(sh, kBarXFull + sx), phx, sh, a)) break;
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar_at(sh, kBarPEmpty + sp));  // the codes were consumed above
        if (kPair && sh.rank != 0)  // pairs: the leader issues the MMAs
          mbar_arrive_cluster(mapa_shared(bar_at(sh, kBarAFull + sa), 0u));
        else
          mbar_arrive(bar_at(sh, kBarAFull + sa));
      }
      sp += kDecGroups;
      if (sp >= static_cast<uint32_t>(G::kStagesP)) { sp -= G::kStagesP; php ^= 1u; }
      sa += kDecGroups;
      if (sa >= static_cast<uint32_t>(G::kStagesA)) { sa -= G::kStagesA; pha ^= 1u; }
      sx += kDecGroups;
      if (sx >= static_cast<uint32_t>(G::kStagesX)) { sx -= G::kStagesX; phx ^= 1u; }
      m += kDecGroups;
      if (m >= kDecGroups) {
        ms += kDecGroups;
        if (ms >= static_cast<uint32_t>(G::kStagesX)) { ms -= G::kStagesX; mph ^= 1u; }
      } else if (m >= 0) {  // first step with a predecessor in this slot (m < kDecGroups <= kStagesX)
        ms = static_cast<uint32_t>(m);
        mph = 0;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  // A cluster leaves together: no rank exits while another may still write into its
  // shared memory or arrive on its barriers.
  if (a.cs > 1 || kPair) cluster_sync();
  if (warp == kWarpMma) {
    tc_fence_after();
    if (kPair)
      tmem_dealloc_pair(tmem_base, G::kTmemCols);
    else
      tmem_dealloc(tmem_base, G::kTmemCols);
  }
}

// out[t, c] = bf16 (fp16 when F16) of the sum over s in order of ws[s, t, c]; four
// columns per thread.  Used for few splits (the large-M contraction splits).
template <bool F16>
__global__ void __launch_bounds__(256) splitk_reduce_vec_kernel(const float* __restrict__ ws, int splits,
                                                                int64_t M, int64_t ncols,
                                                                uint16_t* __restrict__ out, int64_t ld) {
  grid_dependency_wait();
  allow_dependents();
  const int64_t total = M * ncols;
  const int64_t nq = (ncols + 3) / 4;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < M * nq;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = i / nq, c0 = (i - t * nq) * 4;
    const int64_t e = t * ncols + c0;
    if (c0 + 4 <= ncols && (ncols & 3) == 0 && (ld & 3) == 0) {
      float4 acc = *reinterpret_cast<const float4*>(ws + e);
      for (int s = 1; s < splits; ++s) {
        const float4 v = *reinterpret_cast<const float4*>(ws + static_cast<int64_t>(s) * total + e);
        acc.x = __fadd_rn(acc.x, v.x);
        acc.y = __fadd_rn(acc.y, v.y);
        acc.z = __fadd_rn(acc.z, v.z);
        acc.w = __fadd_rn(acc.w, v.w);
      }
      uint2 pk;
      pk.x = pack16x2<F16>(acc.x, acc.y);
      pk.y = pack16x2<F16>(acc.z, acc.w);
      *reinterpret_cast<uint2*>(out + t * ld + c0) = pk;
    } else {
      for (int64_t c = c0; c < c0 + 4 && c < ncols; ++c) {
        float acc = ws[t * ncols + c];
        for (int s = 1; s < splits; ++s) acc = __fadd_rn(acc, ws[static_cast<int64_t>(s) * total + t * ncols + c]);
        out[t * ld + c] = to16<F16>(acc);
      }
    }
  }
}

// out[t, c] = bf16 (fp16 when F16) of the sum over s of ws[s, t, c] in a fixed
// order: a CTA owns 32 consecutive elements of one row; its 8 thread groups sum the
// splits g, g+8, g+16, ... sequentially, then the 8 group sums are added in group
// order.
template <bool F16>
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const float* __restrict__ ws, int splits,
                                                            int64_t M, int64_t ncols,
                                                            uint16_t* __restrict__ out, int64_t ld) {
  __shared__ float part[8][32];
  grid_dependency_wait();
  allow_dependents();
  const int64_t total = M * ncols;
  const int64_t slices = (ncols + 31) / 32;
  const int c = threadIdx.x & 31, g = threadIdx.x >> 5;
  for (int64_t blk = blockIdx.x; blk < M * slices; blk += gridDim.x) {
    const int64_t t = blk / slices;
    const int64_t col = (blk - t * slices) * 32 + c;
    float v = 0.0f;
    if (col < ncols) {
      const float* p = ws + t * ncols + col;
      if (g < splits) v = p[static_cast<int64_t>(g) * total];
      for (int s = g + 8; s < splits; s += 8) v = __fadd_rn(v, p[static_cast<int64_t>(s) * total]);
    }
    part[g][c] = v;
    __syncthreads();
    if (g == 0 && col < ncols) {
      float acc = part[0][c];
      for (int q = 1; q < 8 && q < splits; ++q) acc = __fadd_rn(acc, part[q][c]);
      out[t * ld + col] = to16<F16>(acc);
    }
    __syncthreads();
  }
}

#if NF4_GEMM_MAIN_TU
// out[t] = sum over p in order of part[p * T + t] for rows inside the expert ranges
// (offsets[0] <= t < offsets[E]), 0 elsewhere: the routing-weight gradient of the
// SwiGLU backward from its per-32-column partials.
__global__ void __launch_bounds__(256) row_partial_sum_kernel(const float* __restrict__ part, int P,
                                                              int64_t T, const int32_t* __restrict__ offsets,
                                                              int E, float* __restrict__ out) {
  grid_dependency_wait();
  allow_dependents();
  const int64_t lo = offsets[0], hi = offsets[E];
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < T;
       t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float acc = 0.0f;
    if (t >= lo && t < hi)
      for (int p = 0; p < P; ++p) acc = (p == 0) ? part[t] : __fadd_rn(acc, part[static_cast<int64_t>(p) * T + t]);
    out[t] = acc;
  }
}
#endif

template <int MODE, int BT, int BITS, bool F16>
cudaError_t launch_one(const GemmArgs& a, const CUtensorMap& ta, const CUtensorMap& tp,
                       const CUtensorMap& to, int grid,
                       cudaStream_t s) {
  static bool configured = false;
  auto kern = nf4_gemm_kernel<MODE, BT, BITS, F16>;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Geo<BT, BITS>::kSmem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = Geo<BT, BITS>::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  // Clusters: a cluster split (one tile per cluster of cs CTAs) or a CTA pair.
  const unsigned cluster = Geo<BT, BITS>::kPair ? 2u : (a.cs > 1 ? static_cast<unsigned>(a.cs) : 1u);
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = cluster > 1 ? 2 : 1;
  MapSet<1> maps;
  maps.act[0] = ta;
  maps.pk[0] = tp;
  maps.out[0] = to;
  return cudaLaunchKernelEx(&cfg, kern, maps, a);
}

#if NF4_GEMM_MAIN_TU
// A multi-product launch (classic schedule, no clusters).
template <int MODE, int BT>
cudaError_t launch_multi_one(const GemmArgs& a, const MapSet<kMaxProds>& maps, int grid, cudaStream_t s) {
  static bool configured = false;
  auto kern = nf4_gemm_kernel<MODE, BT, 4, false, true>;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Geo<BT, 4>::kSmem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = Geo<BT, 4>::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, maps, a);
}
#endif

template <int MODE>
cudaError_t launch_mode(int bt, const GemmArgs& a, const CUtensorMap& ta, const CUtensorMap& tp,
                        const CUtensorMap& to, int grid, cudaStream_t s) {
#if NF4_GEMM_MAIN_TU
  switch (bt) {
    case 16: return launch_one<MODE, 16, 4, false>(a, ta, tp, to, grid, s);
    case 32: return launch_one<MODE, 32, 4, false>(a, ta, tp, to, grid, s);
    case 64: return launch_one<MODE, 64, 4, false>(a, ta, tp, to, grid, s);
    case 128: return launch_one<MODE, 128, 4, false>(a, ta, tp, to, grid, s);
    case 256: return launch_one<MODE, 256, 4, false>(a, ta, tp, to, grid, s);
    case 512: return launch_one<MODE, 512, 4, false>(a, ta, tp, to, grid, s);
    default: return cudaErrorInvalidValue;
  }
#elif NF4_GEMM_F16
  switch (bt) {
    case 16: return launch_one<MODE, 16, 4, true>(a, ta, tp, to, grid, s);
    case 32: return launch_one<MODE, 32, 4, true>(a, ta, tp, to, grid, s);
    case 64: return launch_one<MODE, 64, 4, true>(a, ta, tp, to, grid, s);
    case 128: return launch_one<MODE, 128, 4, true>(a, ta, tp, to, grid, s);
    case 256: return launch_one<MODE, 256, 4, true>(a, ta, tp, to, grid, s);
    case 512: return launch_one<MODE, 512, 4, true>(a, ta, tp, to, grid, s);
    default: return cudaErrorInvalidValue;
  }
#else
  switch (bt) {
    case 16: return launch_one<MODE, 16, 8, false>(a, ta, tp, to, grid, s);
    case 32: return launch_one<MODE, 32, 8, false>(a, ta, tp, to, grid, s);
    case 64: return launch_one<MODE, 64, 8, false>(a, ta, tp, to, grid, s);
    case 128: return launch_one<MODE, 128, 8, false>(a, ta, tp, to, grid, s);
    default: return cudaErrorInvalidValue;
  }
#endif
}

}  // namespace

#if NF4_GEMM_F16
// The fp16-operand instances (this file compiled again, from nf4_gemm_f16.cu).
cudaError_t launch_gemm_f16(int mode, int bt, const GemmArgs& a, const CUtensorMap& tmap_act,
                            const CUtensorMap& tmap_packed, const CUtensorMap& tmap_out, int grid,
                            cudaStream_t s) {
  if (mode == 0) return launch_mode<0>(bt, a, tmap_act, tmap_packed, tmap_out, grid, s);
  return launch_mode<1>(bt, a, tmap_act, tmap_packed, tmap_out, grid, s);
}
#elif NF4_GEMM_BITS == 8
// The 8-bit-code instances (this file compiled a second time, from nf4_gemm8.cu).
cudaError_t launch_gemm_8bit(int mode, int bt, const GemmArgs& a, const CUtensorMap& tmap_act,
                             const CUtensorMap& tmap_packed, const CUtensorMap& tmap_out, int grid,
                             cudaStream_t s) {
  if (mode == 0) return launch_mode<0>(bt, a, tmap_act, tmap_packed, tmap_out, grid, s);
  return launch_mode<1>(bt, a, tmap_act, tmap_packed, tmap_out, grid, s);
}
#else

size_t gemm_exchange_bytes(int bt, int bits) {
  switch (bits == 8 ? bt + 1 : bt) {
    case 16: return size_t(Geo<16, 4>::kOffOut);
    case 32: return size_t(Geo<32, 4>::kOffOut);
    case 64: return size_t(Geo<64, 4>::kOffOut);
    case 128: return size_t(Geo<128, 4>::kOffOut);
    case 256: return size_t(Geo<256, 4>::kOffOut);
    case 17: return size_t(Geo<16, 8>::kOffOut);
    case 33: return size_t(Geo<32, 8>::kOffOut);
    case 65: return size_t(Geo<64, 8>::kOffOut);
    case 129: return size_t(Geo<128, 8>::kOffOut);
    default: return 0;
  }
}

template <int MODE, int BT>
int cluster_capacity_bt(int cs) {
  auto kern = nf4_gemm_kernel<MODE, BT, 4, false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Geo<BT, 4>::kSmem) !=
      cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(cs), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = Geo<BT, 4>::kSmem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cs);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

int gemm_cluster_capacity(int mode, int bt, int cs) {
  struct Entry {
    int dev, mode, bt, cs, n;
  };
  static std::mutex mu;
  static Entry cache[64];
  static int used = 0;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  std::lock_guard<std::mutex> lk(mu);
  for (int i = 0; i < used; ++i)
    if (cache[i].dev == dev && cache[i].mode == mode && cache[i].bt == bt && cache[i].cs == cs)
      return cache[i].n;
  int n = 0;
  switch (bt) {
    case 64: n = mode == 0 ? cluster_capacity_bt<0, 64>(cs) : cluster_capacity_bt<1, 64>(cs); break;
    case 128: n = mode == 0 ? cluster_capacity_bt<0, 128>(cs) : cluster_capacity_bt<1, 128>(cs); break;
    case 256: n = mode == 0 ? cluster_capacity_bt<0, 256>(cs) : cluster_capacity_bt<1, 256>(cs); break;
    case 512: n = mode == 0 ? cluster_capacity_bt<0, 512>(cs) : cluster_capacity_bt<1, 512>(cs); break;
    default: n = 0;
  }
  if (used < 64) cache[used++] = Entry{dev, mode, bt, cs, n};
  return n;
}

cudaError_t launch_gemm_multi(int mode, int bt, const GemmArgs& a, const MapSet<kMaxProds>& maps, int grid,
                              cudaStream_t s) {
  if (a.nprod < 1 || a.nprod > kMaxProds || a.sk || a.cs > 1 || a.splits != 1 || a.grouped)
    return cudaErrorInvalidValue;
  switch (mode * 1000 + bt) {
    case 128: return launch_multi_one<0, 128>(a, maps, grid, s);
    case 256: return launch_multi_one<0, 256>(a, maps, grid, s);
    case 1128: return launch_multi_one<1, 128>(a, maps, grid, s);
    case 1256: return launch_multi_one<1, 256>(a, maps, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_gemm(int mode, int bt, int bits, bool f16, const GemmArgs& a,
                        const CUtensorMap& tmap_act, const CUtensorMap& tmap_packed,
                        const CUtensorMap& tmap_out, int grid, cudaStream_t s) {
  if (f16) {
    if (bits != 4) return cudaErrorInvalidValue;
    return launch_gemm_f16(mode, bt, a, tmap_act, tmap_packed, tmap_out, grid, s);
  }
  if (bits == 8) return launch_gemm_8bit(mode, bt, a, tmap_act, tmap_packed, tmap_out, grid, s);
  if (mode == 0) return launch_mode<0>(bt, a, tmap_act, tmap_packed, tmap_out, grid, s);
  return launch_mode<1>(bt, a, tmap_act, tmap_packed, tmap_out, grid, s);
}

cudaError_t launch_row_partial_sum(const float* part, int P, int64_t T, const int32_t* offsets,
                                   int E, float* out, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  int64_t grid = (T + 255) / 256;
  if (grid > 4096) grid = 4096;
  if (grid < 1) grid = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, row_partial_sum_kernel, part, P, T, offsets, E, out);
}

cudaError_t launch_splitk_reduce(const float* ws, int splits, int64_t M, int64_t ncols,
                                 void* out_, int64_t ld, bool f16, cudaStream_t s) {
  uint16_t* out = static_cast<uint16_t*>(out_);
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (splits <= 8) {
    int64_t grid = (M * ((ncols + 3) / 4) + 255) / 256;
    if (grid > 8192) grid = 8192;
    if (grid < 1) grid = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    return f16 ? cudaLaunchKernelEx(&cfg, splitk_reduce_vec_kernel<true>, ws, splits, M, ncols, out, ld)
               : cudaLaunchKernelEx(&cfg, splitk_reduce_vec_kernel<false>, ws, splits, M, ncols, out, ld);
  }
  // Many splits (the small-M input gradient): one CTA per 32 outputs.
  int64_t grid = M * ((ncols + 31) / 32);
  if (grid > 16384) grid = 16384;
  if (grid < 1) grid = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  return f16 ? cudaLaunchKernelEx(&cfg, splitk_reduce_kernel<true>, ws, splits, M, ncols, out, ld)
             : cudaLaunchKernelEx(&cfg, splitk_reduce_kernel<false>, ws, splits, M, ncols, out, ld);
}

#endif  // NF4_GEMM_BITS

}  // namespace nf4
