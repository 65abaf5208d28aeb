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
// Structure (one CTA per SM, persistent over work items):
//   warp 0      TMA producer: activation tile [BT tokens x 64] (128B swizzle) and
//               packed-code tile into a ring of kStagesT stages;
//   warps 6-13  decoders: each pair of threads turns one 64-value block (one
//               absmax) into bf16 and stores it in the UMMA canonical 128B-swizzled
//               layout of the A operand (K-major for the forward, MN-major for the
//               input gradient), ring of kStagesA stages;
//   warp 1      MMA issuer: tcgen05.mma M=128 (weight rows / in-features), N=BT
//               (tokens), K=16, fp32 accumulators in tensor memory, two
//               accumulator buffers so the epilogue overlaps the next item;
//   warps 2-5   epilogue: tcgen05.ld of the accumulator, bf16 rounding, store.
// Every output element is produced by exactly one CTA with a fixed order of MMAs;
// when the contraction is split (small M only) the fp32 partials go to a
// workspace and a second kernel adds them in split order.  No atomics anywhere.
// Every wait is bounded; on timeout the kernel records the error and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "sm100_ptx.cuh"

namespace nf4 {
namespace {

using namespace nf4ptx;

constexpr int kThreads = 14 * 32;
constexpr int kWarpTma = 0;
constexpr int kWarpMma = 1;
constexpr int kWarpEpi0 = 2;
constexpr int kNumEpiWarps = 4;
constexpr int kWarpDec0 = 6;
constexpr int kNumDecWarps = 8;
constexpr int kAStage = kTileW * kTileK * 2;  // 16 KB of bf16
constexpr int kPkStage = kTileW * kTileK / 2;  // 4 KB of packed codes
constexpr int kStagesA = 4;
constexpr int kMiscBytes = 8192;
constexpr uint64_t kTimeoutNs = 2000000000ull;

template <int BT>
struct Geo {
  static constexpr int kXStage = BT * 128;  // BT rows of 64 bf16
  static constexpr int kBudget = 225 * 1024 - kStagesA * kAStage - kMiscBytes - 1024;
  static constexpr int kStagesT0 = kBudget / (kXStage + kPkStage);
  static constexpr int kStagesT = kStagesT0 > 16 ? 16 : kStagesT0;
  static constexpr int kOffA = 0;
  static constexpr int kOffX = kOffA + kStagesA * kAStage;
  static constexpr int kOffPk = kOffX + kStagesT * kXStage;
  static constexpr int kOffMisc = kOffPk + kStagesT * kPkStage;
  static constexpr int kSmem = kOffMisc + kMiscBytes + 1024;
  static constexpr uint32_t kTmemCols = (2 * BT < 32) ? 32u : static_cast<uint32_t>(2 * BT);
  static_assert(kStagesT >= 2, "pipeline too shallow");
  static_assert(kXStage % 1024 == 0, "activation stage must keep 1024-byte alignment");
};

// Barrier slots in the misc region.
constexpr int kBarTmaFull = 0;
constexpr int kBarTmaEmpty = 16;
constexpr int kBarAFull = 32;
constexpr int kBarAEmpty = 36;
constexpr int kBarAccFull = 40;
constexpr int kBarAccEmpty = 42;
constexpr int kBarDrain = 44;
constexpr int kNumBars = 45;

struct Item {
  int64_t tok0, tok_end;
  int64_t wrow0;  // forward: first weight row of the tile; input gradient: first row of the expert
  int64_t col0;   // first output column of the tile
  int ks0, ks1;
  int split;
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
};

__device__ __forceinline__ uint32_t bar_at(const Shared& sh, int i) { return sh.bars + 8u * i; }

__device__ __forceinline__ void record_error(const GemmArgs& a, int code) {
  *reinterpret_cast<volatile int*>(a.status) = code;
}

// Bounded wait: true once the phase completed; false on abort (another role
// gave up) or after kTimeoutNs, in which case the timeout is recorded.
__device__ __noinline__ bool wait_phase(uint32_t bar, uint32_t parity, const Shared& sh,
                                        const GemmArgs& a) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*sh.abort_flag) return false;
    if (globaltimer_ns() - t0 > kTimeoutNs) {
      *sh.abort_flag = 1;
      record_error(a, kStatusTimeout);
      return false;
    }
  }
}

// Wait used while draining on exit: bounded, ignores the abort flag.
__device__ __noinline__ void drain_phase(uint32_t bar, uint32_t parity, const GemmArgs& a) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kTimeoutNs) {
      record_error(a, kStatusTimeout);
      return;
    }
  }
}

template <int MODE, int BT>
__device__ __forceinline__ Item get_item(int64_t idx, const GemmArgs& a, const Shared& sh) {
  Item it;
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
    it.col0 = wt * kTileW;
    it.wrow0 = (MODE == 0) ? wt * kTileW : 0;
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
    it.wrow0 = (MODE == 0) ? static_cast<int64_t>(e) * a.N_e + wt * kTileW
                           : static_cast<int64_t>(e) * a.N_e;
  }
  return it;
}

// Decoded block scale: absmax, or fp32(fp32(code8[q] * nested) + offset).
__device__ __forceinline__ float load_scale(const GemmArgs& a, const float* code8_s, int64_t n,
                                            int64_t kb, float offset) {
  if (n >= a.N_total || kb >= a.KB) return 0.0f;
  const int64_t b = n * a.KB + kb;
  if (!a.dq) return __ldg(a.absmax + b);
  const float t = __fmul_rn(code8_s[__ldg(a.absmax_q + b)], __ldg(a.nested_absmax + (b >> 8)));
  return __fadd_rn(t, offset);
}

// Eight packed codes (one 32-bit word; byte j holds value 2j high, 2j+1 low) to
// eight bf16 values bf16(fp32(code4[q] * s)), packed pairwise, value 0 lowest.
__device__ __forceinline__ uint4 decode8(uint32_t w, const float* code4_s, float s) {
  uint32_t o[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t byte = (w >> (8 * j)) & 0xFFu;
    const float f0 = __fmul_rn(code4_s[byte >> 4], s);
    const float f1 = __fmul_rn(code4_s[byte & 15u], s);
    __nv_bfloat162 p = __floats2bfloat162_rn(f0, f1);
    o[j] = *reinterpret_cast<uint32_t*>(&p);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

template <int MODE, int BT>
__global__ void __launch_bounds__(kThreads, 1)
    nf4_gemm_kernel(const __grid_constant__ CUtensorMap tmap_act,
                    const __grid_constant__ CUtensorMap tmap_pk, const GemmArgs a) {
  using G = Geo<BT>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  const uint32_t pad = (1024u - (raw_addr & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw_addr + pad;

  Shared sh;
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
  if (threadIdx.x < 16) sh.code4[threadIdx.x] = a.code4[threadIdx.x];
  if (a.dq)
    for (int j = threadIdx.x; j < 256; j += kThreads) sh.code8[j] = a.code8[j];
  if (threadIdx.x == 0) {
    for (int i = 0; i < G::kStagesT; ++i) {
      mbar_init(bar_at(sh, kBarTmaFull + i), 1);
      mbar_init(bar_at(sh, kBarTmaEmpty + i), 1);
    }
    for (int i = 0; i < kStagesA; ++i) {
      mbar_init(bar_at(sh, kBarAFull + i), kNumDecWarps);
      mbar_init(bar_at(sh, kBarAEmpty + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_at(sh, kBarAccFull + i), 1);
      mbar_init(bar_at(sh, kBarAccEmpty + i), kNumEpiWarps);
    }
    mbar_init(bar_at(sh, kBarDrain), 1);
    *sh.abort_flag = 0;
    fence_mbar_init();
  }
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
  if (warp == kWarpTma && lane == 0) {
    prefetch_tensormap(&tmap_act);
    prefetch_tensormap(&tmap_pk);
  }
  if (warp == kWarpMma) {
    tmem_alloc(smem_addr(sh.tmem_slot), G::kTmemCols);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *sh.tmem_slot;
  const int64_t total_items =
      a.grouped ? static_cast<int64_t>(*item_count) * a.wtiles : a.total_items;

  if (warp == kWarpTma) {
    // ------------------------------------------------------------ producer --
    if (lane == 0) {
      uint32_t st = 0, ph = 0, issued = 0, par = 0;
      bool ok = true;
      for (int64_t idx = blockIdx.x; ok && idx < total_items; idx += gridDim.x) {
        const Item it = get_item<MODE, BT>(idx, a, sh);
        for (int ks = it.ks0; ks < it.ks1; ++ks) {
          if (!wait_phase(bar_at(sh, kBarTmaEmpty + st), ph ^ 1u, sh, a)) { ok = false; break; }
          const uint32_t full = bar_at(sh, kBarTmaFull + st);
          mbar_arrive_expect_tx(full, G::kXStage + kPkStage);
          tma_load_2d(sbase + G::kOffX + st * G::kXStage, &tmap_act, full, ks * kTileK,
                      static_cast<int32_t>(it.tok0));
          if (MODE == 0)
            tma_load_2d(sbase + G::kOffPk + st * kPkStage, &tmap_pk, full, ks * (kTileK / 2),
                        static_cast<int32_t>(it.wrow0));
          else
            tma_load_2d(sbase + G::kOffPk + st * kPkStage, &tmap_pk, full,
                        static_cast<int32_t>(it.col0 / 2),
                        static_cast<int32_t>(it.wrow0 + static_cast<int64_t>(ks) * kTileK));
          issued |= 1u << st;
          par = (par & ~(1u << st)) | (ph << st);
          if (++st == G::kStagesT) { st = 0; ph ^= 1u; }
        }
      }
      // Every load issued must have landed before the CTA may exit.
      for (int s = 0; s < G::kStagesT; ++s)
        if (issued & (1u << s)) drain_phase(bar_at(sh, kBarTmaFull + s), (par >> s) & 1u, a);
    }
  } else if (warp == kWarpMma) {
    // ---------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kTileW, BT, MODE == 1, false);
      uint32_t st = 0, ph = 0, sa = 0, pha = 0;
      int acc_i = 0;
      bool ok = true;
      for (int64_t idx = blockIdx.x; ok && idx < total_items; idx += gridDim.x, ++acc_i) {
        const Item it = get_item<MODE, BT>(idx, a, sh);
        const int ab = acc_i & 1;
        const uint32_t acc_ph = (acc_i >> 1) & 1;
        if (!wait_phase(bar_at(sh, kBarAccEmpty + ab), acc_ph ^ 1u, sh, a)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(ab * BT);
        for (int ks = it.ks0; ks < it.ks1; ++ks) {
          if (!wait_phase(bar_at(sh, kBarTmaFull + st), ph, sh, a)) { ok = false; break; }
          if (!wait_phase(bar_at(sh, kBarAFull + sa), pha, sh, a)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a_base = sbase + G::kOffA + sa * kAStage;
          const uint32_t b_base = sbase + G::kOffX + st * G::kXStage;
#pragma unroll
          for (int kk = 0; kk < kTileK / 16; ++kk) {
            const uint64_t adesc = (MODE == 0) ? smem_desc_sw128(a_base + kk * 32, 16, 1024)
                                               : smem_desc_sw128(a_base + kk * 2048, 8192, 1024);
            const uint64_t bdesc = smem_desc_sw128(b_base + kk * 32, 16, 1024);
            mma_bf16_ss(d_tmem, adesc, bdesc, idesc, (ks > it.ks0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(bar_at(sh, kBarTmaEmpty + st));
          mma_commit(bar_at(sh, kBarAEmpty + sa));
          if (++st == G::kStagesT) { st = 0; ph ^= 1u; }
          if (++sa == kStagesA) { sa = 0; pha ^= 1u; }
        }
        if (!ok) break;
        mma_commit(bar_at(sh, kBarAccFull + ab));
      }
      // All MMAs issued must be complete before tensor memory is released.
      mma_commit(bar_at(sh, kBarDrain));
      drain_phase(bar_at(sh, kBarDrain), 0, a);
    }
    __syncwarp();
  } else if (warp < kWarpDec0) {
    // ------------------------------------------------------------ epilogue --
    const int q = warp & 3;  // tensor-memory lane quarter this warp may access
    const int row = 32 * q + lane;
    int acc_i = 0;
    for (int64_t idx = blockIdx.x; idx < total_items; idx += gridDim.x, ++acc_i) {
      const Item it = get_item<MODE, BT>(idx, a, sh);
      const int ab = acc_i & 1;
      const uint32_t acc_ph = (acc_i >> 1) & 1;
      if (!wait_phase(bar_at(sh, kBarAccFull + ab), acc_ph, sh, a)) break;
      tc_fence_after();
      const int64_t col = it.col0 + row;
      const bool col_ok = col < a.ncols;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(ab * BT);
#pragma unroll 1
      for (int c0 = 0; c0 < BT; c0 += 16) {
        uint32_t v[16];
        tmem_ld_32x32b_x16(taddr + c0, v);
        tmem_wait_ld();
        if (col_ok) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int64_t tok = it.tok0 + c0 + j;
            if (tok < it.tok_end) {
              const float f = __uint_as_float(v[j]);
              if (a.splits > 1)
                a.ws[(static_cast<int64_t>(it.split) * a.M + tok) * a.ncols + col] = f;
              else
                a.out[tok * a.ld_out + col] = __float2bfloat16_rn(f);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_at(sh, kBarAccEmpty + ab));
    }
  } else {
    // ------------------------------------------------------------ decoders --
    const int d = threadIdx.x - kWarpDec0 * 32;  // 0..255
    const int rb = d >> 1;                       // row-block 0..127
    const int h = d & 1;                         // which 32 values of the block
    const float offset = a.dq ? __ldg(a.nested_offset) : 0.0f;
    // Geometry of this thread's 128-byte line in the A tile and in the packed tile.
    int line_off, key, pk_off;
    if (MODE == 0) {
      line_off = (rb >> 3) * 1024 + (rb & 7) * 128;
      key = rb & 7;
      pk_off = rb * 32 + h * 16;
    } else {
      const int nl = rb & 63, j = rb >> 6;
      line_off = j * 8192 + (nl >> 3) * 1024 + (nl & 7) * 128;
      key = nl & 7;
      pk_off = nl * 64 + j * 32 + h * 16;
    }
    uint32_t st = 0, ph = 0, sa = 0, pha = 0;
    bool ok = true;
    for (int64_t idx = blockIdx.x; ok && idx < total_items; idx += gridDim.x) {
      const Item it = get_item<MODE, BT>(idx, a, sh);
      for (int ks = it.ks0; ks < it.ks1; ++ks) {
        int64_t n, kb;
        if (MODE == 0) {
          n = it.wrow0 + rb;
          kb = ks;
        } else {
          n = it.wrow0 + static_cast<int64_t>(ks) * kTileK + (rb & 63);
          kb = (it.col0 >> 6) + (rb >> 6);
        }
        const float s = load_scale(a, sh.code8, n, kb, offset);
        if (!wait_phase(bar_at(sh, kBarTmaFull + st), ph, sh, a)) { ok = false; break; }
        if (!wait_phase(bar_at(sh, kBarAEmpty + sa), pha ^ 1u, sh, a)) { ok = false; break; }
        const uint4 w4 = *reinterpret_cast<const uint4*>(smem + G::kOffPk + st * kPkStage + pk_off);
        uint8_t* A = smem + G::kOffA + sa * kAStage + line_off;
        const uint32_t wv[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int c = 4 * h + i;
          *reinterpret_cast<uint4*>(A + ((c ^ key) << 4)) = decode8(wv[i], sh.code4, s);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_at(sh, kBarAFull + sa));
        if (++st == G::kStagesT) { st = 0; ph ^= 1u; }
        if (++sa == kStagesA) { sa = 0; pha ^= 1u; }
      }
    }
  }

  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem_base, G::kTmemCols);
  }
}

// out[t, c] = bf16(sum over s in order of ws[s, t, c]).
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const float* __restrict__ ws, int splits,
                                                            int64_t M, int64_t ncols,
                                                            __nv_bfloat16* __restrict__ out, int64_t ld) {
  const int64_t total = M * ncols;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = i / ncols, c = i - t * ncols;
    float acc = ws[i];
    for (int s = 1; s < splits; ++s) acc = __fadd_rn(acc, ws[static_cast<int64_t>(s) * total + i]);
    out[t * ld + c] = __float2bfloat16_rn(acc);
  }
}

template <int MODE, int BT>
cudaError_t launch_one(const GemmArgs& a, const CUtensorMap& ta, const CUtensorMap& tp, int grid,
                       cudaStream_t s) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(nf4_gemm_kernel<MODE, BT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, Geo<BT>::kSmem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  nf4_gemm_kernel<MODE, BT><<<grid, kThreads, Geo<BT>::kSmem, s>>>(ta, tp, a);
  return cudaGetLastError();
}

template <int MODE>
cudaError_t launch_mode(int bt, const GemmArgs& a, const CUtensorMap& ta, const CUtensorMap& tp,
                        int grid, cudaStream_t s) {
  switch (bt) {
    case 16: return launch_one<MODE, 16>(a, ta, tp, grid, s);
    case 32: return launch_one<MODE, 32>(a, ta, tp, grid, s);
    case 64: return launch_one<MODE, 64>(a, ta, tp, grid, s);
    case 128: return launch_one<MODE, 128>(a, ta, tp, grid, s);
    case 256: return launch_one<MODE, 256>(a, ta, tp, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

int gemm_smem_bytes(int bt) {
  switch (bt) {
    case 16: return Geo<16>::kSmem;
    case 32: return Geo<32>::kSmem;
    case 64: return Geo<64>::kSmem;
    case 128: return Geo<128>::kSmem;
    case 256: return Geo<256>::kSmem;
    default: return -1;
  }
}

cudaError_t launch_gemm(int mode, int bt, const GemmArgs& a, const CUtensorMap& tmap_act,
                        const CUtensorMap& tmap_packed, int grid, cudaStream_t s) {
  if (mode == 0) return launch_mode<0>(bt, a, tmap_act, tmap_packed, grid, s);
  return launch_mode<1>(bt, a, tmap_act, tmap_packed, grid, s);
}

cudaError_t launch_splitk_reduce(const float* ws, int splits, int64_t M, int64_t ncols,
                                 __nv_bfloat16* out, int64_t ld, cudaStream_t s) {
  const int64_t total = M * ncols;
  int64_t grid = (total + 255) / 256;
  if (grid > 4096) grid = 4096;
  if (grid < 1) grid = 1;
  splitk_reduce_kernel<<<static_cast<unsigned>(grid), 256, 0, s>>>(ws, splits, M, ncols, out, ld);
  return cudaGetLastError();
}

}  // namespace nf4
