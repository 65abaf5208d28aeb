// nf4_skinny.cu -- small-M tensor-core path of the fused NF4 products: a few
// activation rows (M <= 16) against a packed NF4 weight, where the work is bound
// by streaming the packed codes from HBM (Soup issue #842, "Design sketch":
// forward and transposed backward computed straight from the packed codes,
// deterministic reduction, no atomics).
//
// Decode.  Every CTA holds in shared memory a 256-entry table that maps one
// byte made of two 4-bit codes to the fp32 pair (code4[high nibble],
// code4[low nibble]), one copy per lane so that the 32 lookups of a warp touch
// 32 different 8-byte slots.  A lookup is one byte permute (which also forms the
// address), one 8-byte shared load, one paired fp32 multiply by the values'
// block scales and one bf16x2 conversion per two weight values, and yields
// exactly the dequantised operand bf16(fp32(code4[q] * scale)) in a register of
// the warp-level bf16 MMA (mma.sync.m16n8k16, fp32 accumulation), which does the
// multiply-adds for up to 16 activation rows.  The work is spread over the
// shared-memory, fp32 and integer pipes (a register-resident codebook would load
// the integer pipe alone, which on this GPU issues at half rate).
//
// Work split.  The grid is C clusters of S CTAs (one CTA of 16 warps per SM).
// Cluster c owns a contiguous range of output tiles, balanced to within one
// tile; CTA rank r owns one slice of the contraction.  The (tile, contraction
// step) units of a CTA are dealt to its 16 warps as contiguous ranges, and each
// warp streams its units' packed codes through its own two-slot ring of
// shared-memory slots: one tensor (TMA) tile copy per unit, issued by lane 0 and
// completing on the slot's barrier, one unit ahead of the one it decodes (the
// copy engine keeps the slices of all 16 warps in flight at once, which 16-byte
// copies from every lane could not).  The tile copies write the codes in the
// swizzled layouts the decode reads conflict-free (128B swizzle for the forward's
// 128-byte rows, 32B swizzle for the input gradient's 32-byte rows).  The forward decodes each unit's block scales per lane
// from statistics fetched along with the unit's codes and stages its
// activation slice in shared memory once; the input gradient decodes the block
// scales of its slice once into shared memory and carries grad_y in the ring
// slots next to the codes.  Every sum runs in a fixed order:
// inside an MMA, over a warp's units in order, over the warps of a CTA in warp
// order through shared memory, and over the cluster's ranks in rank order
// through distributed shared memory.  No atomics, no workspace.
//
// Launched with programmatic stream serialisation: a kernel may start while its
// predecessor on the stream drains and waits for it (griddepcontrol.wait)
// before it reads activations or writes the output.  When the caller declares
// the weight read-only for the duration (`prefetch`), the codebook table, the
// block scales and the first units' packed codes are read before that wait.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <vector>

#include "internal.h"
#include "sm100_ptx.cuh"

namespace nf4 {
namespace {

using nf4ptx::cluster_sync;
using nf4ptx::mapa_shared;
using nf4ptx::smem_addr;

// Bounded wait (2 s) for the phase of `parity` of a ring barrier; false after
// recording NF4_ERR_TIMEOUT in the status word.
__device__ __noinline__ bool ring_wait_slow(uint32_t bar, uint32_t parity, int* status) {
  const uint64_t t0 = nf4ptx::globaltimer_ns();
  while (!nf4ptx::mbar_try_wait(bar, parity)) {
    if (nf4ptx::globaltimer_ns() - t0 > 2000000000ull) {
      if (status) *reinterpret_cast<volatile int*>(status) = kStatusTimeout;
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ bool ring_wait(uint32_t bar, uint32_t parity, int* status) {
  if (nf4ptx::mbar_test_wait(bar, parity)) return true;
  return ring_wait_slow(bar, parity, status);
}

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kTableBytes = 256 * 256;    // 256 entries x 32 lanes x 8 bytes
constexpr size_t kMaxSmem = 227 * 1024;

__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void allow_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// d += a * b: one warp-level 16x8x16 bf16 (or fp16 when F16) product, fp32
// accumulation.
template <bool F16>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  if constexpr (F16)
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  else
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// One output value: bf16, or IEEE fp16 when F16 (round to nearest even).
template <bool F16>
__device__ __forceinline__ void store16(__nv_bfloat16* p, float v) {
  if constexpr (F16)
    *reinterpret_cast<__half*>(p) = __float2half_rn(v);
  else
    *p = __float2bfloat16_rn(v);
}

// The byte-pair table: entry e = (code4[e >> 4], code4[e & 15]) as two fp32 (the
// even value of a packed byte first), copy for lane l at byte offset 256 e + 8 l.
// Written as 8 rounds of one 16-byte store per thread (16-byte unit
// i = 512 k + thread, entry i / 16, so a warp's stores are contiguous).  The
// codebook values a thread needs are loaded first (table_src), so that their round
// trip overlaps the kernel's other first loads, and stored later (store_table).
struct TableSrc {
  uint32_t lo;      // low code of the thread's entries (fixed per thread)
  uint32_t hi[8];   // high code of entry 32 k + thread / 16 in round k
};

__device__ __forceinline__ TableSrc table_src(const float* code4) {
  static_assert(kThreads == 512, "the table is 8 rounds of 512 16-byte units");
  const int tid = static_cast<int>(threadIdx.x);
  const int odd = (tid >> 8) & 1;  // unit 512 k + tid holds entry 32 k + tid / 16
  TableSrc t;
  t.lo = __float_as_uint(__ldg(code4 + ((tid >> 4) & 15)));
#pragma unroll
  for (int k = 0; k < 8; ++k) t.hi[k] = __float_as_uint(__ldg(code4 + 2 * k + odd));  // code 2 k + tid / 256
  return t;
}

__device__ __forceinline__ void store_table(uint8_t* smem, const TableSrc& src) {
  uint4* t = reinterpret_cast<uint4*>(smem);
  const int tid = static_cast<int>(threadIdx.x);
#pragma unroll
  for (int k = 0; k < 8; ++k) t[k * kThreads + tid] = make_uint4(src.hi[k], src.lo, src.hi[k], src.lo);
}

// Dequantised pair of the packed byte that `sel` picks from w: bf16(fp32(code4[q]
// * s)) (fp16 when F16) for both nibbles, the even value in the low half.
// The permute puts the byte into bits 8..15 and lane*8 (byte 0 of lane8) into
// bits 0..7 of the table offset; s2 holds the two values' scales (low word:
// even value).
template <bool F16>
__device__ __forceinline__ uint32_t lookup(const uint8_t* smem, uint32_t w, uint32_t lane8,
                                           uint32_t sel, uint64_t s2) {
  const uint2 c = *reinterpret_cast<const uint2*>(smem + __byte_perm(w, lane8, sel));
  uint64_t p;
  asm("mul.rn.f32x2 %0, %1, %2;"
      : "=l"(p)
      : "l"((static_cast<uint64_t>(c.y) << 32) | c.x), "l"(s2));
  const float lo = __uint_as_float(static_cast<uint32_t>(p));
  const float hi = __uint_as_float(static_cast<uint32_t>(p >> 32));
  if constexpr (F16) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
  } else {
    const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&b);
  }
}

__device__ __forceinline__ uint64_t pair2(float lo, float hi) {
  return (static_cast<uint64_t>(__float_as_uint(hi)) << 32) | __float_as_uint(lo);
}

// Selector for byte b of the first operand (see lookup).
__host__ __device__ constexpr uint32_t lookup_sel(uint32_t b) { return 0x5504u | (b << 4); }

// Raw statistics of one block (absmax, or 8-bit code + nested absmax), fetched
// ahead; finished into the decoded scale when the block is used.  The loads are
// unconditional (a block that does not exist reads block 0 and is marked invalid)
// so that nothing merges their values at fetch time: the thread runs on until the
// values are used.
struct Raw {
  float v;
  uint32_t q;
  bool ok;
};

__device__ __forceinline__ Raw fetch_raw(const SkinnyArgs& a, int64_t b, bool valid) {
  Raw r;
  // (checked build: a valid block lies inside the statistics arrays)
  if (valid && !in_bounds(b >= 0 && b < a.N * a.KB, a.status)) valid = false;
  const int64_t bi = valid ? b : 0;
  r.ok = valid;
  if (!a.dq) {
    r.v = __ldg(a.absmax + bi);
    r.q = 0u;
  } else {
    r.q = __ldg(a.absmax_q + bi);
    r.v = __ldg(a.nested_absmax + (bi >> 8));
  }
  return r;
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint4 lds128(const void* p) {
  return *reinterpret_cast<const uint4*>(p);
}

// A unit's packed codes in a ring slot: 16 rows x 32 bytes, the 16-byte half h
// of row r at 16-byte unit 2r + (h ^ ((r >> 2) & 1)); the swizzle keeps the
// forward's 16-byte and the input gradient's 4-byte reads free of bank
// conflicts.
__device__ __forceinline__ int code_unit(int r, int h) { return 2 * r + (h ^ ((r >> 2) & 1)); }

// Decoded block scales of `count` blocks into sc[0 .. count): block `block_of(idx)`
// (-1 for none: scale 0), four blocks per thread per batch (idx = i0 + j kThreads).
// A batch's statistics are fetched together (fetch_scales), then decoded with the
// 8-bit codebook staged in shared memory (`code8s`, 256 floats; finish_scales), so
// the first batch can be fetched along with the kernel's other first loads.
struct ScaleBatch {
  Raw r[4];
};

template <typename BlockOf>
__device__ __forceinline__ ScaleBatch fetch_scales(const SkinnyArgs& a, int i0, int count,
                                                   BlockOf block_of) {
  ScaleBatch s;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int idx = i0 + j * kThreads;
    const int64_t b = idx < count ? block_of(idx) : -1;
    s.r[j] = fetch_raw(a, b, b >= 0);
  }
  return s;
}

__device__ __forceinline__ void finish_scales(const SkinnyArgs& a, float* sc, const float* code8s,
                                              float offset, int i0, int count, const ScaleBatch& s) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int idx = i0 + j * kThreads;
    if (idx >= count) break;
    float v = 0.0f;
    if (s.r[j].ok) v = a.dq ? __fadd_rn(__fmul_rn(code8s[s.r[j].q], s.r[j].v), offset) : s.r[j].v;
    sc[idx] = v;
  }
}

// Warp w's contiguous range [lo, hi) of a CTA's U units; per_tile units make
// one output tile.  A range touches at most two tiles (the plan ensures it).
struct WarpRange {
  int lo, hi, t0;
};

__device__ __forceinline__ WarpRange warp_range(int w, int U, int per_tile) {
  WarpRange r;
  r.lo = (w * U) >> 4;
  r.hi = ((w + 1) * U) >> 4;
  r.t0 = r.lo < r.hi ? r.lo / per_tile : 0;
  return r;
}

// Element e of tile i summed over the warps of the CTA, in warp order.  Warp w
// keeps its last tile's partial at last + w * last_stride and, when its range
// started in the tile below its last one, that first tile's partial at
// first + w * first_stride.  The warps touching tile i are those whose unit
// range [w U / 16, (w + 1) U / 16) meets [i per_tile, (i + 1) per_tile); all
// sixteen candidates' loads go out before the adds (shifts and compares only, no
// division), and the adds run in warp order.
__device__ __forceinline__ float cta_sum(int i, int e, int U, int per_tile, const float* first,
                                         int first_stride, const float* last, int last_stride) {
  static_assert(kWarps == 16, "warp ranges use w * U / 16");
  const int a0 = i * per_tile, a1 = a0 + per_tile;
  float p[kWarps];
  bool use[kWarps];
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const int lo = (w * U) >> 4, hi = ((w + 1) * U) >> 4;
    use[w] = lo < hi && lo < a1 && hi > a0;
    p[w] = use[w] ? (hi <= a1 ? last[w * last_stride + e] : first[w * first_stride + e]) : 0.0f;
  }
  float v = 0.0f;
#pragma unroll
  for (int w = 0; w < kWarps; ++w)
    if (use[w]) v = __fadd_rn(v, p[w]);
  return v;
}

__device__ __forceinline__ void st_dsmem(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// Cluster reduction: the `total` elements are cut into S chunks of
// len = ceil(total / S); rank r owns chunk r.  Every rank stores its CTA sum of
// element e into the owner's receive buffer (row = the sending rank), then one
// cluster barrier, then the owner adds the S rows in rank order.
struct ClusterShare {
  int e0, e1, len;  // this rank's elements [e0, e1); row length of the receive buffer
};

__device__ __forceinline__ ClusterShare cluster_share(int rank, int S, int total) {
  ClusterShare c;
  c.len = (total + S - 1) / S;
  c.e0 = rank * c.len < total ? rank * c.len : total;
  c.e1 = c.e0 + c.len < total ? c.e0 + c.len : total;
  return c;
}

__device__ __forceinline__ void cluster_push(float* recv, int rank, int S, int total, int e,
                                             float v) {
  const int len = (total + S - 1) / S;
  const int owner = e / len;
  const int local = e - owner * len;
  st_dsmem(mapa_shared(smem_addr(recv + rank * len + local), static_cast<uint32_t>(owner)), v);
}

template <typename Store>
__device__ __forceinline__ void cluster_finish(const float* recv, int rank, int S, int total,
                                               Store store) {
  cluster_sync();
  const ClusterShare c = cluster_share(rank, S, total);
  for (int e = c.e0 + static_cast<int>(threadIdx.x); e < c.e1; e += kThreads) {
    float v = 0.0f;
    for (int q = 0; q < S; ++q) v = __fadd_rn(v, recv[q * c.len + (e - c.e0)]);
    store(e, v);
  }
}

constexpr int kFwdQuad = 4;      // 64-value blocks per forward unit (256 values per row)
constexpr int kFwdUnit = 2048;   // bytes of a forward unit: 16 rows x 128
constexpr int kFwdDepth = 2;     // ring slots per warp (forward)
constexpr int kBwdDepth = 2;     // ring slots per warp (input gradient)
constexpr int kBwdRows = 64;     // weight rows per input-gradient unit

// Input-gradient ring slots: 64 rows x 32 bytes of codes (a whole number of
// 256-byte swizzle atoms) in one ring, the unit's grad_y (padded rows per token)
// in a second ring.
constexpr int kBwdCodeUnit = kBwdRows * 32;
__host__ __device__ constexpr int bwd_gy_unit_bytes(int mt) { return mt * 8 * (kBwdRows * 2 + 16); }

// Shared-memory layout of a CTA (byte offsets), common to the plan and the kernels.
using Layout = SkinnyLayout;

__host__ __device__ inline Layout make_layout(int mode, int mt, int S, int64_t cc, int64_t nt_max) {
  Layout L;
  const int slot_elems = mode == 0 ? mt * 8 * 16 : mt * 8 * 64;
  const int unit = mode == 0 ? kFwdUnit : kBwdCodeUnit;
  const int depth = mode == 0 ? kFwdDepth : kBwdDepth;
  L.table = 0;
  L.ring = kTableBytes;
  L.gy = L.ring + kWarps * depth * unit;
  L.first = L.gy + (mode == 0 ? 0 : kWarps * depth * bwd_gy_unit_bytes(mt));
  L.recv = L.first + kWarps * slot_elems * 4;
  const int64_t total = nt_max * slot_elems;
  const int64_t len = (total + S - 1) / S;
  L.scales = L.recv + static_cast<int>((S > 1 ? S * len * 4 : 0) + 15) / 16 * 16;
  // input gradient: the decoded block scales of the CTA's slice (forward: none)
  const int64_t nscales = mode == 0 ? 0 : nt_max * cc;
  L.code8 = L.scales + static_cast<int>((nscales * 4 + 15) / 16 * 16);
  // Forward: one ring barrier per warp and slot here.  The input gradient keeps its
  // two per warp in the unused padding of its first grad_y row (bytes 128-143).
  L.bars = L.code8 + 256 * 4;
  L.act = L.bars + (mode == 0 ? kWarps * kFwdDepth * 8 : 0);
  const int64_t nch = (cc / 64 + kFwdQuad - 1) / kFwdQuad * kFwdQuad;  // forward: chunks of 64
  L.total = mode == 0 ? L.act + static_cast<int>(mt * 8 * nch * 128) : L.act;
  return L;
}

// ---------------------------------------------------------------- forward --
//
// Tile = 16 weight rows; a unit = one tile x four 64-value blocks (256 values
// per row).  Lane (g, t4) holds rows g and g+8 of the tile and block t4 of the
// unit: 64 values per row, one block scale per row.  MMA j (0..15) of a
// unit gives contraction slots (2t4, 2t4+1) the values 4j, 4j+1 of block t4 and
// slots (2t4+8, 2t4+9) the values 4j+2, 4j+3, for A (the weight) and B (the
// activations) alike; the sum over the 16 slots is the same whatever order the
// values take.  A unit's codes (16 rows x 128 bytes) land in a ring slot with
// the 16-byte chunk c of row r at chunk c ^ (r & 7), which makes the lanes'
// 16-byte reads conflict-free.  The activation slice of the CTA's contraction
// sits in shared memory as 64-value chunks per token whose eight 16-byte units
// are XOR-swizzled by (chunk & 3) | (token & 1) << 2, so the eight lanes of a
// quarter warp (two tokens, four chunks, one unit index) hit different banks.
template <int MT, bool F16>  // 8-token MMA tiles: 1 (M <= 8) or 2 (M <= 16); fp16 operands
__global__ void __launch_bounds__(kThreads, 1)
    skinny_fwd_kernel(const __grid_constant__ CUtensorMap tmap, const SkinnyArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  // The tile copies' swizzle follows absolute shared-memory address bits: the
  // ring must start on a 1024-byte boundary (it does, after the 64 KB table, when
  // the dynamic shared memory does).
  if ((smem_addr(smem) & 1023u) != 0) {
    if (threadIdx.x == 0 && a.status) *reinterpret_cast<volatile int*>(a.status) = NF4_ERR_UNSUPPORTED;
    return;
  }
  constexpr int D = kFwdDepth;
  static_assert(D == 2, "the statistics rotate through two register sets");
  constexpr int kSlotElems = MT * 8 * 16;  // [token][row], a power of two
  constexpr int kSlotShift = MT == 1 ? 7 : 8;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int S = a.S;
  const int rank = static_cast<int>(blockIdx.x) & (S - 1);
  const int cl = static_cast<int>(blockIdx.x) >> a.log2S;
  // cl * T / C and (cl + 1) * T / C from T = tq C + tr (32-bit divisions only)
  const int64_t tile0 = cl * a.tq + (cl * a.tr) / a.C;
  const int nt = static_cast<int>((cl + 1) * a.tq + ((cl + 1) * a.tr) / a.C - tile0);
  const int64_t nt_max = a.nt_max;
  const int nbs = static_cast<int>(a.cc >> 6);  // blocks per contraction slice
  const int64_t kb0 = static_cast<int64_t>(rank) * nbs;
  const int nbr = static_cast<int>(a.KB - kb0 < nbs ? a.KB - kb0 : nbs);  // >= 1 by the plan
  const int nq = (nbr + kFwdQuad - 1) / kFwdQuad;  // units per tile
  const int nch = (nbs + kFwdQuad - 1) / kFwdQuad * kFwdQuad;
  const int U = nt * nq;
  const WarpRange mine = warp_range(warp, U, nq);
  const int nunits = mine.hi - mine.lo;
  const Layout L = a.lay;
  uint8_t* ring = smem + L.ring + warp * D * kFwdUnit;
  float* first = reinterpret_cast<float*>(smem + L.first);
  float* recv = reinterpret_cast<float*>(smem + L.recv);
  float* code8s = reinterpret_cast<float*>(smem + L.code8);
  uint4* xs = reinterpret_cast<uint4*>(smem + L.act);           // [token][chunk][8 units]
  // The warp's ring barriers (one per slot), initialised by its lane 0.
  const uint32_t bars_s = smem_addr(smem + L.bars) + warp * D * 8;
  if (lane == 0) {
    for (int j = 0; j < D; ++j) nf4ptx::mbar_init(bars_s + 8 * j, 1);
    nf4ptx::fence_mbar_init();
  }
  __syncwarp();

  // Copies: lane 0 issues one tile copy of a unit's 16 rows x 128 bytes (rows
  // past N and bytes past the row read as zeros); (ii, iq) = (tile, block quad) of
  // the next unit to copy.  The same call fetches, per lane, the statistics of the
  // lane's two blocks (rows g and g+8, block t4).
  const uint32_t ring_s = smem_addr(ring);
  int issued = 0, ii = mine.t0, iq = mine.lo - mine.t0 * nq;
  struct Stats {
    Raw a, b;
  };
  auto fetch = [&](int64_t n, int64_t kb, bool ok) -> Raw { return fetch_raw(a, n * a.KB + kb, ok); };
  auto issue = [&]() -> Stats {
    Stats st{Raw{0.0f, 0u, false}, Raw{0.0f, 0u, false}};
    if (issued < nunits) {
      const int slot = issued & (D - 1);
      const int64_t n16 = (tile0 + ii) * 16;
      const int64_t kbq = kb0 + kFwdQuad * iq;
      // Blocks of the quad past this rank's slice come in too; their scales (and
      // activations) are zero, so they add nothing.
      if (lane == 0) {
        const uint32_t bar = bars_s + 8 * slot;
        nf4ptx::mbar_arrive_expect_tx(bar, kFwdUnit);
        nf4ptx::tma_load_2d(ring_s + slot * kFwdUnit, &tmap, bar, static_cast<int32_t>(kbq * 32),
                            static_cast<int32_t>(n16));
      }
      const bool bok = kFwdQuad * iq + t4 < nbr;
      st.a = fetch(n16 + g, kbq + t4, bok && n16 + g < a.N);
      st.b = fetch(n16 + g + 8, kbq + t4, bok && n16 + g + 8 < a.N);
      if (++iq == nq) {
        iq = 0;
        ++ii;
      }
    }
    ++issued;
    return st;
  };
  // The first loads all go out together, so that the kernel start costs about one
  // memory round trip: the first two units' tile copies and statistics, the
  // codebook values of the byte-pair table, the 8-bit codebook entry and the nested
  // offset (the weight side, read before the grid dependency resolves when the
  // weight is declared frozen), then the activation slice; the table and codebook
  // stores wait for their values after that.
  Stats s0, s1;  // statistics of the units in ring slots (q and q+1)
  TableSrc tsrc;
  float c8, offset;  // 8-bit codebook entry, nested offset (double quantisation)
  auto weight_side = [&]() {
    s0 = issue();
    s1 = issue();
    tsrc = table_src(a.code4);
    // unconditional loads from valid addresses (used only under double quantisation)
    c8 = __ldg(a.dq ? a.code8 + (threadIdx.x & 255) : a.code4);
    offset = __ldg(a.dq ? a.nested_offset : a.code4);
  };

  // One call site for the weight side (the dependency wait goes before or after
  // it), so that no branch merge makes the thread wait for the loaded values here.
  if (!a.prefetch) grid_dependency_wait();
  weight_side();
  if (a.prefetch) grid_dependency_wait();
  {  // activation slice -> shared memory (asynchronous copies): tokens < M, zero beyond the slice
    const int units = nch * 8;  // 16-byte units per token
    const uint32_t xs_s = smem_addr(xs);
    for (int tok = 0; tok < a.M; ++tok) {
      const __nv_bfloat16* xrow = a.act + tok * a.ld_act + kb0 * 64;
      for (int e = threadIdx.x; e < units; e += kThreads) {
        const int c = e >> 3, q = e & 7;
        const int slot = ((tok * nch + c) << 3) + (q ^ ((c & 3) | ((tok & 1) << 2)));
        cp_async16(xs_s + slot * 16, c < nbr ? xrow + 8 * e : a.act, c < nbr);
      }
    }
    cp_async_commit();
  }
  allow_dependents();
  store_table(smem, tsrc);
  static_assert(kThreads >= 256, "one 8-bit codebook entry per thread");
  if (a.dq && threadIdx.x < 256) code8s[threadIdx.x] = c8;
  cp_async_wait<0>();
  __syncthreads();

  const uint32_t lane8 = static_cast<uint32_t>(lane) << 3;
  constexpr uint32_t kSel0 = lookup_sel(0), kSel1 = lookup_sel(1), kSel2 = lookup_sel(2),
                     kSel3 = lookup_sel(3);
  const int f = t4 | ((g & 1) << 2);  // activation swizzle of this lane's chunks
  const int sw = g & 7;               // ring swizzle of rows g and g+8
  auto scale = [&](const Raw& r) -> float {
    if (!a.dq) return r.ok ? r.v : 0.0f;
    return r.ok ? __fadd_rn(__fmul_rn(code8s[r.q], r.v), offset) : 0.0f;
  };
  float acc[MT][4];
#pragma unroll
  for (int t = 0; t < MT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.0f;
  int ctile = mine.t0;
  int ci = mine.t0, cq = mine.lo - mine.t0 * nq;  // (tile, block quad) being decoded

  auto store_acc = [&](float* p) {
#pragma unroll
    for (int t = 0; t < MT; ++t) {
      const int tok = 8 * t + 2 * t4;
      p[tok * 16 + g] = acc[t][0];
      p[(tok + 1) * 16 + g] = acc[t][1];
      p[tok * 16 + g + 8] = acc[t][2];
      p[(tok + 1) * 16 + g + 8] = acc[t][3];
      acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.0f;
    }
  };

  int q = 0;
  for (; q < nunits; ++q) {
    if (!ring_wait(bars_s + 8 * (q & (D - 1)), static_cast<uint32_t>(q / D) & 1u, a.status)) break;
    const uint8_t* slot = ring + (q & (D - 1)) * kFwdUnit;
    const int i = ci, kbl = kFwdQuad * cq + t4;
    if (++cq == nq) {
      cq = 0;
      ++ci;
    }
    if (i != ctile) {  // first tile done (a range touches at most two)
      store_acc(first + warp * kSlotElems);
      ctile = i;
    }
    const float sA = scale(s0.a), sB = scale(s0.b);
    const uint64_t sA2 = pair2(sA, sA), sB2 = pair2(sB, sB);
    const uint4 ca0 = lds128(slot + (g * 8 + ((2 * t4) ^ sw)) * 16);
    const uint4 ca1 = lds128(slot + (g * 8 + ((2 * t4 + 1) ^ sw)) * 16);
    const uint4 cb0 = lds128(slot + ((g + 8) * 8 + ((2 * t4) ^ sw)) * 16);
    const uint4 cb1 = lds128(slot + ((g + 8) * 8 + ((2 * t4 + 1) ^ sw)) * 16);
    const uint4* xr[MT];
#pragma unroll
    for (int t = 0; t < MT; ++t) xr[t] = xs + (((8 * t + g) * nch + kbl) << 3);
    const uint32_t wa[8] = {ca0.x, ca0.y, ca0.z, ca0.w, ca1.x, ca1.y, ca1.z, ca1.w};
    const uint32_t wb[8] = {cb0.x, cb0.y, cb0.z, cb0.w, cb1.x, cb1.y, cb1.z, cb1.w};
#pragma unroll
    for (int u = 0; u < 8; ++u) {  // 16-byte activation unit u: MMAs 2u and 2u+1
      uint4 xv[MT];
#pragma unroll
      for (int t = 0; t < MT; ++t) xv[t] = xr[t][u ^ f];
      // word u holds values 8u .. 8u+7 of the block: bytes 0, 1 feed MMA 2u, bytes 2, 3 MMA 2u+1
      const uint32_t af[4] = {lookup<F16>(smem, wa[u], lane8, kSel0, sA2),
                              lookup<F16>(smem, wb[u], lane8, kSel0, sB2),
                              lookup<F16>(smem, wa[u], lane8, kSel1, sA2),
                              lookup<F16>(smem, wb[u], lane8, kSel1, sB2)};
#pragma unroll
      for (int t = 0; t < MT; ++t) mma16816<F16>(acc[t], af, xv[t].x, xv[t].y);
      const uint32_t ag[4] = {lookup<F16>(smem, wa[u], lane8, kSel2, sA2),
                              lookup<F16>(smem, wb[u], lane8, kSel2, sB2),
                              lookup<F16>(smem, wa[u], lane8, kSel3, sA2),
                              lookup<F16>(smem, wb[u], lane8, kSel3, sB2)};
#pragma unroll
      for (int t = 0; t < MT; ++t) mma16816<F16>(acc[t], ag, xv[t].z, xv[t].w);
    }
    __syncwarp();
    s0 = s1;
    s1 = issue();
  }
  // After a wait that ran out, the copies still in flight land before the ring is
  // reused or the CTA exits.
  for (; q < issued && q < nunits; ++q)
    ring_wait(bars_s + 8 * (q & (D - 1)), static_cast<uint32_t>(q / D) & 1u, nullptr);
  __syncwarp();
  if (nunits > 0) store_acc(reinterpret_cast<float*>(ring));  // last tile -> own ring
  __syncthreads();

  // element e = (tile i, token, row): i = e >> kSlotShift; tokens >= M are skipped
  const int M = static_cast<int>(a.M);
  const int total = nt << kSlotShift;
  const float* last = reinterpret_cast<const float*>(smem + L.ring);
  auto store = [&](int e, float v) {
    const int i = e >> kSlotShift, r = e & (kSlotElems - 1);
    const int64_t n = (tile0 + i) * 16 + (r & 15);
    if ((r >> 4) < M && n < a.N && in_bounds(n >= 0 && n < a.ld_out, a.status))
      store16<F16>(a.out + (r >> 4) * a.ld_out + n, v);
  };
  for (int e = threadIdx.x; e < total; e += kThreads) {
    const int i = e >> kSlotShift, r = e & (kSlotElems - 1);
    if ((r >> 4) >= M) continue;
    const float v = cta_sum(i, r, U, nq, first, kSlotElems, last, D * kFwdUnit / 4);
    if (S == 1)
      store(e, v);
    else
      cluster_push(recv, rank, S, total, e, v);
  }
  if (S > 1) cluster_finish(recv, rank, S, total, store);
}

// ---------------------------------------------------------- input gradient --
//
// grad_x^T = W^T grad_y^T: the MMA's rows are in-features and its contraction
// runs over weight rows.  Tile = one 64-value block column (64 in-features); a
// unit = one tile x 64 weight rows, taken as four groups of 16.  In a group,
// lane (g, t4) holds weight rows {2t4, 2t4+1, 2t4+8, 2t4+9} (contraction slots)
// at the in-features 8g .. 8g+7 of the block (one 4-byte word per row).  MMA m
// (0..3) gives output row g the in-feature 8g + 2m (high nibble of byte m) and
// row g+8 the value 8g + 2m + 1 (low nibble), so the A operand pair of slots
// (2t4, 2t4+1) at one in-feature is a byte made of one nibble of each of two
// weight rows, looked up in the same table and scaled by the two rows' block
// scales; a lane's accumulators stay on its own 16 in-features for the whole
// column.  The unit's grad_y values travel in the same ring slot as its codes.
template <int MT, bool F16>
__global__ void __launch_bounds__(kThreads, 1)
    skinny_dgrad_kernel(const __grid_constant__ CUtensorMap tmap, const SkinnyArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  // The tile copies' swizzle follows absolute shared-memory address bits: the
  // ring must start on a 1024-byte boundary (it does, after the 64 KB table, when
  // the dynamic shared memory does).
  if ((smem_addr(smem) & 1023u) != 0) {
    if (threadIdx.x == 0 && a.status) *reinterpret_cast<volatile int*>(a.status) = NF4_ERR_UNSUPPORTED;
    return;
  }
  constexpr int D = kBwdDepth;
  constexpr int kRows = kBwdRows;                  // weight rows per unit
  constexpr int kGyPitch = kRows * 2 + 16;         // bytes per token (padded)
  constexpr int kUnit = kBwdCodeUnit;              // code ring slot
  constexpr int kGyUnit = bwd_gy_unit_bytes(MT);   // grad_y ring slot
  constexpr int kSlotElems = MT * 8 * 64;          // [token][in-feature]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int S = a.S;
  const int rank = static_cast<int>(blockIdx.x) & (S - 1);
  const int cl = static_cast<int>(blockIdx.x) >> a.log2S;
  // cl * T / C and (cl + 1) * T / C from T = tq C + tr (32-bit divisions only)
  const int64_t col0 = cl * a.tq + (cl * a.tr) / a.C;
  const int nt = static_cast<int>((cl + 1) * a.tq + ((cl + 1) * a.tr) / a.C - col0);
  const int64_t nr0 = static_cast<int64_t>(rank) * a.cc;
  const int64_t nr1 = a.N - nr0 < a.cc ? a.N : nr0 + a.cc;  // this CTA's weight rows
  const int nn = static_cast<int>((nr1 - nr0 + kRows - 1) / kRows);
  const int U = nt * nn;
  const WarpRange mine = warp_range(warp, U, nn);
  const int nunits = mine.hi - mine.lo;
  const Layout L = a.lay;
  uint8_t* ring = smem + L.ring + warp * D * kUnit;
  uint8_t* gyring = smem + L.gy + warp * D * kGyUnit;
  float* first = reinterpret_cast<float*>(smem + L.first);
  float* recv = reinterpret_cast<float*>(smem + L.recv);
  float* sc = reinterpret_cast<float*>(smem + L.scales);  // [column][row - nr0]
  const int ccs = static_cast<int>(a.cc);
  // The warp's ring barriers (one per slot, for the code tiles), initialised by
  // its lane 0: the padding bytes 128-143 of grad_y slot 0's first token row,
  // which no copy writes and no lookup reads.
  static_assert(kGyPitch >= kRows * 2 + 8 * D, "barriers in the grad_y row padding");
  const uint32_t bars_s = smem_addr(gyring) + kRows * 2;
  if (lane == 0) {
    for (int j = 0; j < D; ++j) nf4ptx::mbar_init(bars_s + 8 * j, 1);
    nf4ptx::fence_mbar_init();
  }
  __syncwarp();

  // Copies of unit (ii, ij): one tile copy by lane 0 of the codes of rows n0 ..
  // n0 + 63 of block column kb (rows past N read as zeros; rows of the next rank
  // come in too and meet zero scales and zero grad_y), and grad_y chunks lane +
  // 32 j (token c >> 3, rows 8 (c & 7) ..) by every lane; ragged ends and absent
  // tokens are written directly.
  const uint32_t ring_s = smem_addr(ring);
  int issued = 0, ii = mine.t0, ij = mine.lo - mine.t0 * nn;
  auto gy_edge = [&](uint8_t* d, int tok, int64_t ng) {  // 8 values from row ng, zero-padded
    uint16_t v[8];
#pragma unroll
    for (int q = 0; q < 8; ++q)
      v[q] = (tok < a.M && ng + q < nr1)
                 ? reinterpret_cast<const uint16_t*>(a.act + tok * a.ld_act)[ng + q]
                 : static_cast<uint16_t>(0);
    *reinterpret_cast<uint4*>(d) =
        make_uint4(v[0] | (static_cast<uint32_t>(v[1]) << 16), v[2] | (static_cast<uint32_t>(v[3]) << 16),
                   v[4] | (static_cast<uint32_t>(v[5]) << 16), v[6] | (static_cast<uint32_t>(v[7]) << 16));
  };
  auto copy_gy = [&](int slot, int64_t n0, bool async) {
#pragma unroll
    for (int j = 0; j < MT * 8 * 8 / 32; ++j) {
      const int c = lane + 32 * j, tok = c >> 3, part = c & 7;
      const int64_t ng = n0 + 8 * part;
      const uint32_t off = slot * kGyUnit + tok * kGyPitch + part * 16;
      if (tok >= a.M) continue;  // absent tokens only feed discarded outputs
      if (ng + 8 <= nr1) {
        if (async)
          cp_async16(smem_addr(gyring) + off, a.act + tok * a.ld_act + ng, true);
        else
          *reinterpret_cast<uint4*>(gyring + off) =
              *reinterpret_cast<const uint4*>(a.act + tok * a.ld_act + ng);
      } else {
        gy_edge(gyring + off, tok, ng);
      }
    }
  };
  auto issue = [&](bool with_gy) {
    if (issued < nunits) {
      const int slot = issued % D;
      const int64_t kb = col0 + ii;
      const int64_t n0 = nr0 + static_cast<int64_t>(kRows) * ij;
      if (lane == 0) {
        const uint32_t bar = bars_s + 8 * slot;
        nf4ptx::mbar_arrive_expect_tx(bar, kRows * 32);
        nf4ptx::tma_load_2d(ring_s + slot * kUnit, &tmap, bar, static_cast<int32_t>(kb * 32),
                            static_cast<int32_t>(n0));
      }
      if (with_gy) copy_gy(slot, n0, true);
      if (++ij == nn) {
        ij = 0;
        ++ii;
      }
    }
    ++issued;
    cp_async_commit();
  };
  // The first loads all go out together, so that the kernel start costs about one
  // memory round trip: the first units' tile copies (and their grad_y, once the
  // grid dependency has resolved), the codebook values of the byte-pair table, the
  // 8-bit codebook entry, the nested offset and the first batch of block
  // statistics; the stores that need those values follow.
  // Scales: [column][row - nr0], whole units; zero beyond the CTA's rows.
  const int nsc = nt * ccs;
  auto block_of = [&](int idx) -> int64_t {
    const int i = idx / ccs, nl = idx - i * ccs;
    const int64_t n = nr0 + nl;
    return n < nr1 ? n * a.KB + col0 + i : -1;
  };
  float* code8s = reinterpret_cast<float*>(smem + L.code8);
  TableSrc tsrc;
  ScaleBatch sb0;
  float c8, offset;  // 8-bit codebook entry, nested offset (double quantisation)
  auto weight_side = [&](bool with_gy) {
    for (int j = 0; j < D; ++j) issue(with_gy);
    tsrc = table_src(a.code4);
    // unconditional loads from valid addresses (used only under double quantisation)
    c8 = __ldg(a.dq ? a.code8 + (threadIdx.x & 255) : a.code4);
    offset = __ldg(a.dq ? a.nested_offset : a.code4);
    sb0 = fetch_scales(a, threadIdx.x, nsc, block_of);
  };

  // One call site for the weight side (the dependency wait goes before or after
  // it), so that no branch merge makes the thread wait for the loaded values here.
  if (!a.prefetch) grid_dependency_wait();
  weight_side(!a.prefetch);
  if (a.prefetch) {
    grid_dependency_wait();
    // grad_y of the prefetched units, now that it is final: one group per unit, in order
    for (int j = 0, gj = mine.lo - mine.t0 * nn; j < D; ++j, gj = gj + 1 == nn ? 0 : gj + 1) {
      if (j < nunits) copy_gy(j, nr0 + static_cast<int64_t>(kRows) * gj, true);
      cp_async_commit();
    }
  }
  allow_dependents();
  store_table(smem, tsrc);
  static_assert(kThreads >= 256, "one 8-bit codebook entry per thread");
  if (a.dq && threadIdx.x < 256) code8s[threadIdx.x] = c8;
  __syncthreads();  // code8s
  finish_scales(a, sc, code8s, offset, threadIdx.x, nsc, sb0);
  for (int i0 = threadIdx.x + 4 * kThreads; i0 < nsc; i0 += 4 * kThreads)
    finish_scales(a, sc, code8s, offset, i0, nsc, fetch_scales(a, i0, nsc, block_of));
  __syncthreads();

  const uint32_t lane8 = static_cast<uint32_t>(lane) << 3;
  const int rr[4] = {2 * t4, 2 * t4 + 1, 2 * t4 + 8, 2 * t4 + 9};
  float acc[MT][4][4];
#pragma unroll
  for (int t = 0; t < MT; ++t)
#pragma unroll
    for (int m = 0; m < 4; ++m) acc[t][m][0] = acc[t][m][1] = acc[t][m][2] = acc[t][m][3] = 0.0f;
  int ccol = mine.t0;
  int ci = mine.t0, cj = mine.lo - mine.t0 * nn;  // (column, row unit) being decoded

  auto store_acc = [&](float* p) {
#pragma unroll
    for (int t = 0; t < MT; ++t)
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int tok = 8 * t + 2 * t4, k = 8 * g + 2 * m;
        p[tok * 64 + k] = acc[t][m][0];
        p[(tok + 1) * 64 + k] = acc[t][m][1];
        p[tok * 64 + k + 1] = acc[t][m][2];
        p[(tok + 1) * 64 + k + 1] = acc[t][m][3];
        acc[t][m][0] = acc[t][m][1] = acc[t][m][2] = acc[t][m][3] = 0.0f;
      }
  };

  int q = 0;
  for (; q < nunits; ++q) {
    cp_async_wait<D - 1>();  // this unit's grad_y
    __syncwarp();
    if (!ring_wait(bars_s + 8 * (q % D), static_cast<uint32_t>(q / D) & 1u, a.status)) break;
    const uint8_t* slot = ring + (q % D) * kUnit;
    const uint8_t* gslot = gyring + (q % D) * kGyUnit;
    const int i = ci;
    const int nl0 = kRows * cj;  // first row of the unit, relative to nr0
    if (++cj == nn) {
      cj = 0;
      ++ci;
    }
    if (i != ccol) {  // first column done (a range touches at most two)
      store_acc(first + warp * kSlotElems);
      ccol = i;
    }
    const float* scol = sc + i * ccs + nl0;
#pragma unroll
    for (int rg = 0; rg < kRows / 16; ++rg) {  // 16-row groups of the unit
      uint32_t w[4];
      float s[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int r = 16 * rg + rr[k];
        w[k] = *reinterpret_cast<const uint32_t*>(slot + code_unit(r, g >> 2) * 16 + (g & 3) * 4);
        s[k] = scol[r];
      }
      const uint64_t s01 = pair2(s[0], s[1]), s23 = pair2(s[2], s[3]);
      uint32_t b[MT][2];
#pragma unroll
      for (int t = 0; t < MT; ++t) {
        const uint8_t* gy = gslot + (8 * t + g) * kGyPitch + (16 * rg + 2 * t4) * 2;
        b[t][0] = *reinterpret_cast<const uint32_t*>(gy);
        b[t][1] = *reinterpret_cast<const uint32_t*>(gy + 16);
      }
      // table indices: byte m = (code of row 2t4, code of row 2t4+1) at in-feature
      // 8g + 2m (even) or 8g + 2m + 1 (odd); likewise rows 2t4+8, 2t4+9
      const uint32_t e01 = (w[0] & 0xf0f0f0f0u) | ((w[1] >> 4) & 0x0f0f0f0fu);
      const uint32_t o01 = ((w[0] << 4) & 0xf0f0f0f0u) | (w[1] & 0x0f0f0f0fu);
      const uint32_t e23 = (w[2] & 0xf0f0f0f0u) | ((w[3] >> 4) & 0x0f0f0f0fu);
      const uint32_t o23 = ((w[2] << 4) & 0xf0f0f0f0u) | (w[3] & 0x0f0f0f0fu);
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const uint32_t sel = lookup_sel(static_cast<uint32_t>(m));
        const uint32_t af[4] = {lookup<F16>(smem, e01, lane8, sel, s01), lookup<F16>(smem, o01, lane8, sel, s01),
                                lookup<F16>(smem, e23, lane8, sel, s23), lookup<F16>(smem, o23, lane8, sel, s23)};
#pragma unroll
        for (int t = 0; t < MT; ++t) mma16816<F16>(acc[t][m], af, b[t][0], b[t][1]);
      }
    }
    __syncwarp();
    issue(true);
  }
  // After a wait that ran out, the copies still in flight land before the ring is
  // reused or the CTA exits.
  for (; q < issued && q < nunits; ++q)
    ring_wait(bars_s + 8 * (q % D), static_cast<uint32_t>(q / D) & 1u, nullptr);
  cp_async_wait<0>();
  __syncwarp();
  if (nunits > 0) store_acc(reinterpret_cast<float*>(ring));  // last column -> own ring
  __syncthreads();

  const int M = static_cast<int>(a.M);
  const int total = nt * M * 64;  // (column, token, in-feature)
  const float* last = reinterpret_cast<const float*>(smem + L.ring);
  auto store = [&](int e, float v) {
    const int i = e / (M * 64), r = e - i * M * 64;
    const int64_t k = (col0 + i) * 64 + (r & 63);  // in-feature
    if (in_bounds((r >> 6) < a.M && k >= 0 && k < a.K && k < a.ld_out, a.status))
      store16<F16>(a.out + (r >> 6) * a.ld_out + k, v);
  };
  for (int e = threadIdx.x; e < total; e += kThreads) {
    const int i = e / (M * 64), r = e - i * M * 64;
    const float v = cta_sum(i, r, U, nn, first, kSlotElems, last, D * kUnit / 4);
    if (S == 1)
      store(e, v);
    else
      cluster_push(recv, rank, S, total, e, v);
  }
  if (S > 1) cluster_finish(recv, rank, S, total, store);
}

using SkinnyKernel = void (*)(CUtensorMap, SkinnyArgs);

template <int MODE, int MT, bool F16>
cudaError_t configure(SkinnyKernel& kern) {
  kern = MODE == 0 ? skinny_fwd_kernel<MT, F16> : skinny_dgrad_kernel<MT, F16>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kMaxSmem));
    if (e != cudaSuccess) return e;
    configured = true;
  }
  return cudaSuccess;
}

// Clusters of S CTAs (with `smem` bytes each) that can be resident at once.
template <int MODE, int MT, bool F16>
int max_clusters_mt(int S, size_t smem) {
  SkinnyKernel kern = nullptr;
  if (configure<MODE, MT, F16>(kern) != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(S), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(S);
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

// Cached per (mode, tiles, operand type, S, shared-memory size).
int max_clusters(int mode, int mt, bool f16, int S, size_t smem) {
  struct Entry {
    int mode, mt, f16, S;
    size_t smem;
    int n;
  };
  static std::mutex mu;
  static std::vector<Entry> cache;
  std::lock_guard<std::mutex> lk(mu);
  for (const Entry& e : cache)
    if (e.mode == mode && e.mt == mt && e.f16 == static_cast<int>(f16) && e.S == S && e.smem == smem)
      return e.n;
  int n;
  if (f16) {
    if (mode == 0)
      n = mt == 1 ? max_clusters_mt<0, 1, true>(S, smem) : max_clusters_mt<0, 2, true>(S, smem);
    else
      n = mt == 1 ? max_clusters_mt<1, 1, true>(S, smem) : max_clusters_mt<1, 2, true>(S, smem);
  } else {
    if (mode == 0)
      n = mt == 1 ? max_clusters_mt<0, 1, false>(S, smem) : max_clusters_mt<0, 2, false>(S, smem);
    else
      n = mt == 1 ? max_clusters_mt<1, 1, false>(S, smem) : max_clusters_mt<1, 2, false>(S, smem);
  }
  cache.push_back(Entry{mode, mt, static_cast<int>(f16), S, smem, n});
  return n;
}

template <int MODE, int MT, bool F16>
cudaError_t launch_mt(const SkinnyArgs& a, const SkinnyPlan& p, const CUtensorMap& tmap,
                      cudaStream_t s) {
  SkinnyKernel kern = nullptr;
  cudaError_t ce = configure<MODE, MT, F16>(kern);
  if (ce != cudaSuccess) return ce;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.C * p.S), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (p.S > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = static_cast<unsigned>(p.S);
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, tmap, a);
}

}  // namespace

// Plan: the contraction split S (cluster size) and the number C of clusters
// (one CTA per SM).  Tiles are dealt to clusters in balanced contiguous ranges;
// the cost is the busiest CTA's weight values plus a charge per rank for the
// cluster reduction.  A warp's unit range must touch at most two tiles, and the
// shared memory must fit.  A deterministic function of the shape and the SM
// count.
bool skinny_plan(int mode, int64_t M, int64_t N, int64_t K, int sms, SkinnyPlan* out, bool f16) {
  if (M < 1 || M > kSkinnyMaxM || sms < 1 || K % 64 != 0) return false;
  const int mt = M <= 8 ? 1 : 2;
  const int64_t KB = K / 64;
  const int64_t T = mode == 0 ? (N + 15) / 16 : KB;      // output tiles
  const int64_t steps = mode == 0 ? KB : (N + kBwdRows - 1) / kBwdRows;  // contraction steps
  const int64_t gran = mode == 0 ? 64 : kBwdRows;                        // contraction per step
  double best = 1e300;
  SkinnyPlan bp;
  const int ss[4] = {1, 2, 4, 8};
  for (int si = 0; si < 4; ++si) {
    const int S = ss[si];
    const int64_t per = (steps + S - 1) / S;  // steps per rank
    if ((steps + per - 1) / per != S) continue;
    int64_t C64 = sms / S;
    if (C64 > T) C64 = T;
    if (C64 < 1) continue;
    int C = static_cast<int>(C64);
    int64_t nt_max = (T + C - 1) / C;
    Layout L = make_layout(mode, mt, S, per * gran, nt_max);
    // clusters must all be resident at once (a GPC holds whole clusters only)
    for (int it = 0; S > 1 && it < 4; ++it) {
      const int cmax = max_clusters(mode, mt, f16, S, static_cast<size_t>(L.total));
      if (cmax >= C) break;
      C = cmax;
      if (C < 1) break;
      nt_max = (T + C - 1) / C;
      L = make_layout(mode, mt, S, per * gran, nt_max);
    }
    if (C < 1) continue;
    const int64_t upt = mode == 0 ? (per + kFwdQuad - 1) / kFwdQuad : per;  // units per tile
    if ((nt_max * upt + kWarps - 1) / kWarps > upt) continue;  // ranges span <= 2 tiles
    if (static_cast<size_t>(L.total) > kMaxSmem) continue;
    // cycles at ~24 weight values per clock and SM, plus the cluster exchange
    const double cost = static_cast<double>(nt_max) * per * (mode == 0 ? 1024 : 4096) / 24.0 +
                        (S > 1 ? 1500.0 : 0.0);
    if (cost < best * 0.999) {
      best = cost;
      bp.S = S;
      bp.C = C;
      bp.T = T;
      bp.cc = per * gran;
      bp.smem = static_cast<size_t>(L.total);
    }
  }
  if (bp.S == 0) return false;
  *out = bp;
  return true;
}

cudaError_t launch_skinny(int mode, const SkinnyArgs& args, const SkinnyPlan& p, const CUtensorMap& tmap,
                          cudaStream_t s) {
  SkinnyArgs a = args;
  const bool mt1 = a.M <= 8;
  a.nt_max = (p.T + p.C - 1) / p.C;
  a.tq = p.T / p.C;
  a.tr = static_cast<int>(p.T % p.C);
  a.log2S = p.S == 1 ? 0 : p.S == 2 ? 1 : p.S == 4 ? 2 : 3;
  a.lay = make_layout(mode, mt1 ? 1 : 2, p.S, p.cc, a.nt_max);
  if (a.f16) {
    if (mode == 0) return mt1 ? launch_mt<0, 1, true>(a, p, tmap, s) : launch_mt<0, 2, true>(a, p, tmap, s);
    return mt1 ? launch_mt<1, 1, true>(a, p, tmap, s) : launch_mt<1, 2, true>(a, p, tmap, s);
  }
  if (mode == 0) return mt1 ? launch_mt<0, 1, false>(a, p, tmap, s) : launch_mt<0, 2, false>(a, p, tmap, s);
  return mt1 ? launch_mt<1, 1, false>(a, p, tmap, s) : launch_mt<1, 2, false>(a, p, tmap, s);
}

}  // namespace nf4
