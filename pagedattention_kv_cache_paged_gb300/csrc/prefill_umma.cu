// tcgen05 causal chunked prefill over a paged history (bf16/fp16, block_size % 16 == 0).
//
// JuliaPagedAttn README "Features" (batched prefill) with the online softmax of "Online Softmax":
// the chunk of m_b queries holds the last m_b positions of sequence b's context and query r
// attends to positions 0 .. n_b - m_b + r through the block table.  Computed on the 5th-generation
// tensor cores with accumulators in tensor memory.
//
// Persistent: one CTA per SM walks the work items (blockIdx, blockIdx + gridDim, ...).  An item =
// 256 (query token, head) rows of one KV head, split into two 128-row Q tiles that share every K/V
// tile (kRows / G tokens x the G heads of the group: read-time GQA, nanoserve Day 19 "What I
// learned" 4).  11 warps; the producers and the MMA warp run on lane 0 alone (a warp whose lanes
// meet at warp-collective steps between long single-lane stretches loses about a thousand cycles
// per meeting):
//   warps 0-3 / 4-7  softmax groups 0 / 1: thread t of group k owns row 128k + t (TMEM lane t of
//              S_k and O_k); turns each S_k tile into probabilities (compact code: 64-key blocks
//              in a loop; one instantiation per masking mode, see ScoreFix), rescales O_k in TMEM
//              only when its stabilising maximum has to move up by more than 2^8, writes P_k
//              (bf16/fp16) back into the TMEM columns of S_k, and normalises O_k at the end;
//   warp 8     K producer: finds each item's segments (the rows of one sequence: an 8-way search
//              over query_start_loc, then the sequence's bounds and length; for the next item this
//              runs one step per K tile of the current one, so that its dependent loads overlap
//              useful waiting) and publishes the item's tile count (for the MMA warp) and a record
//              per segment (for the V producer and the softmax groups) through small shared-memory
//              rings; streams 128-key K tiles (TMA boxes of 16 keys x 64 columns from the physical
//              blocks the table names, the table entries read one tile ahead) into a
//              kUmKStages-deep ring and publishes which sub-tiles hold data;
//   warp 9     V producer: each item's two Q tiles (one TMA box per 64-column half, once the
//              previous item's S products are done; the next item's Q tiles are prefetched into
//              L2 meanwhile), then the matching V tiles into a kUmVStages-deep ring;
//   warp 10    MMA: allocates TMEM (S_0, S_1: 128 columns each; O_0, O_1: 128 columns each) and
//              issues S_k = Q_k K^T (M 128, N 128, both operands in shared memory) and
//              O_k += P_k V (M 128, N head_dim, P read from TMEM, V an MN-major shared-memory
//              operand) with tcgen05.mma in the order S_0(j), P_1(j-1) V, S_1(j), P_0(j) V, so
//              that the tensor core works on one group's products while the other group computes
//              its softmax.  P_k lives in the columns the next S_k overwrites: S_k of the next
//              tile is issued right after O_k += P_k V of this one, and tcgen05 products of one
//              thread run in issue order, so the P V reads P_k first.  The commit that signals
//              the new S_k also covers that P V, so O_k is stable whenever a group sees a new S_k
//              and rescaling needs no extra wait.
// Every mbarrier wait is bounded (PA_DEVERR_TIMEOUT, with a cooperative abort); TMEM is always
// released.  The stabilising maximum is exact bookkeeping: numerator and denominator use the
// same one, so the result equals the running-max form of "Online Softmax" in real arithmetic.
#include <cudaTypedefs.h>

#include <algorithm>

#include "pa_common.cuh"
#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {

constexpr int kUmThreads = 352;            // 8 softmax warps, K producer, V producer, MMA
constexpr int kUmTileRows = 128;            // rows per Q tile (MMA M)
constexpr int kUmRows = 2 * kUmTileRows;    // rows per CTA
constexpr int kUmKeys = 128;                // keys per K/V tile (N of S, K of PV)
constexpr int kUmSub = kUmKeys / 16;
constexpr int kUmTmemCols = 512;
constexpr int kUmSegSlots = 8;   // segment records in flight between the K producer and their readers
constexpr int kUmItemSlots = 4;  // item tile counts in flight between the K producer and the MMA warp
// Ring depths (build-time overridable): K 2 / V 3 measured 1 % faster than K 3 / V 2 (V tiles are
// needed later in a tile's chain, so their loads profit from the deeper ring)
#ifndef PA_UM_KSTAGES
#define PA_UM_KSTAGES 2
#endif
#ifndef PA_UM_VSTAGES
#define PA_UM_VSTAGES 3
#endif
constexpr int kUmKStages = PA_UM_KSTAGES;   // K ring depth
constexpr int kUmVStages = PA_UM_VSTAGES;   // V ring depth
constexpr float kUmRescaleThreshold = 8.f;  // log2 units: O is rescaled when the max grows by > 2^8

template <int D>
struct UmCfg {
  static constexpr int kHalves = D / 64;
  static constexpr int kQHalf = kUmTileRows * 128;   // one 64-column half of a Q tile
  static constexpr int kQBytes = kUmTileRows * D * 2;
  static constexpr int kKvHalf = kUmKeys * 128;      // one 64-column half of a K or V tile
  static constexpr int kKvBytes = kUmKeys * D * 2;
  static constexpr int kSmemBytes = 1024 + 1024 + 2 * kQBytes + (kUmKStages + kUmVStages) * kKvBytes;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
};

// Byte offset of (row r, 8-element chunk c) in a [half][rows][128 B] swizzled operand.
__device__ __forceinline__ uint32_t sw_off(int r, int c, int half_bytes) {
  return (uint32_t)((c >> 3) * half_bytes + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// Softmax helpers: one thread owns one row of S (its TMEM lane); `taddr` is the row's first column.
//
// One code path serves every tile.  The exponentials are taken as 2^(sc * s - m) with sc > 0, so
// the row maximum can be taken over the raw scores and scaled once.  A tile that has masked keys
// (outside the causal bound, or in a sub-tile that was not loaded), or a non-positive scale, first
// rewrites the loaded scores in registers (ScoreFix): a masked key becomes -inf, whose probability
// is exactly 0.  The common case, keys [0, nv) valid (the causal bound and the end of the loaded
// keys both cut a prefix), costs one compare and select per key of the 64-key blocks that the cut
// falls in, and a block wholly past the cut for every row of the warp is skipped.  Anything else
// (a sub-tile skipped for an out-of-range block id, or a scale <= 0) takes the general rewrite: key c valid when bit c % 32 of mask[c / 32] is set, a negative scale flips
// the sign of every score and uses |scale| (the same products sc * s), a zero scale makes every
// score 0 with scale 1 (the same uniform weights).

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// v = -inf unless j < nv (one compare, one select)
__device__ __forceinline__ void keep_below(uint32_t& v, int j, int nv) {
  asm("{\n\t.reg .pred p;\n\tsetp.lt.s32 p, %1, %2;\n\tselp.b32 %0, %0, 0xff800000, p;\n\t}"
      : "+r"(v)
      : "r"(j), "r"(nv));
}

struct ScoreFix {
  int mode;       // 0: scores used as loaded; 1: keys >= nv masked; 2: general rewrite
  int nv;         // mode 1: keys [0, nv) of the tile are valid
  uint32_t flip;  // mode 2: sign bit flipped (negative scale)
  bool zero;      // mode 2: scores replaced by 0 (zero scale)
};

// The softmax code runs once per tile on every SM; it is kept compact (one 64-column block in a
// loop, not the whole row unrolled) so that it stays in the instruction cache: fully unrolled rows,
// with a separate masked variant, measured slower from instruction fetch alone.

// Columns [c0, c0 + 64) of the row of S into registers (two loads in flight, one wait), rewritten
// as `fix` says; m0 / m1 are the mask words of the block's two 32-key chunks.  One instantiation
// per masking mode (kMode = fix.mode): mode 0 runs no masking code at all, mode 1 applies the prefix
// cut only in a block that the cut falls in, mode 2 is the rare general rewrite.  (One copy of the
// code for modes 0 and 1, the cut behind a warp-uniform branch, measured slower.)
template <int kMode>
__device__ __forceinline__ void s_load64(uint32_t taddr, uint32_t (&sv)[64], const ScoreFix& fix, int c0,
                                         uint32_t m0, uint32_t m1) {
  tmem_ld32(taddr, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
  tmem_ld32(taddr + 32u, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
  tmem_wait_ld();
  tmem_pin32(*reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
  tmem_pin32(*reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
  if (kMode == 1) {
    const int nv = fix.nv - c0;
    if (nv < 64) {
#pragma unroll
      for (int j = 0; j < 64; ++j) keep_below(sv[j], j, nv);
    }
  } else if (kMode == 2) {
#pragma unroll
    for (int j = 0; j < 64; ++j) {
      const uint32_t v = fix.zero ? 0u : (sv[j] ^ fix.flip);
      sv[j] = (((j < 32 ? m0 : m1) >> (j & 31)) & 1u) ? v : 0xff800000u;  // -inf
    }
  }
}

// Maximum of the 64 scores held in sv, times sc (> 0).
__device__ __forceinline__ float s_max64(const uint32_t (&sv)[64], float sc) {
  float m[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
  for (int j = 0; j < 64; j += 8)
#pragma unroll
    for (int u = 0; u < 4; ++u) m[u] = fmax3(m[u], __uint_as_float(sv[j + 2 * u]), __uint_as_float(sv[j + 2 * u + 1]));
  return fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3])) * sc;
}

// Probabilities 2^(sc * s - m_sub) of the 64 keys held in sv, written as 16-bit pairs into the 32
// columns at taddr (keys 2c and 2c + 1 in column c); returns their sum.  Packed pairs: one f32x2 fma
// for the scaled, shifted arguments and one f32x2 add for the sum.
template <bool kBf16>
__device__ __forceinline__ float p_store64(uint32_t taddr, const uint32_t (&sv)[64], float sc, float m_sub) {
  const uint64_t sc2 = f2_pack(sc, sc), nm2 = f2_pack(-m_sub, -m_sub);
  uint64_t acc2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
  uint32_t w[32];
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    float x0, x1;
    f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[2 * c]), __uint_as_float(sv[2 * c + 1])), sc2, nm2), x0, x1);
    const uint64_t e2 = f2_pack(fast_exp2(x0), fast_exp2(x1));
    acc2[c & 1] = f2_add(acc2[c & 1], e2);
    float e0, e1;
    f2_unpack(e2, e0, e1);
    w[c] = pack2<kBf16>(e0, e1);
  }
  tmem_st32(taddr, w);
  float a0, a1, b0, b1;
  f2_unpack(acc2[0], a0, a1);
  f2_unpack(acc2[1], b0, b1);
  return (a0 + b0) + (a1 + b1);
}

// Row maximum and probabilities of one S tile, in two blocks of 64 keys read twice (once for the
// maximum, once for the exponentials, so that only 64 scores are held in registers at a time; the
// P of block h goes to columns [32h, 32h + 32), which block h has already been read from).  Moves
// the stabilising maximum m_use when it has to and returns the factor the earlier sum and O must be
// scaled by.  sc > 0 (see ScoreFix).
template <bool kBf16, int kMode>
__device__ __forceinline__ float row_softmax(uint32_t srow, float sc, const ScoreFix& fix,
                                             const uint32_t (&mask)[kUmKeys / 32], float& m_use, float& l_run) {
  static_assert(kUmKeys == 128, "two blocks of 64 keys");
  // a 64-key block masked for every row of the warp (past the causal cut or the loaded keys)
  // contributes nothing: it is neither read nor exponentiated, its P is written as zeros
  auto block_empty = [&](int h) {
    return kMode == 1 && __all_sync(0xffffffffu, fix.nv - 64 * h <= 0);
  };
  float mx = -INFINITY;
#pragma unroll 1
  for (int h = 0; h < 2; ++h) {
    if (block_empty(h)) continue;
    uint32_t sv[64];
    s_load64<kMode>(srow + 64u * h, sv, fix, 64 * h, h ? mask[2] : mask[0], h ? mask[3] : mask[1]);
    mx = fmaxf(mx, s_max64(sv, sc));
  }
  // move the stabiliser only when it must: first finite maximum, or growth beyond 2^8
  float corr = 1.f;
  if (mx > m_use + kUmRescaleThreshold || (m_use == -INFINITY && mx != -INFINITY)) {
    corr = fast_exp2(m_use - mx);  // m_use = -inf -> 0
    m_use = mx;
  }
  const float m_sub = m_use == -INFINITY ? 0.f : m_use;
  float rs = 0.f;
#pragma unroll 1
  for (int h = 0; h < 2; ++h) {
    if (block_empty(h)) {
      uint32_t z[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) z[c] = 0u;
      tmem_st32(srow + 32u * h, z);
      continue;
    }
    uint32_t sv[64];
    s_load64<kMode>(srow + 64u * h, sv, fix, 64 * h, h ? mask[2] : mask[0], h ? mask[3] : mask[1]);
    rs += p_store64<kBf16>(srow + 32u * h, sv, sc, m_sub);
  }
  l_run = l_run * corr + rs;
  return corr;
}

// Sequence of query row t: the largest b < batch with qsl[b] <= t, searched by one thread with
// rounds of 8 independent loads (three rounds for batch <= 512).
__device__ __forceinline__ int find_sequence_8(const int32_t* qsl, int batch, int t) {
  int lo = 0, n = batch;
  while (n > 1) {
    const int step = (n + 7) >> 3;
    int v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] = k * step < n ? ld_nc_s32(qsl + lo + k * step) : INT32_MAX;
    int top = 0;
#pragma unroll
    for (int k = 1; k < 8; ++k)
      if (k * step < n && v[k] <= t) top = k;
    const int nlo = lo + top * step;
    n = min(step, lo + n - nlo);
    lo = nlo;
  }
  return lo;
}

template <typename T, int D, int G>
__global__ void __launch_bounds__(kUmThreads)
    prefill_umma_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap qmap) {
  using Cfg = UmCfg<D>;
  constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
  constexpr int kHalves = Cfg::kHalves;
  constexpr int kQB = kUmRows / G;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(base);
  uint64_t* kfull = bars + 0;     // [kUmKStages]
  uint64_t* kempty = bars + 4;    // [kUmKStages] completes when both groups' S products have read the tile
  uint64_t* vfull = bars + 8;     // [kUmVStages]
  uint64_t* vempty = bars + 12;   // [kUmVStages] completes when both groups' P V products have read the tile
  uint64_t* q_ready = bars + 16;  // one phase per work item: both Q tiles landed
  // per group k, one phase per tile
  uint64_t* s_full = bars + 17;   // [2] S_k computed (and, with it, every earlier product of the CTA)
  uint64_t* p_full = bars + 19;   // [2] P_k written to TMEM (and O_k rescaled)
  uint64_t* pv_done = bars + 21;  // [2] O_k += P_k V finished
  uint64_t* fin = bars + 23;
  uint64_t* mready = bars + 24;   // [8] per tile slot: the sub-tile mask below is written
  uint64_t* q_empty = bars + 32;  // one phase per work item: its S products completed, Q may be reloaded
  uint64_t* o_free = bars + 33;   // [2] one phase per work item: group k has read O_k
  uint64_t* seg_full = bars + 36;    // [kUmSegSlots] the record in the slot is written
  uint64_t* seg_empty = bars + 44;   // [kUmSegSlots] the V producer and all 8 softmax warps have read it
  uint64_t* item_full = bars + 52;   // [kUmItemSlots] the item's tile count is written
  uint64_t* item_empty = bars + 56;  // [kUmItemSlots] the MMA warp has read it
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + 512);
  int* item_tiles = reinterpret_cast<int*>(base + 516);       // [kUmItemSlots]
  uint32_t* kmask = reinterpret_cast<uint32_t*>(base + 544);  // [8] sub-tiles holding data, per tile slot
  int* seg_recs = reinterpret_cast<int*>(base + 576);         // [kUmSegSlots][8] segment records
  uint8_t* qs = base + 1024;                       // [2][Q tile]
  uint8_t* ks = qs + 2 * Cfg::kQBytes;             // [kUmKStages][K tile]
  uint8_t* vs = ks + kUmKStages * Cfg::kKvBytes;   // [kUmVStages][V tile]
  static_assert(kUmKStages <= 4 && kUmVStages <= 4, "barrier slots");
  static_assert(576 + kUmSegSlots * 32 <= 1024 && 60 * 8 <= 512, "records and barriers fit their 1 KB slot");

  // Work items are (block of kQB query tokens, KV head) pairs; this CTA takes items blockIdx.x,
  // blockIdx.x + gridDim.x, ...  Query rows, positions and lengths all fit in int32
  // (query_start_loc and context_lens are int32).
  const int rows = (int)a.rows;
  const int n_items = (rows + kQB - 1) / kQB * a.n_kv_heads;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int max_len = (int)min(a.bt_stride << a.block_shift, (int64_t)INT32_MAX);
  const int bmask = a.block_size - 1;

  if (threadIdx.x == 0) {
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
    prefetch_tensormap(&qmap);
    // one commit per tile closes a K (V) stage: it follows both groups' S (P V) products of the tile
    for (int s = 0; s < kUmKStages; ++s) {
      mbar_init(&kfull[s], 1);
      mbar_init(&kempty[s], 1);
    }
    for (int s = 0; s < kUmVStages; ++s) {
      mbar_init(&vfull[s], 1);
      mbar_init(&vempty[s], 1);
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(&s_full[k], 1);
      mbar_init(&p_full[k], 128);
      mbar_init(&pv_done[k], 1);
      mbar_init(&o_free[k], 128);
    }
    mbar_init(q_ready, 1);
    mbar_init(q_empty, 1);
    for (int k = 0; k < kUmSegSlots; ++k) {
      mbar_init(&seg_full[k], 1);
      mbar_init(&seg_empty[k], 9);  // V producer, 8 softmax warps
    }
    for (int k = 0; k < kUmItemSlots; ++k) {
      mbar_init(&item_full[k], 1);
      mbar_init(&item_empty[k], 1);
    }
    mbar_init(fin, 1);
    for (int s = 0; s < 8; ++s) mbar_init(&mready[s], 1);
    fence_barrier_init();
  }
  if (warp == 10) tmem_alloc(tmem_slot, kUmTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // S_k at columns [128k, +128) (P_k, two 16-bit values per column, in its first 64), O_k at
  // [256 + 128k, +D)
  auto tS = [&](int k) { return tmem + 128u * (uint32_t)k; };
  auto tO = [&](int k) { return tmem + 256u + 128u * (uint32_t)k; };

  struct Seg {
    int b;
    int seg1, n, pos0, q0, kv_end;
    bool ok;
  };
  // the rows [t, seg1) of rows [t, T1) that belong to sequence b (query rows [q0, q1), context
  // length n), which holds row t
  auto make_seg = [&](int t, int T1, int b, int q0, int q1, int n) -> Seg {
    Seg sg;
    sg.b = b;
    sg.seg1 = min(q1, T1);
    if (sg.seg1 <= t) sg.seg1 = t + 1;
    sg.ok = q0 <= t && t < q1 && (int64_t)n >= (int64_t)q1 - q0 && n <= max_len;
    if (!sg.ok) n = 0;
    sg.n = n;
    sg.q0 = q0;
    sg.pos0 = n - (q1 - q0);
    sg.kv_end = sg.ok ? sg.pos0 + (sg.seg1 - 1 - q0) + 1 : 0;
    return sg;
  };
  auto tiles_of = [](const Seg& sg) -> int { return (sg.kv_end + kUmKeys - 1) / kUmKeys; };
  // Segment record idx of the K producer's stream, read by the whole warp, which then releases the
  // slot (every reader releases a record as soon as it has read it, so the ring never holds up a
  // reader the K producer waits for).  ok = false: the wait gave up (nothing is read).
  auto seg_take = [&](int idx, bool& ok) -> Seg {
    const int slot = idx % kUmSegSlots;
    Seg sg{};
    ok = __all_sync(0xffffffffu, mbar_wait(&seg_full[slot], (unsigned)((idx / kUmSegSlots) & 1), a.err, a.epoch));
    if (ok) {
      const int* rec = seg_recs + 8 * slot;
      sg.b = rec[0];
      sg.seg1 = rec[1];
      sg.n = rec[2];
      sg.pos0 = rec[3];
      sg.q0 = rec[4];
      sg.kv_end = rec[5];
      sg.ok = rec[6] != 0;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&seg_empty[slot]);
    return sg;
  };

  if (warp == 8 || warp == 9) {
    // ------- producers: warp 8 streams K tiles; warp 9 each item's Q tiles, then its V tiles -------
    // Each runs on lane 0 alone: a warp whose lanes meet at warp-collective steps between long
    // single-lane stretches was measured to lose about a thousand cycles per meeting at item
    // boundaries, so nothing here needs the other lanes.
    if (lane == 0) {
      const bool is_v = warp == 9;
      uint64_t* full = is_v ? vfull : kfull;
      uint64_t* empty = is_v ? vempty : kempty;
      uint8_t* ring = is_v ? vs : ks;
      const CUtensorMap* map = is_v ? &vmap : &kmap;
      const int depth = is_v ? kUmVStages : kUmKStages;
      int i = 0;      // tiles issued, counted over all items of the CTA
      int nq = 0;     // Q loads issued
      int rec = 0;    // segment records written (K) or read (V)
      int nit = 0;    // item tile counts written (K)
      bool alive = true;
      // the segment of rows [t, T1) holding row t, looked up now
      auto seg_lookup = [&](int t, int T1) -> Seg {
        const int b = find_sequence_8(a.query_start_loc, a.batch, t);
        return make_seg(t, T1, b, ld_nc_s32(a.query_start_loc + b), ld_nc_s32(a.query_start_loc + b + 1),
                        ld_nc_s32(a.context_lens + b));
      };
      // K producer: the lookup of the next item's first segment runs one step per K tile of the
      // current item (a round of 8 loads of the search over query_start_loc, then the loads of the
      // sequence's bounds and length), each step's loads used by the next step, so that their
      // latency passes while the warp waits for ring slots.  la_stage: 0 idle, 1 a search round in
      // flight, 2 the final loads in flight, 3 done (la_seg holds the result).
      int la_stage = 0, la_t = 0, la_T1 = 0, la_lo = 0, la_n = 0;
      int la_v[8];
      Seg la_seg{};
      auto la_issue = [&]() {
        if (la_n > 1) {
          const int step = (la_n + 7) >> 3;
#pragma unroll
          for (int k = 0; k < 8; ++k)
            la_v[k] = k * step < la_n ? ld_nc_s32(a.query_start_loc + la_lo + k * step) : INT32_MAX;
          la_stage = 1;
        } else {
          la_v[0] = ld_nc_s32(a.query_start_loc + la_lo);
          la_v[1] = ld_nc_s32(a.query_start_loc + la_lo + 1);
          la_v[2] = ld_nc_s32(a.context_lens + la_lo);
          la_stage = 2;
        }
      };
      auto la_advance = [&]() {
        if (la_stage == 1) {
          const int step = (la_n + 7) >> 3;
          int top = 0;
#pragma unroll
          for (int k = 1; k < 8; ++k)
            if (k * step < la_n && la_v[k] <= la_t) top = k;
          const int nlo = la_lo + top * step;
          la_n = min(step, la_lo + la_n - nlo);
          la_lo = nlo;
          la_issue();
        } else if (la_stage == 2) {
          la_seg = make_seg(la_t, la_T1, la_lo, la_v[0], la_v[1], la_v[2]);
          la_stage = 3;
        }
      };
      for (int w = blockIdx.x; w < n_items && alive; w += gridDim.x) {
        const int kvh = w % a.n_kv_heads;
        const int T0 = w / a.n_kv_heads * kQB;
        const int T1 = min(T0 + kQB, rows);
        if (is_v) {
          // both Q tiles of the item, once every S product of the previous item has completed; the
          // CTA's next item's Q tiles are prefetched into L2 meanwhile
          if (nq > 0 && !mbar_wait(q_empty, (unsigned)((nq - 1) & 1), a.err, a.epoch)) {
            alive = false;
            break;
          }
          mbar_arrive_expect_tx(q_ready, 2 * Cfg::kQBytes);
#pragma unroll
          for (int k = 0; k < 2; ++k)
#pragma unroll
            for (int h = 0; h < kHalves; ++h)
              tma_load_3d(qs + k * Cfg::kQBytes + h * Cfg::kQHalf, &qmap, h * 64, kvh * G,
                          T0 + k * (kUmTileRows / G), q_ready);
          const int wn = w + (int)gridDim.x;
          if (wn < n_items) {
            const int kvh_n = wn % a.n_kv_heads;
            const int T0_n = wn / a.n_kv_heads * kQB;
#pragma unroll
            for (int k = 0; k < 2; ++k)
#pragma unroll
              for (int h = 0; h < kHalves; ++h)
                tma_prefetch_3d(&qmap, h * 64, kvh_n * G, T0_n + k * (kUmTileRows / G));
          }
          ++nq;
        }
        Seg first{};
        if (!is_v) {
          // the item's segments: first its tile count for the MMA warp (the first segment was
          // looked up during the previous item)
          if (la_stage != 0 && la_t == T0) {
            while (la_stage != 3) la_advance();
            first = la_seg;
          } else {
            first = seg_lookup(T0, T1);
          }
          la_stage = 0;
          int n_all = tiles_of(first);
          for (int t = first.seg1; t < T1;) {
            const Seg sg = seg_lookup(t, T1);
            n_all += tiles_of(sg);
            t = sg.seg1;
          }
          const int slot = nit % kUmItemSlots;
          if (nit >= kUmItemSlots &&
              !mbar_wait(&item_empty[slot], (unsigned)((nit / kUmItemSlots - 1) & 1), a.err, a.epoch)) {
            alive = false;
            break;
          }
          item_tiles[slot] = n_all;
          mbar_arrive(&item_full[slot]);
          ++nit;
          const int wn = w + (int)gridDim.x;
          if (wn < n_items) {
            la_t = wn / a.n_kv_heads * kQB;
            la_T1 = min(la_t + kQB, rows);
            la_lo = 0;
            la_n = a.batch;
            la_issue();
          }
        }
        for (int t = T0; t < T1 && alive;) {
          Seg sg;
          const int slot = rec % kUmSegSlots;
          if (is_v) {
            if (!mbar_wait(&seg_full[slot], (unsigned)((rec / kUmSegSlots) & 1), a.err, a.epoch)) {
              alive = false;
              break;
            }
            const int* r = seg_recs + 8 * slot;
            sg.b = r[0];
            sg.seg1 = r[1];
            sg.n = r[2];
            sg.pos0 = r[3];
            sg.q0 = r[4];
            sg.kv_end = r[5];
            sg.ok = r[6] != 0;
            mbar_arrive(&seg_empty[slot]);
          } else {
            // then each segment's record, for the V producer and the softmax groups
            sg = t == T0 ? first : seg_lookup(t, T1);
            if (rec >= kUmSegSlots &&
                !mbar_wait(&seg_empty[slot], (unsigned)((rec / kUmSegSlots - 1) & 1), a.err, a.epoch)) {
              alive = false;
              break;
            }
            int* r = seg_recs + 8 * slot;
            r[0] = sg.b;
            r[1] = sg.seg1;
            r[2] = sg.n;
            r[3] = sg.pos0;
            r[4] = sg.q0;
            r[5] = sg.kv_end;
            r[6] = sg.ok ? 1 : 0;
            mbar_arrive(&seg_full[slot]);
          }
          ++rec;
          const int32_t* table = a.block_table + (int64_t)sg.b * a.bt_stride;
          const int nt = tiles_of(sg);
          // the table entries of a tile's 16-key sub-tiles (-1: past the segment's keys), read one
          // tile ahead so that their latency passes during the wait for the ring slot
          int ys[kUmSub];
          auto table_of = [&](int tile, int (&dst)[kUmSub]) {
#pragma unroll
            for (int sub = 0; sub < kUmSub; ++sub) {
              const int k0 = tile * kUmKeys + sub * 16;
              dst[sub] = k0 < sg.kv_end ? ld_nc_s32(table + (k0 >> a.block_shift)) : -1;
            }
          };
          if (nt > 0) table_of(0, ys);
          for (int tile = 0; tile < nt; ++tile, ++i) {
            int ys_next[kUmSub];
            if (tile + 1 < nt) table_of(tile + 1, ys_next);
            const int s = i % depth;
            const int round = i / depth;
            if (round > 0 && !mbar_wait(&empty[s], (unsigned)((round - 1) & 1), a.err, a.epoch)) {
              alive = false;
              break;
            }
            unsigned m = 0;
#pragma unroll
            for (int sub = 0; sub < kUmSub; ++sub) {
              const int k0 = tile * kUmKeys + sub * 16;
              if (k0 < sg.kv_end) {
                if (ys[sub] < 0 || ys[sub] >= a.num_blocks) {
                  if (!is_v) raise_error(a.err, PA_DEVERR_BLOCK_ID);
                } else {
                  m |= 1u << sub;
                }
              }
            }
            if (!is_v) {
              // publish which sub-tiles hold data; the softmax groups read it instead of the
              // table.  Slot i % 8 was last read for tile i - 8, which both groups finished long
              // ago: K tile i is loaded only after both S products of tile i - kUmKStages
              // completed, which needed each group's P of tile i - kUmKStages - 1.
              kmask[i & 7] = m;
              mbar_arrive(&mready[i & 7]);
            }
            uint8_t* st = ring + s * Cfg::kKvBytes;
            if (m == 0) {
              mbar_arrive(&full[s]);
            } else {
              mbar_arrive_expect_tx(&full[s], (uint32_t)__popc(m) * kHalves * 2048u);
#pragma unroll
              for (int sub = 0; sub < kUmSub; ++sub) {
                if (!((m >> sub) & 1u)) continue;
                const int yo = (tile * kUmKeys + sub * 16) & bmask;
#pragma unroll
                for (int h = 0; h < kHalves; ++h)
                  tma_load_3d(st + h * Cfg::kKvHalf + sub * 2048, map, kvh * D + h * 64, yo, ys[sub], &full[s]);
              }
            }
            if (!is_v) la_advance();
#pragma unroll
            for (int sub = 0; sub < kUmSub; ++sub) ys[sub] = ys_next[sub];
          }
          t = sg.seg1;
        }
      }
      if (!alive) raise_timeout(a.err, a.epoch);
      // Leave no copy in flight: after a normal run every issued tile was consumed and these waits
      // return at once; after a timeout elsewhere they wait (bounded) for this ring's last tiles.
      for (int k = i > depth ? i - depth : 0; k < i; ++k) mbar_wait(&full[k % depth], (unsigned)((k / depth) & 1));
      if (nq > 0) mbar_wait(q_ready, (unsigned)((nq - 1) & 1));
    }
  } else if (warp == 10) {
    // ------------------------------------------ MMA ---------------------------------------------
    const uint32_t id_s = umma_idesc_f16(kBf16, 128, kUmKeys, false, false);
    const uint32_t id_pv = umma_idesc_f16(kBf16, 128, D, false, true);
    auto issue_s = [&](int k, int g) {
      const uint32_t qa = smem_u32(qs + k * Cfg::kQBytes);
      const uint32_t ka = smem_u32(ks + (g % kUmKStages) * Cfg::kKvBytes);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t qo = (kk >> 2) * Cfg::kQHalf + (kk & 3) * 32;
        const uint32_t ko = (kk >> 2) * Cfg::kKvHalf + (kk & 3) * 32;
        umma_ss(tS(k), umma_desc_sw128(qa + qo, 16, 1024), umma_desc_sw128(ka + ko, 16, 1024), id_s,
                kk > 0 ? 1u : 0u);
      }
      umma_commit(&s_full[k]);
    };
    auto issue_pv = [&](int k, int g, bool first) {
      const uint32_t va = smem_u32(vs + (g % kUmVStages) * Cfg::kKvBytes);
      // A = P_k from TMEM: 16 keys = 8 columns per instruction; an item's first tile starts O_k
#pragma unroll
      for (int kk = 0; kk < kUmKeys / 16; ++kk)
        umma_ts(tO(k), tS(k) + 8u * (uint32_t)kk, umma_desc_sw128(va + kk * 2048, Cfg::kKvHalf, 1024), id_pv,
                (!first || kk > 0) ? 1u : 0u);
      umma_commit(&pv_done[k]);
    };
    // lane 0 alone issues (no warp-collective step, as for the producers)
    int g = 0;  // tiles of earlier items
    int n = 0;  // items done
    bool alive = lane == 0;
    for (int w = blockIdx.x; w < n_items && alive; w += gridDim.x, ++n) {
      // the item's tile count, from the K producer
      int n_all = 0;
      bool ok = true;
      {
        const int slot = n % kUmItemSlots;
        ok = mbar_wait(&item_full[slot], (unsigned)((n / kUmItemSlots) & 1), a.err, a.epoch);
        if (ok) n_all = item_tiles[slot];
        mbar_arrive(&item_empty[slot]);
      }
      if (ok) {
        auto wait = [&](uint64_t* bar, unsigned parity) {
          ok = ok && mbar_wait(bar, parity, a.err, a.epoch);
          return ok;
        };
        // the item's first P V into O_k waits until group k has read O_k of the previous item
        bool o_ready[2] = {n == 0, n == 0};
        auto own_o = [&](int k) {
          if (!o_ready[k]) {
            o_ready[k] = true;
            return wait(&o_free[k], (unsigned)((n - 1) & 1));
          }
          return ok;
        };
        // O_k += P_k V of item tile j; group 1's product closes the V tile
        auto pv_of = [&](int k, int j) {
          const int gj = g + j;
          if (!own_o(k) || !wait(&p_full[k], (unsigned)(gj & 1)) ||
              !wait(&vfull[gj % kUmVStages], (unsigned)((gj / kUmVStages) & 1)))
            return false;
          tc_fence_after();
          issue_pv(k, gj, j == 0);
          if (k == 1) umma_commit(&vempty[gj % kUmVStages]);
          return true;
        };
        // Fixed issue order per tile: S_0(j), P_1(j-1) V, S_1(j), P_0(j) V.  While group 0 turns
        // S_0(j) into P_0(j) the tensor core runs group 1's P V and next S, and the other way round.
        // S_k overwrites the previous tile's P_k (also across items), so it waits for that P V.
        wait(q_ready, (unsigned)(n & 1));
        for (int j = 0; j < n_all && ok; ++j) {
          const int gj = g + j;
          if (!wait(&kfull[gj % kUmKStages], (unsigned)((gj / kUmKStages) & 1))) break;
          tc_fence_after();
          issue_s(0, gj);
          if (j > 0 && !pv_of(1, j - 1)) break;
          tc_fence_after();
          issue_s(1, gj);
          umma_commit(&kempty[gj % kUmKStages]);
          if (j == n_all - 1) umma_commit(q_empty);  // after the item's last S products
          if (!pv_of(0, j)) break;
        }
        if (ok && n_all > 0) pv_of(1, n_all - 1);
        if (ok && n_all == 0) umma_commit(q_empty);
        own_o(0);  // an item without tiles still takes its turn of both O buffers
        own_o(1);
      }
      alive = ok;
      g += n_all;
    }
    if (lane == 0) {
      if (!alive) raise_timeout(a.err, a.epoch);
      if (g > 0) {
        umma_commit(fin);
        mbar_wait(fin, 0, a.err, a.epoch);
      }
    }
  } else {
    // --------------------------------------- softmax groups ---------------------------------------
    const int grp = warp >> 2;           // 0 or 1
    const int r = threadIdx.x & 127;     // row inside the Q tile = TMEM lane
    const int row = grp * kUmTileRows + r;
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    int i = 0;    // tiles of this CTA so far
    int rec = 0;  // segment records read
    bool alive = true;
    for (int w = blockIdx.x; w < n_items && alive; w += gridDim.x) {
      const int kvh = w % a.n_kv_heads;
      const int T0 = w / a.n_kv_heads * kQB;
      const int T1 = min(T0 + kQB, rows);
      const int tok = T0 + row / G;
      const int head = kvh * G + row % G;
      const int i0 = i;
      float m_use = -INFINITY;  // stabilising maximum (log2 domain) the exponentials are taken against
      float l_run = 0.f;
      for (int t = T0; t < T1 && alive;) {
        bool got = true;
        const Seg sg = seg_take(rec++, got);
        if (!got) {
          alive = false;
          break;
        }
        if (!sg.ok && threadIdx.x == 0) raise_error(a.err, PA_DEVERR_QUERY_LOC);
        const int bound = (sg.ok && tok >= t && tok < sg.seg1) ? sg.pos0 + (tok - sg.q0) : -1;
        const int nt = tiles_of(sg);
        for (int tile = 0; tile < nt; ++tile, ++i) {
          const int kb = tile * kUmKeys;
          if (!__all_sync(0xffffffffu, mbar_wait(&mready[i & 7], (unsigned)((i >> 3) & 1), a.err, a.epoch))) {
            alive = false;
            break;
          }
          const unsigned loaded = kmask[i & 7];
          // S_k of this tile is complete, and with it O_k += P_k V of the previous tile (issued before)
          if (!__all_sync(0xffffffffu, mbar_wait(&s_full[grp], (unsigned)(i & 1), a.err, a.epoch))) {
            alive = false;
            break;
          }
          tc_fence_after();
          // tiles wholly inside every row's causal bound of the warp, with every sub-tile loaded,
          // need no mask (the common case); the others mask per 32-key chunk
          const float sc = a.scale_log2;
          const unsigned all_sub = (1u << kUmSub) - 1u;
          const bool unmasked = __all_sync(0xffffffffu, loaded == all_sub && kb + kUmKeys - 1 <= bound);
          uint32_t mask[kUmKeys / 32];
          {
            const int lim = bound - kb;  // keys c <= lim are causal
            const int nv = lim < 0 ? 0 : (lim >= kUmKeys ? kUmKeys : lim + 1);
#pragma unroll
            for (int q = 0; q < kUmKeys / 32; ++q) {
              const int lo = 32 * q;
              const uint32_t cm = nv >= lo + 32 ? 0xFFFFFFFFu : (nv <= lo ? 0u : ((1u << (nv - lo)) - 1u));
              const uint32_t lm = (((loaded >> (2 * q)) & 1u) ? 0x0000FFFFu : 0u) |
                                  (((loaded >> (2 * q + 1)) & 1u) ? 0xFFFF0000u : 0u);
              mask[q] = cm & lm;
            }
          }
          const uint32_t srow = tS(grp) + lane_base;
          ScoreFix fix;
          {
            const int lim = bound - kb;  // keys c <= lim are causal
            const int nvc = lim < 0 ? 0 : (lim >= kUmKeys ? kUmKeys : lim + 1);
            const int nvl = 16 * __popc(loaded);
            const bool prefix = (loaded & (loaded + 1u)) == 0u;  // the loaded sub-tiles are 0 .. k-1
            fix.mode = (unmasked && sc > 0.f) ? 0 : ((prefix && sc > 0.f) ? 1 : 2);
            fix.nv = nvc < nvl ? nvc : nvl;
            fix.flip = sc < 0.f ? 0x80000000u : 0u;
            fix.zero = sc == 0.f;
          }
          const float sc_pos = sc > 0.f ? sc : (sc < 0.f ? -sc : 1.f);
          const float corr = fix.mode == 0   ? row_softmax<kBf16, 0>(srow, sc_pos, fix, mask, m_use, l_run)
                             : fix.mode == 1 ? row_softmax<kBf16, 1>(srow, sc_pos, fix, mask, m_use, l_run)
                                             : row_softmax<kBf16, 2>(srow, sc_pos, fix, mask, m_use, l_run);
          // O_k is stable here (its last product completed before this S_k was issued); the item's
          // first tile starts O_k afresh, so only later tiles rescale it
          if (i > i0 && __any_sync(0xffffffffu, corr != 1.f)) {
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
              uint32_t v[32];
              tmem_ld32_sync(tO(grp) + lane_base + c0, v);
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * corr);
              tmem_st32(tO(grp) + lane_base + c0, v);
            }
          }
          // group 0 zeroes V rows that hold no data or lie past the context (group 1's P V is issued
          // after group 0's, so it sees the zeros too)
          if (grp == 0 && (kb + kUmKeys > sg.n || loaded != all_sub)) {
            if (!__all_sync(0xffffffffu, mbar_wait(&vfull[i % kUmVStages], (unsigned)((i / kUmVStages) & 1), a.err, a.epoch))) {
              alive = false;
              break;
            }
            uint8_t* vst = vs + (i % kUmVStages) * Cfg::kKvBytes;
            for (int e = r; e < kUmKeys * 8 * kHalves; e += 128) {
              const int key = e / (8 * kHalves);
              const int c = e % (8 * kHalves);
              if (kb + key >= sg.n || !((loaded >> (key >> 4)) & 1u))
                *reinterpret_cast<uint4*>(vst + sw_off(key, c, Cfg::kKvHalf)) = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
          }
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(&p_full[grp]);
        }
        t = sg.seg1;
      }
      if (!alive && lane == 0) raise_timeout(a.err, a.epoch);
      if (alive && i > i0) {
        alive = __all_sync(0xffffffffu, mbar_wait(&pv_done[grp], (unsigned)((i - 1) & 1), a.err, a.epoch));
        tc_fence_after();
      }
      const bool have = alive && i > i0 && l_run != 0.f;
      const float inv = have ? 1.f / l_run : 0.f;
      T* orow = static_cast<T*>(a.out) + ((int64_t)tok * a.n_q_heads + head) * D;
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t v[32];
        tmem_ld32_sync(tO(grp) + lane_base + c0, v);
        if (tok < T1) {
#pragma unroll
          for (int j = 0; j < 32; j += 8) {
            float f[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = have ? __uint_as_float(v[j + e]) * inv : 0.f;
            uint4 wv;
            wv.x = pack2<kBf16>(f[0], f[1]);
            wv.y = pack2<kBf16>(f[2], f[3]);
            wv.z = pack2<kBf16>(f[4], f[5]);
            wv.w = pack2<kBf16>(f[6], f[7]);
            *reinterpret_cast<uint4*>(orow + c0 + j) = wv;
          }
        }
      }
      // O_k has been read: the next item's first P V may overwrite it
      tc_fence_before();
      mbar_arrive(&o_free[grp]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 10) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kUmTmemCols);
  }
}

// ------------------------------------------------------------------------------------------------

template <typename T, int D, int G>
static cudaError_t launch_um_g(const AttnArgs& a, const CUtensorMap& km, const CUtensorMap& vm, cudaStream_t s) {
  CUtensorMap qm;
  if (!encode_q_map(&qm, a.q, std::is_same<T, __nv_bfloat16>::value ? PA_BF16 : PA_FP16, a.rows, a.n_q_heads, D, G,
                    kUmTileRows / G))
    return cudaErrorInvalidValue;
  constexpr int smem = UmCfg<D>::kSmemBytes;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(prefill_umma_kernel<T, D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  constexpr int qb = kUmRows / G;
  const int64_t items = ((a.rows + qb - 1) / qb) * a.n_kv_heads;
  if (items <= 0) return cudaSuccess;
  if (items > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  // persistent: one CTA per SM walks the work items, so the next item's loads overlap this one's end
  static int sm_count[64] = {};
  int sms = dev >= 0 && dev < 64 ? sm_count[dev] : 0;
  if (sms == 0) {
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) sm_count[dev] = sms;
  }
  const int64_t grid = std::min<int64_t>(items, sms);
  prefill_umma_kernel<T, D, G><<<(unsigned)grid, kUmThreads, smem, s>>>(a, km, vm, qm);
  return cudaGetLastError();
}

template <typename T, int D>
static cudaError_t launch_um_d(const AttnArgs& a, const CUtensorMap& km, const CUtensorMap& vm, cudaStream_t s) {
  switch (a.group) {
    case 1: return launch_um_g<T, D, 1>(a, km, vm, s);
    case 2: return launch_um_g<T, D, 2>(a, km, vm, s);
    case 4: return launch_um_g<T, D, 4>(a, km, vm, s);
    case 8: return launch_um_g<T, D, 8>(a, km, vm, s);
    case 16: return launch_um_g<T, D, 16>(a, km, vm, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_prefill_umma(const AttnArgs& a, pa_dtype dt, cudaStream_t s, int* launches) {
  if (a.rows == 0) return cudaSuccess;
  CUtensorMap km, vm;
  if (!encode_pool_map(&km, a.k_pool, dt, a.num_blocks, a.block_size, a.n_kv_heads, a.head_dim, a.kv_block_stride) ||
      !encode_pool_map(&vm, a.v_pool, dt, a.num_blocks, a.block_size, a.n_kv_heads, a.head_dim, a.kv_block_stride))
    return cudaErrorInvalidValue;
  cudaError_t e;
  if (dt == PA_BF16)
    e = a.head_dim == 64 ? launch_um_d<__nv_bfloat16, 64>(a, km, vm, s) : launch_um_d<__nv_bfloat16, 128>(a, km, vm, s);
  else
    e = a.head_dim == 64 ? launch_um_d<__half, 64>(a, km, vm, s) : launch_um_d<__half, 128>(a, km, vm, s);
  ++*launches;
  return e;
}

}  // namespace pa
