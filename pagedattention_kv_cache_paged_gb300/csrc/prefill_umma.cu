// tcgen05 causal chunked prefill over a paged history (bf16/fp16, block_size % 16 == 0).
//
// Computes the same thing as prefill_tc.cu — JuliaPagedAttn README "Features" (batched prefill)
// with the online softmax of "Online Softmax": the chunk of m_b queries holds the last m_b
// positions of sequence b's context and query r attends to positions 0 .. n_b - m_b + r through
// the block table — on the 5th-generation tensor cores with accumulators in tensor memory.
//
// CTA = 256 (query token, head) rows of one KV head, split into two 128-row Q tiles that share
// every K/V tile (kRows / G tokens x the G heads of the group: read-time GQA, nanoserve Day 19
// "What I learned" 4).  10 warps:
//   warps 0-3 / 4-7  softmax groups 0 / 1: thread t of group k owns row 128k + t (TMEM lane t of
//              S_k and O_k); stages its Q row, turns each S_k tile into probabilities, rescales O_k
//              in TMEM only when its stabilising maximum has to move up by more than 2^8, writes
//              P_k (bf16/fp16) back into the TMEM columns of S_k, and normalises O_k at the end;
//   warp 8     producer: lane 0 streams 128-key K tiles, lane 1 the matching V tiles (TMA boxes
//              of 16 keys x 64 columns from the physical blocks the table names) into 2-stage
//              rings;
//   warp 9     MMA: allocates TMEM (S_0, S_1: 128 columns each; O_0, O_1: 128 columns each) and
//              issues S_k = Q_k K^T (M 128, N 128, both operands in shared memory) and
//              O_k += P_k V (M 128, N head_dim, P read from TMEM, V an MN-major shared-memory
//              operand) with tcgen05.mma as soon as each product's inputs are ready, so that the
//              tensor core works on one group's products while the other group computes its
//              softmax.  S_k of the next tile is issued only after O_k += P_k V of this one has
//              completed, because P_k lives in the columns the next S_k overwrites; that same
//              ordering makes O_k stable whenever a group sees a new S_k, so rescaling needs no
//              extra wait.
// Every mbarrier wait is bounded (PA_DEVERR_TIMEOUT, with a cooperative abort); TMEM is always
// released.  The stabilising maximum is exact bookkeeping: numerator and denominator use the
// same one, so the result equals the running-max form of "Online Softmax" in real arithmetic.
#include <cudaTypedefs.h>

#include "pa_common.cuh"
#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {

constexpr int kUmThreads = 320;
constexpr int kUmTileRows = 128;            // rows per Q tile (MMA M)
constexpr int kUmRows = 2 * kUmTileRows;    // rows per CTA
constexpr int kUmKeys = 128;                // keys per K/V tile (N of S, K of PV)
constexpr int kUmSub = kUmKeys / 16;
constexpr int kUmTmemCols = 512;
constexpr int kUmKStages = 2;               // K ring depth
constexpr int kUmVStages = 2;               // V ring depth
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
// Keys whose bit is clear in mask[q] (chunk q = columns 32q .. 32q + 31) are outside the causal
// bound or were not loaded; kMasked = false is the common case of a tile with every key valid.

// Row maximum of the scaled scores.
template <bool kMasked>
__device__ __forceinline__ float s_row_max(uint32_t taddr, float sc, const uint32_t (&mask)[kUmKeys / 32]) {
  float m[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
  for (int q = 0; q < kUmKeys / 32; ++q) {
    uint32_t v[32];
    tmem_ld32(taddr + 32u * q, v);
    tmem_wait_ld();
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      float x = __uint_as_float(v[j]) * sc;
      if (kMasked) x = (mask[q] & (1u << j)) ? x : -INFINITY;
      m[j & 3] = fmaxf(m[j & 3], x);
    }
  }
  return fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3]));
}

// Probabilities 2^(sc * s - m_sub) (0 for masked keys), written back as 16-bit pairs into the first
// kUmKeys / 2 columns of the row (keys 2c and 2c + 1 in column c); returns their sum.  Columns
// [32 h, 32 h + 32) of P hold keys [64 h, 64 h + 64), which are read before they are overwritten.
template <bool kMasked, bool kBf16>
__device__ __forceinline__ float p_row_store(uint32_t taddr, float sc, float m_sub,
                                             const uint32_t (&mask)[kUmKeys / 32]) {
  static_assert(kUmKeys == 128, "two halves of 64 keys");
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1  // one half at a time keeps the register footprint at one chunk in, one chunk out
  for (int h = 0; h < 2; ++h) {
    uint32_t w[32];
#pragma unroll
    for (int q2 = 0; q2 < 2; ++q2) {
      const int q = 2 * h + q2;
      const uint32_t mq = h == 0 ? mask[q2] : mask[2 + q2];
      uint32_t v[32];
      tmem_ld32(taddr + 32u * q, v);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        float e0 = fast_exp2(fmaf(__uint_as_float(v[j]), sc, -m_sub));
        float e1 = fast_exp2(fmaf(__uint_as_float(v[j + 1]), sc, -m_sub));
        if (kMasked) {
          e0 = (mq & (1u << j)) ? e0 : 0.f;
          e1 = (mq & (2u << j)) ? e1 : 0.f;
        }
        acc[j & 3] += e0;
        acc[(j + 1) & 3] += e1;
        w[16 * q2 + j / 2] = pack2<kBf16>(e0, e1);
      }
    }
    tmem_st32(taddr + 32u * h, w);
  }
  return (acc[0] + acc[1]) + (acc[2] + acc[3]);
}

template <typename T, int D, int G>
__global__ void __launch_bounds__(kUmThreads, 1)
    prefill_umma_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap) {
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
  uint64_t* q_ready = bars + 16;
  // per group k, one phase per tile
  uint64_t* s_full = bars + 17;   // [2] S_k computed (and, with it, every earlier product of the CTA)
  uint64_t* p_full = bars + 19;   // [2] P_k written to TMEM (and O_k rescaled)
  uint64_t* pv_done = bars + 21;  // [2] O_k += P_k V finished
  uint64_t* fin = bars + 23;
  uint64_t* mready = bars + 24;   // [8] per tile slot: the sub-tile mask below is written
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + 512);
  uint32_t* kmask = reinterpret_cast<uint32_t*>(base + 768);  // [8] sub-tiles holding data, per tile slot
  uint8_t* qs = base + 1024;                       // [2][Q tile]
  uint8_t* ks = qs + 2 * Cfg::kQBytes;             // [3 stages][K tile]
  uint8_t* vs = ks + kUmKStages * Cfg::kKvBytes;   // [2 stages][V tile]

  const int kvh = blockIdx.x % a.n_kv_heads;
  const int64_t T0 = (int64_t)(blockIdx.x / a.n_kv_heads) * kQB;
  const int64_t T1 = min(T0 + kQB, a.rows);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t max_len = a.bt_stride << a.block_shift;
  const int bmask = a.block_size - 1;

  if (threadIdx.x == 0) {
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
    for (int s = 0; s < kUmKStages; ++s) {
      mbar_init(&kfull[s], 1);
      mbar_init(&kempty[s], 2);
    }
    for (int s = 0; s < kUmVStages; ++s) {
      mbar_init(&vfull[s], 1);
      mbar_init(&vempty[s], 2);
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(&s_full[k], 1);
      mbar_init(&p_full[k], 128);
      mbar_init(&pv_done[k], 1);
    }
    mbar_init(q_ready, 256);
    mbar_init(fin, 1);
    for (int s = 0; s < 8; ++s) mbar_init(&mready[s], 1);
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 9) tmem_alloc(tmem_slot, kUmTmemCols);
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
    int64_t seg1, n, pos0, q0, kv_end;
    bool ok;
  };
  auto segment_at = [&](int64_t t) -> Seg {
    Seg sg;
    const int b = find_sequence(a.query_start_loc, a.batch, t);
    const int64_t q0 = __ldg(a.query_start_loc + b);
    const int64_t q1 = __ldg(a.query_start_loc + b + 1);
    int64_t n = __ldg(a.context_lens + b);
    sg.b = b;
    sg.seg1 = min(q1, T1);
    if (sg.seg1 <= t) sg.seg1 = t + 1;
    sg.ok = q0 <= t && t < q1 && n >= q1 - q0 && n <= max_len;
    if (!sg.ok) n = 0;
    sg.n = n;
    sg.q0 = q0;
    sg.pos0 = n - (q1 - q0);
    sg.kv_end = sg.ok ? sg.pos0 + (sg.seg1 - 1 - q0) + 1 : 0;
    return sg;
  };
  auto tiles_of = [](const Seg& sg) -> int { return (int)((sg.kv_end + kUmKeys - 1) / kUmKeys); };

  if (warp == 8) {
    // --------------------------- producer: lane 0 -> K tiles, lane 1 -> V tiles --------------------
    if (lane < 2) {
      const bool is_v = lane == 1;
      uint64_t* full = is_v ? vfull : kfull;
      uint64_t* empty = is_v ? vempty : kempty;
      uint8_t* ring = is_v ? vs : ks;
      const CUtensorMap* map = is_v ? &vmap : &kmap;
      const int depth = is_v ? kUmVStages : kUmKStages;
      int i = 0;
      bool alive = true;
      for (int64_t t = T0; t < T1 && alive;) {
        const Seg sg = segment_at(t);
        const int32_t* table = a.block_table + (int64_t)sg.b * a.bt_stride;
        const int nt = tiles_of(sg);
        for (int tile = 0; tile < nt; ++tile, ++i) {
          const int s = i % depth;
          const int round = i / depth;
          if (round > 0 && !mbar_wait(&empty[s], (unsigned)((round - 1) & 1), a.err)) {
            raise_error(a.err, PA_DEVERR_TIMEOUT);
            alive = false;
            break;
          }
          int ys[kUmSub], yo[kUmSub];
          uint32_t bytes = 0;
#pragma unroll
          for (int sub = 0; sub < kUmSub; ++sub) {
            const int64_t k0 = (int64_t)tile * kUmKeys + sub * 16;
            ys[sub] = -1;
            if (k0 < sg.kv_end) {
              const int blk = __ldg(table + (k0 >> a.block_shift));
              if (blk < 0 || blk >= a.num_blocks) {
                if (!is_v) raise_error(a.err, PA_DEVERR_BLOCK_ID);
              } else {
                ys[sub] = blk;
                yo[sub] = (int)(k0 & bmask);
                bytes += kHalves * 2048;
              }
            }
          }
          if (!is_v) {
            // publish which sub-tiles hold data; the softmax groups read it instead of the table.
            // Slot i % 8 was last read for tile i - 8, which both groups finished long ago: K tile
            // i is loaded only after both S products of tile i - 2 completed, which needed each
            // group's P of tile i - 3.
            unsigned m = 0;
#pragma unroll
            for (int sub = 0; sub < kUmSub; ++sub) m |= (ys[sub] >= 0 ? 1u : 0u) << sub;
            kmask[i & 7] = m;
            mbar_arrive(&mready[i & 7]);
          }
          uint8_t* st = ring + s * Cfg::kKvBytes;
          if (bytes == 0) {
            mbar_arrive(&full[s]);
          } else {
            mbar_arrive_expect_tx(&full[s], bytes);
#pragma unroll
            for (int sub = 0; sub < kUmSub; ++sub) {
              if (ys[sub] < 0) continue;
#pragma unroll
              for (int h = 0; h < kHalves; ++h)
                tma_load_3d(st + h * Cfg::kKvHalf + sub * 2048, map, kvh * D + h * 64, yo[sub], ys[sub], &full[s]);
            }
          }
        }
        t = sg.seg1;
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------ MMA ---------------------------------------------
    if (lane == 0) {
      int n_all = 0;
      for (int64_t t = T0; t < T1;) {
        const Seg sg = segment_at(t);
        n_all += tiles_of(sg);
        t = sg.seg1;
      }
      const uint32_t id_s = umma_idesc_f16(kBf16, 128, kUmKeys, false, false);
      const uint32_t id_pv = umma_idesc_f16(kBf16, 128, D, false, true);
      auto issue_s = [&](int k, int i) {
        const uint32_t qa = smem_u32(qs + k * Cfg::kQBytes);
        const uint32_t ka = smem_u32(ks + (i % kUmKStages) * Cfg::kKvBytes);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t qo = (kk >> 2) * Cfg::kQHalf + (kk & 3) * 32;
          const uint32_t ko = (kk >> 2) * Cfg::kKvHalf + (kk & 3) * 32;
          umma_ss(tS(k), umma_desc_sw128(qa + qo, 16, 1024), umma_desc_sw128(ka + ko, 16, 1024), id_s,
                  kk > 0 ? 1u : 0u);
        }
        umma_commit(&s_full[k]);
      };
      auto issue_pv = [&](int k, int i) {
        const uint32_t va = smem_u32(vs + (i % kUmVStages) * Cfg::kKvBytes);
        // A = P_k from TMEM: 16 keys = 8 columns per instruction
#pragma unroll
        for (int kk = 0; kk < kUmKeys / 16; ++kk)
          umma_ts(tO(k), tS(k) + 8u * (uint32_t)kk, umma_desc_sw128(va + kk * 2048, Cfg::kKvHalf, 1024), id_pv,
                  (i > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&pv_done[k]);
      };
      // Event-driven issue: each group's next S (needs the K tile and its previous P V finished) and
      // next P V (needs its P and the V tile) are issued as soon as they are ready, so a slow group
      // never holds back the other group's products.
      bool alive = mbar_wait(q_ready, 0, a.err);
      int next_s[2] = {0, 0}, next_pv[2] = {0, 0};
      int idle = 0;
      while (alive && (next_pv[0] < n_all || next_pv[1] < n_all)) {
        bool progress = false;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          // S_k(j) overwrites P_k(j - 1): O_k += P_k(j - 1) V must have completed
          const int j = next_s[k];
          if (j < n_all && j == next_pv[k] && (j == 0 || mbar_test(&pv_done[k], (unsigned)((j - 1) & 1))) &&
              mbar_test(&kfull[j % kUmKStages], (unsigned)((j / kUmKStages) & 1))) {
            tc_fence_after();
            issue_s(k, j);
            umma_commit(&kempty[j % kUmKStages]);
            next_s[k] = j + 1;
            progress = true;
          }
          const int jp = next_pv[k];
          // group 1's P V follows group 0's for the same tile: group 0 zeroes the tile's stale V
          // rows before it signals p_full, and group 1 must not read them earlier
          if (jp < next_s[k] && (k == 0 || next_pv[0] > jp) && mbar_test(&p_full[k], (unsigned)(jp & 1)) &&
              mbar_test(&vfull[jp % kUmVStages], (unsigned)((jp / kUmVStages) & 1))) {
            tc_fence_after();
            issue_pv(k, jp);
            umma_commit(&vempty[jp % kUmVStages]);
            next_pv[k] = jp + 1;
            progress = true;
          }
        }
        if (progress) {
          idle = 0;
        } else if (++idle > kWaitSpins ||
                   (idle > 4096 && (*reinterpret_cast<const volatile unsigned*>(a.err) & PA_DEVERR_TIMEOUT))) {
          alive = false;
        }
      }
      if (!alive) raise_error(a.err, PA_DEVERR_TIMEOUT);
      if (n_all > 0) {
        umma_commit(fin);
        mbar_wait(fin, 0, a.err);
      }
    }
  } else {
    // --------------------------------------- softmax groups ---------------------------------------
    const int grp = warp >> 2;           // 0 or 1
    const int r = threadIdx.x & 127;     // row inside the Q tile = TMEM lane
    const int row = grp * kUmTileRows + r;
    const int64_t tok = T0 + row / G;
    const int head = kvh * G + row % G;
    uint8_t* q_tile = qs + grp * Cfg::kQBytes;
    {
      const uint4* qrow = reinterpret_cast<const uint4*>(static_cast<const T*>(a.q) + (tok * a.n_q_heads + head) * D);
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        const uint4 v = tok < T1 ? __ldg(qrow + c) : make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(q_tile + sw_off(r, c, Cfg::kQHalf)) = v;
      }
      fence_proxy_async_smem();
      mbar_arrive(q_ready);
    }
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    float m_use = -INFINITY;  // stabilising maximum (log2 domain) the exponentials are taken against
    float l_run = 0.f;
    int i = 0;
    bool alive = true;
    for (int64_t t = T0; t < T1 && alive;) {
      const Seg sg = segment_at(t);
      if (!sg.ok && threadIdx.x == 0) raise_error(a.err, PA_DEVERR_QUERY_LOC);
      const int64_t bound = (sg.ok && tok >= t && tok < sg.seg1) ? sg.pos0 + (tok - sg.q0) : -1;
      const int nt = tiles_of(sg);
      for (int tile = 0; tile < nt; ++tile, ++i) {
        const int64_t kb = (int64_t)tile * kUmKeys;
        if (!__all_sync(0xffffffffu, mbar_wait(&mready[i & 7], (unsigned)((i >> 3) & 1), a.err))) {
          alive = false;
          break;
        }
        const unsigned loaded = kmask[i & 7];
        // S_k of this tile is complete, and with it O_k += P_k V of the previous tile (issued before)
        if (!__all_sync(0xffffffffu, mbar_wait(&s_full[grp], (unsigned)(i & 1), a.err))) {
          alive = false;
          break;
        }
        tc_fence_after();
        // tiles wholly inside every row's causal bound of the warp, with every sub-tile loaded, need
        // no mask (the common case); the others mask per 32-key chunk
        const float sc = a.scale_log2;
        const unsigned all_sub = (1u << kUmSub) - 1u;
        const bool unmasked = __all_sync(0xffffffffu, loaded == all_sub && kb + kUmKeys - 1 <= bound);
        uint32_t mask[kUmKeys / 32];
        {
          const int64_t lim = bound - kb;  // keys c <= lim are causal
          const int nv = lim < 0 ? 0 : (lim >= kUmKeys ? kUmKeys : (int)lim + 1);
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
        const float mx = unmasked ? s_row_max<false>(srow, sc, mask) : s_row_max<true>(srow, sc, mask);
        // move the stabiliser only when it must: first finite maximum, or growth beyond 2^8
        float corr = 1.f;
        if (mx > m_use + kUmRescaleThreshold || (m_use == -INFINITY && mx != -INFINITY)) {
          corr = fast_exp2(m_use - mx);  // m_use = -inf -> 0
          m_use = mx;
        }
        const float m_sub = m_use == -INFINITY ? 0.f : m_use;
        const float rs = unmasked ? p_row_store<false, kBf16>(srow, sc, m_sub, mask)
                                  : p_row_store<true, kBf16>(srow, sc, m_sub, mask);
        l_run = l_run * corr + rs;
        // O_k is stable here (its last product completed before this S_k was issued)
        if (i > 0 && __any_sync(0xffffffffu, corr != 1.f)) {
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(tO(grp) + lane_base + c0, v);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * corr);
            tmem_st32(tO(grp) + lane_base + c0, v);
          }
        }
        // group 0 zeroes V rows that hold no data or lie past the context (group 1's P V is issued
        // after group 0's, so it sees the zeros too)
        if (grp == 0 && (kb + kUmKeys > sg.n || loaded != all_sub)) {
          if (!__all_sync(0xffffffffu, mbar_wait(&vfull[i % kUmVStages], (unsigned)((i / kUmVStages) & 1), a.err))) {
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
    if (!alive && lane == 0) raise_error(a.err, PA_DEVERR_TIMEOUT);
    if (alive && i > 0) {
      alive = __all_sync(0xffffffffu, mbar_wait(&pv_done[grp], (unsigned)((i - 1) & 1), a.err));
      tc_fence_after();
    }
    const bool have = alive && i > 0 && l_run != 0.f;
    const float inv = have ? 1.f / l_run : 0.f;
    T* orow = static_cast<T*>(a.out) + (tok * a.n_q_heads + head) * D;
#pragma unroll
    for (int c0 = 0; c0 < D; c0 += 32) {
      uint32_t v[32];
      tmem_ld32(tO(grp) + lane_base + c0, v);
      tmem_wait_ld();
      if (tok < T1) {
#pragma unroll
        for (int j = 0; j < 32; j += 8) {
          float f[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) f[e] = have ? __uint_as_float(v[j + e]) * inv : 0.f;
          uint4 w;
          w.x = pack2<kBf16>(f[0], f[1]);
          w.y = pack2<kBf16>(f[2], f[3]);
          w.z = pack2<kBf16>(f[4], f[5]);
          w.w = pack2<kBf16>(f[6], f[7]);
          *reinterpret_cast<uint4*>(orow + c0 + j) = w;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kUmTmemCols);
  }
}

// ------------------------------------------------------------------------------------------------

template <typename T, int D, int G>
static cudaError_t launch_um_g(const AttnArgs& a, const CUtensorMap& km, const CUtensorMap& vm, cudaStream_t s) {
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
  const int64_t grid = ((a.rows + qb - 1) / qb) * a.n_kv_heads;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  prefill_umma_kernel<T, D, G><<<(unsigned)grid, kUmThreads, smem, s>>>(a, km, vm);
  return cudaGetLastError();
}

template <typename T, int D>
static cudaError_t launch_um_d(const AttnArgs& a, const CUtensorMap& km, const CUtensorMap& vm, cudaStream_t s) {
  switch (a.group) {
    case 1: return launch_um_g<T, D, 1>(a, km, vm, s);
    case 2: return launch_um_g<T, D, 2>(a, km, vm, s);
    case 4: return launch_um_g<T, D, 4>(a, km, vm, s);
    case 8: return launch_um_g<T, D, 8>(a, km, vm, s);
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
