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
//              P_k (bf16/fp16) to shared memory, and normalises O_k at the end;
//   warp 8     producer: lane 0 streams 64-key K tiles, lane 1 the matching V tiles (TMA boxes of
//              16 keys x 64 columns from the physical blocks the table names) into a 3-stage K
//              ring and a 2-stage V ring;
//   warp 9     MMA: allocates TMEM (S_0, S_1: 64 columns each; O_0, O_1: head_dim each) and
//              issues S_k = Q_k K^T (M 128, N 64) and O_k += P_k V (M 128, N head_dim, V as an
//              MN-major operand) with tcgen05.mma, ordered so that the tensor core works on one
//              group's products while the other group computes its softmax; each group releases its S
//              as soon as it has been read out of TMEM, so the next S is computed during its
//              exponentials.
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
constexpr int kUmKeys = 64;                 // keys per K/V tile (N of S, K of PV)
constexpr int kUmSub = kUmKeys / 16;
constexpr int kUmTmemCols = 512;
constexpr int kUmKStages = 3;               // K ring depth
constexpr int kUmVStages = 3;               // V ring depth
constexpr float kUmRescaleThreshold = 8.f;  // log2 units: O is rescaled when the max grows by > 2^8

template <int D>
struct UmCfg {
  static constexpr int kHalves = D / 64;
  static constexpr int kQHalf = kUmTileRows * 128;   // one 64-column half of a Q tile
  static constexpr int kQBytes = kUmTileRows * D * 2;
  static constexpr int kKvHalf = kUmKeys * 128;      // one 64-column half of a K or V tile
  static constexpr int kKvBytes = kUmKeys * D * 2;
  static constexpr int kPBytes = kUmTileRows * kUmKeys * 2;
  static constexpr int kSmemBytes = 1024 + 1024 + 2 * kQBytes + (kUmKStages + kUmVStages) * kKvBytes + 4 * kPBytes;
};

// Byte offset of (row r, 8-element chunk c) in a [half][rows][128 B] swizzled operand.
__device__ __forceinline__ uint32_t sw_off(int r, int c, int half_bytes) {
  return (uint32_t)((c >> 3) * half_bytes + r * 128 + (((c & 7) ^ (r & 7)) << 4));
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
  uint64_t* kfull = bars + 0;     // [3]
  uint64_t* kempty = bars + 3;    // [3] completes when both groups' S products have read the tile
  uint64_t* vfull = bars + 6;     // [3]
  uint64_t* vempty = bars + 9;    // [3] completes when both groups' P V products have read the tile
  uint64_t* q_ready = bars + 12;
  // per group k and buffer b (tile j uses buffer j % 2): [2 * k + b]
  uint64_t* s_full = bars + 13;   // S_k^b computed
  uint64_t* s_free = bars + 17;   // S_k^b read out of TMEM
  uint64_t* p_full = bars + 21;   // P_k^b written (and O_k rescaled)
  uint64_t* pv_done = bars + 25;  // O_k += P_k^b V finished
  uint64_t* fin = bars + 29;
  uint64_t* mready = bars + 30;   // [8] per tile slot: the sub-tile mask below is written
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + 512);
  uint32_t* kmask = reinterpret_cast<uint32_t*>(base + 768);  // [8] sub-tiles holding data, per tile slot
  uint8_t* qs = base + 1024;                       // [2][Q tile]
  uint8_t* ks = qs + 2 * Cfg::kQBytes;             // [3 stages][K tile]
  uint8_t* vs = ks + kUmKStages * Cfg::kKvBytes;   // [2 stages][V tile]
  uint8_t* ps = vs + kUmVStages * Cfg::kKvBytes;   // [2 groups][2 buffers][P tile]

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
    for (int s = 0; s < 4; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&s_free[s], 128);
      mbar_init(&p_full[s], 128);
      mbar_init(&pv_done[s], 1);
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
  // S_k^b at columns [64 (2k + b), +64), O_k at [256 + 128k, +D)
  auto tS = [&](int k, int b) { return tmem + 64u * (uint32_t)(2 * k + b); };
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
            // Slot i % 8 was last read for tile i - 8, which both groups finished long ago: this
            // lane cannot run more than 4 tiles ahead of them (K ring depth + one S in flight).
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
          umma_ss(tS(k, i & 1), umma_desc_sw128(qa + qo, 16, 1024), umma_desc_sw128(ka + ko, 16, 1024), id_s,
                  kk > 0 ? 1u : 0u);
        }
        umma_commit(&s_full[2 * k + (i & 1)]);
      };
      auto issue_pv = [&](int k, int i) {
        const uint32_t pa_ = smem_u32(ps + (2 * k + (i & 1)) * Cfg::kPBytes);
        const uint32_t va = smem_u32(vs + (i % kUmVStages) * Cfg::kKvBytes);
#pragma unroll
        for (int kk = 0; kk < kUmKeys / 16; ++kk)
          umma_ss(tO(k), umma_desc_sw128(pa_ + kk * 32, 16, 1024),
                  umma_desc_sw128(va + kk * 2048, Cfg::kKvHalf, 1024), id_pv, (i > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&pv_done[2 * k + (i & 1)]);
      };
      // Event-driven issue: each group's next S (needs its previous S read out and the K tile) and
      // next P V (needs its P and the V tile) are issued as soon as they are ready, so a slow group
      // never holds back the other group's products.
      bool alive = mbar_wait(q_ready, 0, a.err);
      int next_s[2] = {0, 0}, next_pv[2] = {0, 0};
      int idle = 0;
      while (alive && (next_pv[0] < n_all || next_pv[1] < n_all)) {
        bool progress = false;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          // S_k(j) overwrites buffer j % 2, last holding S_k(j - 2)
          const int j = next_s[k];
          if (j < n_all && (j < 2 || mbar_test(&s_free[2 * k + (j & 1)], (unsigned)(((j >> 1) - 1) & 1))) &&
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
          if (jp < next_s[k] && (k == 0 || next_pv[0] > jp) &&
              mbar_test(&p_full[2 * k + (jp & 1)], (unsigned)((jp >> 1) & 1)) &&
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
        const int bsel = i & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(&s_full[2 * grp + bsel], (unsigned)((i >> 1) & 1), a.err))) {
          alive = false;
          break;
        }
        tc_fence_after();
        float x[kUmKeys];
#pragma unroll
        for (int c0 = 0; c0 < kUmKeys; c0 += 32) {
          uint32_t v[32];
          tmem_ld32(tS(grp, bsel) + lane_base + c0, v);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) x[c0 + j] = __uint_as_float(v[j]);
        }
        tc_fence_before();
        mbar_arrive(&s_free[2 * grp + bsel]);  // this S buffer may now take tile i + 2
        // a tile wholly inside this row's causal bound with every sub-tile loaded needs no mask
        const float sc = a.scale_log2;
        const bool fast = sc > 0.f && loaded == (1u << kUmSub) - 1u && kb + kUmKeys - 1 <= bound;
        float mx = -INFINITY;
        if (fast) {
#pragma unroll
          for (int c = 0; c < kUmKeys; ++c) mx = fmaxf(mx, x[c]);
          mx *= sc;
        } else {
          // bit c of `keep`: key kb + c is loaded and inside the causal bound
          uint64_t keep = 0;
#pragma unroll
          for (int sub = 0; sub < kUmSub; ++sub)
            if ((loaded >> sub) & 1u) keep |= 0xFFFFull << (16 * sub);
          const int64_t lim = bound - kb;  // keys c <= lim are causal
          if (lim < 0) keep = 0;
          else if (lim < kUmKeys - 1) keep &= (2ull << lim) - 1ull;
#pragma unroll
          for (int c = 0; c < kUmKeys; ++c) {
            x[c] = ((keep >> c) & 1ull) ? x[c] * sc : -INFINITY;
            mx = fmaxf(mx, x[c]);
          }
        }
        // move the stabiliser only when it must: first finite maximum, or growth beyond 2^8
        float corr = 1.f;
        if (mx > m_use + kUmRescaleThreshold || (m_use == -INFINITY && mx != -INFINITY)) {
          corr = fast_exp2(m_use - mx);  // m_use = -inf -> 0
          m_use = mx;
        }
        const float m_sub = m_use == -INFINITY ? 0.f : m_use;
        float rs = 0.f;
        if (fast) {
#pragma unroll
          for (int c = 0; c < kUmKeys; ++c) {
            x[c] = fast_exp2(fmaf(x[c], sc, -m_sub));
            rs += x[c];
          }
        } else {
#pragma unroll
          for (int c = 0; c < kUmKeys; ++c) {
            x[c] = fast_exp2(x[c] - m_sub);
            rs += x[c];
          }
        }
        l_run = l_run * corr + rs;
        // the P buffer of tile i - 2 must have been consumed, and O must be stable before a rescale
        if (i >= 2 && !__all_sync(0xffffffffu, mbar_wait(&pv_done[2 * grp + bsel], (unsigned)(((i >> 1) - 1) & 1), a.err))) {
          alive = false;
          break;
        }
        if (i > 0 && __any_sync(0xffffffffu, corr != 1.f)) {
          const int pb = (i - 1) & 1;
          if (!__all_sync(0xffffffffu, mbar_wait(&pv_done[2 * grp + pb], (unsigned)(((i - 1) >> 1) & 1), a.err))) {
            alive = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(tO(grp) + lane_base + c0, v);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * corr);
            tmem_st32(tO(grp) + lane_base + c0, v);
          }
          tmem_wait_st();
        }
        // group 0 zeroes V rows that hold no data or lie past the context (group 1's P V is issued
        // after group 0's, so it sees the zeros too)
        if (grp == 0 && (kb + kUmKeys > sg.n || loaded != (1u << kUmSub) - 1u)) {
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
        }
        // P row into shared memory: [row][64 keys] = one 128-byte swizzled row
#pragma unroll
        for (int c = 0; c < kUmKeys / 8; ++c) {
          uint4 w;
          w.x = pack2<kBf16>(x[8 * c + 0], x[8 * c + 1]);
          w.y = pack2<kBf16>(x[8 * c + 2], x[8 * c + 3]);
          w.z = pack2<kBf16>(x[8 * c + 4], x[8 * c + 5]);
          w.w = pack2<kBf16>(x[8 * c + 6], x[8 * c + 7]);
          *reinterpret_cast<uint4*>(ps + (2 * grp + bsel) * Cfg::kPBytes + sw_off(r, c, kUmTileRows * 128)) = w;
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&p_full[2 * grp + bsel]);
      }
      t = sg.seg1;
    }
    if (!alive && lane == 0) raise_error(a.err, PA_DEVERR_TIMEOUT);
    if (alive && i > 0) {
      alive = __all_sync(0xffffffffu, mbar_wait(&pv_done[2 * grp + ((i - 1) & 1)], (unsigned)(((i - 1) >> 1) & 1), a.err));
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
