// Tensor-core paged decode for bf16/fp16 pools (block_size a multiple of 16).
//
// Same contract and grid as the CUDA-core kernel (attn_simt.cu): one CTA per (sequence, KV head,
// split-K partition) serving the whole GQA query group, online softmax (JuliaPagedAttn README,
// "Online Softmax"), read-time GQA (nanoserve Day 19, "What I learned" 4), output or partial state
// for the log-sum-exp merge.  What differs is how the bytes move and how the dots are formed:
//
// * Data movement.  A 16-token tile of one KV head (K and V, 2 x 16 x head_dim elements) is
//   fetched by TMA from the block the table names: the pool is seen as a 2-D tensor
//   [num_blocks * block_size rows][n_kv_heads * head_dim columns] and each tile is head_dim/64
//   boxes of 16 rows x 64 columns per operand, written to shared memory with the 128-byte swizzle.
//   Each warp owns a private ring of kStages tiles guarded by one mbarrier per stage; lane 0
//   refills a stage as soon as the warp has consumed it, so every warp keeps kStages tiles in
//   flight with no cross-warp synchronisation (the software prefetch / double buffering of
//   JuliaPagedAttn's kernel, done by the copy engine).
// * Arithmetic.  Q K^T and P V are mma.sync m16n8k16 products with fp32 accumulation: the query
//   group (G <= 8 heads) fills the rows of the A operand, K and V tiles are read with ldmatrix
//   (V transposed), and the softmax probabilities are re-packed from the QK accumulator registers
//   straight into the A operand of the PV product.  One online-softmax update per 16-token tile.
// * Ragged ends.  Tokens past the partition's end are masked to -inf before the softmax and their
//   V rows are zeroed in shared memory (a stale NaN times a zero probability would otherwise
//   poison the accumulator).  A tile whose table entry is out of range is skipped and recorded.
//
// The tile loop inside a warp visits tokens in increasing logical order, so the result depends
// only on logical positions, not on where the blocks sit in the pool.
#include <cudaTypedefs.h>

#include <mutex>

#include "pa_common.cuh"
#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {

// Tuning constants (overridable at build time with -D for measurement sweeps).  Measured on
// GB300 at the Llama-3-8B serving shape: 4 warps x 2 stages (66 KB, 3 CTAs per SM) with
// 1024-token partitions beat 2/3/4-stage, 2/8-warp and 1-4 CTA/SM variants.
#ifndef PA_TC_WARPS
#define PA_TC_WARPS 4
#endif
#ifndef PA_TC_STAGES_128
#define PA_TC_STAGES_128 2
#endif
#ifndef PA_TC_STAGES_64
#define PA_TC_STAGES_64 4
#endif
#ifndef PA_TC_MIN_CTAS
#define PA_TC_MIN_CTAS 3
#endif
// 1: decode grids are launched with programmatic dependent launch (see launch_tc_g)
#ifndef PA_DECODE_PDL
#define PA_DECODE_PDL 1
#endif
// 1: K/V tiles are loaded with the L2 evict-first policy (read once), which keeps the split-K
// partials L2-resident for the merge kernel
#ifndef PA_KV_EVICT_FIRST
#define PA_KV_EVICT_FIRST 1
#endif

// One TMA box of a K or V tile, with the evict-first policy when PA_KV_EVICT_FIRST is set.
__device__ __forceinline__ void load_kv_box(void* dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar,
                                            uint64_t policy) {
  if (PA_KV_EVICT_FIRST)
    tma_load_3d_hint(dst, map, x, y, z, bar, policy);
  else
    tma_load_3d(dst, map, x, y, z, bar);
}

constexpr int kTcWarps = PA_TC_WARPS;
constexpr int kTile = 16;          // tokens per tile (one mma k-step of PV)
constexpr int kHalfBytes = kTile * 128;  // 16 rows x 64 columns x 2 bytes

template <int D>
struct TcCfg {
  static constexpr int kHalves = D / 64;
  static constexpr int kStageBytes = 2 * kHalves * kHalfBytes;  // K and V
  static constexpr int kStages = D == 128 ? PA_TC_STAGES_128 : PA_TC_STAGES_64;  // per warp
  static constexpr int kSmemBytes =
      1024 /*barriers*/ + 1024 /*alignment*/ + kTcWarps * kStages * kStageBytes;
  static_assert(kTcWarps * kStages * 8 <= 1024, "barriers must fit their 1 KB slot");
};

// Rows of the mma tile that hold query heads: head g in row g, and for groups of 16 head g + 8 in
// row g + 8 (the second row half of the m16n8k16 tile).
template <int G>
struct RowHalves {
  static constexpr int kN = G > 8 ? 2 : 1;
};

// Q fragments of the mma A operand for the query group of KV head kvh in sequence b: per k-step,
// [0] rows g / cols 2*tig, [1] rows g + 8 / cols 2*tig, [2] rows g / cols 8 + 2*tig, [3] rows
// g + 8 / cols 8 + 2*tig (two elements each).  Rows without a head are zero.
template <typename T, int D, int G>
__device__ __forceinline__ void load_q_frags(const AttnArgs& a, int64_t b, int kvh, int lane,
                                             uint32_t (&qa)[D / 16][4]) {
  const int g = lane >> 2, tig = lane & 3;
  const T* qrow = static_cast<const T*>(a.q) + (b * a.n_q_heads + (int64_t)kvh * G + g) * D;
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int head = g + 8 * hh;
      const bool have = (G > 8 || hh == 0) && head < G;
      qa[ks][hh] = have ? __ldg(reinterpret_cast<const uint32_t*>(qrow + 8 * hh * D + ks * 16 + 2 * tig)) : 0u;
      qa[ks][2 + hh] = have ? __ldg(reinterpret_cast<const uint32_t*>(qrow + 8 * hh * D + ks * 16 + 8 + 2 * tig)) : 0u;
    }
  }
}

// This step's token of KV head kvh, row r of the 16-token tile at st: from k_src / v_src (head_dim
// elements each) into shared memory, swizzled like the TMA boxes, and into the pools at k_dst / v_dst.
template <typename T, int D>
__device__ __forceinline__ void patch_new_token(uint8_t* st, int r, const T* k_src, const T* v_src, T* k_dst,
                                                T* v_dst, int lane) {
  constexpr int kHalves = D / 64;
  constexpr int kChunks = D / 8;
  if (lane < 2 * kChunks) {
    const bool isv = lane >= kChunks;
    const int c = lane % kChunks;
    const uint4 val = __ldg(reinterpret_cast<const uint4*>((isv ? v_src : k_src) + c * 8));
    *reinterpret_cast<uint4*>(st + ((isv ? kHalves : 0) + (c >> 3)) * kHalfBytes + r * 128 +
                              (((c & 7) ^ (r & 7)) << 4)) = val;
    *reinterpret_cast<uint4*>((isv ? v_dst : k_dst) + c * 8) = val;
  }
  __syncwarp();
}

// Folds one 16-token K/V tile (at st, in the swizzled TMA layout) into the warp's online-softmax
// state (o, m_run, l_run; rows = query heads in the mma layout, one state per row half).  Tokens
// >= valid are masked and their V rows zeroed first.
template <typename T, int D, int G>
__device__ __forceinline__ void tile_update(uint8_t* st, int valid, const uint32_t (&qa)[D / 16][4],
                                            float (&o)[D / 8][4], float (&m_run)[2], float (&l_run)[2],
                                            float scale_log2, int lane) {
  constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
  constexpr int kHalves = D / 64;
  constexpr int kKSteps = D / 16;
  constexpr int kDTiles = D / 8;
  constexpr int kRows = RowHalves<G>::kN;
  const int tig = lane & 3;
  const uint32_t k_base = smem_u32(st);
  const uint32_t v_base = smem_u32(st + kHalves * kHalfBytes);
  if (valid < kTile) {
    // zero the V rows past the end (both halves): 16-byte stores, rows valid..15
    const int nz = (kTile - valid) * 8 * kHalves;
    for (int i = lane; i < nz; i += 32) {
      const int h = i / ((kTile - valid) * 8);
      const int r = valid + (i / 8) % (kTile - valid);
      const int c = i % 8;
      *reinterpret_cast<uint4*>(st + (kHalves + h) * kHalfBytes + r * 128 + c * 16) = make_uint4(0, 0, 0, 0);
    }
    __syncwarp();
  }
  // ---- S = Q K^T: two n-tiles of 8 tokens ------------------------------------------------------
  float sc[2][4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
    const int tok = nt * 8 + (lane & 7);
#pragma unroll
    for (int ks = 0; ks < kKSteps; ks += 2) {
      const int chunk = 2 * ks + (lane >> 3);  // 8-element chunk along head_dim
      const uint32_t addr = k_base + (chunk >> 3) * kHalfBytes + tok * 128 + (((chunk & 7) ^ (tok & 7)) << 4);
      uint32_t b0, b1, b2, b3;
      ldsm_x4(addr, b0, b1, b2, b3);
      mma_16816<kBf16>(sc[nt], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
      mma_16816<kBf16>(sc[nt], qa[ks + 1][0], qa[ks + 1][1], qa[ks + 1][2], qa[ks + 1][3], b2, b3);
    }
  }
  // ---- online softmax over the tile, per row half (rows g, then g + 8; columns = tokens) ---------
  uint32_t pa[4] = {0u, 0u, 0u, 0u};  // P as the A operand of P V: [0]/[2] rows g, [1]/[3] rows g + 8
#pragma unroll
  for (int hh = 0; hh < kRows; ++hh) {
    float x[4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int tok = nt * 8 + 2 * tig + e;
        x[nt * 2 + e] = tok < valid ? sc[nt][2 * hh + e] * scale_log2 : -INFINITY;
      }
    }
    float tmax = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
    tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
    tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
    const float m_new = fmaxf(m_run[hh], tmax);
    const float corr = fast_exp2(m_run[hh] - m_new);
    float p[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) p[i] = fast_exp2(x[i] - m_new);
    l_run[hh] = l_run[hh] * corr + ((p[0] + p[1]) + (p[2] + p[3]));
    if (__any_sync(0xffffffffu, corr != 1.f)) {
#pragma unroll
      for (int i = 0; i < kDTiles; ++i) {
        o[i][2 * hh] *= corr;
        o[i][2 * hh + 1] *= corr;
      }
    }
    m_run[hh] = m_new;
    pa[hh] = pack2<kBf16>(p[0], p[1]);
    pa[2 + hh] = pack2<kBf16>(p[2], p[3]);
  }
  // ---- O += P V: P from the score registers, V^T fragments by ldmatrix.trans ---------------------
#pragma unroll
  for (int dt = 0; dt < kDTiles; dt += 2) {
    const int mi = lane >> 3;
    const int tok = (lane & 7) + 8 * (mi & 1);
    const int chunk = dt + (mi >> 1);
    const uint32_t addr = v_base + (chunk >> 3) * kHalfBytes + tok * 128 + (((chunk & 7) ^ (tok & 7)) << 4);
    uint32_t b0, b1, b2, b3;
    ldsm_x4_t(addr, b0, b1, b2, b3);
    mma_16816<kBf16>(o[dt], pa[0], pa[1], pa[2], pa[3], b0, b1);
    mma_16816<kBf16>(o[dt + 1], pa[0], pa[1], pa[2], pa[3], b2, b3);
  }
}

template <typename T, int D, int G>
__global__ void __launch_bounds__(kTcWarps * 32, G > 8 ? 2 : PA_TC_MIN_CTAS)
    decode_tc_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap kmap,
                     const __grid_constant__ CUtensorMap vmap) {
  constexpr int kHalves = TcCfg<D>::kHalves;
  constexpr int kStageBytes = TcCfg<D>::kStageBytes;
  constexpr int kStages = TcCfg<D>::kStages;
  constexpr int kKSteps = D / 16;
  constexpr int kDTiles = D / 8;
  static_assert(G <= 16, "query group must fit the 16 rows of the mma tile");
  constexpr int kRows = RowHalves<G>::kN;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(base);
  uint8_t* stages = base + 1024;

  // grid order: KV heads innermost (CTAs touching one physical block run together)
  const int kvh = (int)(blockIdx.x % a.n_kv_heads);
  const int part = (int)((blockIdx.x / a.n_kv_heads) % a.max_parts);
  const int64_t row = (int64_t)(blockIdx.x / a.n_kv_heads) / a.max_parts;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int g = lane >> 2;   // mma row group: query head g of the group
  const int tig = lane & 3;  // thread in group

  // set-up that reads no global memory: this warp's ring barriers and the tensor maps
  uint64_t* my_bars = bars + warp * kStages;
  uint8_t* my_stages = stages + warp * kStages * kStageBytes;
  if (lane == 0) {
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
    for (int s = 0; s < kStages; ++s) mbar_init(&my_bars[s], 1);
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  __syncwarp();

  // launched with programmatic serialization: wait for the preceding grid (its outputs may be this
  // call's inputs, and its reads of out / workspace must end before this grid writes them)
  pdl_wait_primary();
  const int64_t max_len = a.bt_stride << a.block_shift;
  const int b = (int)row;
  const int32_t* table = a.block_table + (int64_t)b * a.bt_stride;
  const int64_t t_begin = (int64_t)part * a.part_tokens;
  // tile j of this warp covers tokens [tile_t0(j), tile_t0(j) + 16)
  auto tile_t0 = [&](int j) -> int64_t { return t_begin + (int64_t)(warp + kTcWarps * j) * kTile; };
  auto tile_block = [&](int j) -> int { return __ldg(table + (tile_t0(j) >> a.block_shift)); };
  // The loads that do not depend on one another go out together, so that their latencies overlap:
  // the context length, the table entries of this warp's first tiles (read ahead of the length:
  // every position below the table's capacity has an entry) and the Q fragments.
  int64_t len = __ldg(a.context_lens + b);
  int blk_first[kStages];
#pragma unroll
  for (int j = 0; j < kStages; ++j)
    blk_first[j] = (lane == 0 && tile_t0(j) < max_len) ? tile_block(j) : -1;
  uint32_t qa[kKSteps][4];
  load_q_frags<T, D, G>(a, row, kvh, lane, qa);
  if (len < 0 || len > max_len) {
    if (threadIdx.x == 0) raise_error(a.err, PA_DEVERR_CONTEXT_LEN);
    len = len < 0 ? 0 : max_len;
  }
  const int n_parts_row = len == 0 ? 1 : (int)((len + a.part_tokens - 1) / a.part_tokens);
  if (part >= n_parts_row) return;
  const int64_t t_end = min(t_begin + a.part_tokens, len);
  const int n_tiles = (int)((t_end - t_begin + kTile - 1) / kTile);
  const int my_tiles = n_tiles > warp ? (n_tiles - warp + kTcWarps - 1) / kTcWarps : 0;
  const int bmask = a.block_size - 1;

  pdl_launch_dependents();  // the split-K merge may begin launching; it waits for this grid's results

  const uint64_t kv_policy = l2_policy_evict_first();  // K/V are read once per launch
  auto issue = [&](int j, int blk) {  // lane 0 only; blk = the table entry of tile j
    const int s = j % kStages;
    if (blk < 0 || blk >= a.num_blocks) {
      raise_error(a.err, PA_DEVERR_BLOCK_ID);
      mbar_arrive(&my_bars[s]);  // complete the phase without data; the consumer skips the tile
      return;
    }
    const int off = (int)(tile_t0(j) & bmask);
    uint8_t* st = my_stages + s * kStageBytes;
    mbar_arrive_expect_tx(&my_bars[s], kStageBytes);
#pragma unroll
    for (int h = 0; h < kHalves; ++h)
      load_kv_box(st + h * kHalfBytes, &kmap, kvh * D + h * 64, off, blk, &my_bars[s], kv_policy);
#pragma unroll
    for (int h = 0; h < kHalves; ++h)
      load_kv_box(st + (kHalves + h) * kHalfBytes, &vmap, kvh * D + h * 64, off, blk, &my_bars[s], kv_policy);
  };
  if (lane == 0) {
    const int pre = my_tiles < kStages ? my_tiles : kStages;
#pragma unroll
    for (int j = 0; j < kStages; ++j)
      if (j < pre) issue(j, blk_first[j]);
  }

  // fused write: the CTA holding the last context position writes this step's K/V row of its KV
  // head there and uses it straight from k_new / v_new (nanoserve Day 19, "What I added today":
  // write this step's K/V, then attend over the whole history).  Looked up once the first copies
  // are on their way.
  int64_t new_row = -1;  // element offset of the new token's pool row
  if (a.k_new != nullptr && len > 0 && part == n_parts_row - 1) {
    const int64_t last = len - 1;
    const int64_t s_new = __ldg(a.slot_mapping + b);
    const int blk_last = __ldg(table + (last >> a.block_shift));
    const int64_t expect = (blk_last >= 0 && blk_last < a.num_blocks)
                               ? ((int64_t)blk_last << a.block_shift) + (last & bmask) : -2;
    if (s_new >= 0) {
      if (s_new == expect)
        new_row = (int64_t)blk_last * a.kv_block_stride + (last & bmask) * ((int64_t)a.n_kv_heads * D);
      else if (threadIdx.x == 0)
        raise_error(a.err, PA_DEVERR_SLOT);
    }
  }
  const int patch_tile = new_row >= 0 ? (int)((len - 1 - t_begin) / kTile) : -1;

  float o[kDTiles][4];
#pragma unroll
  for (int i = 0; i < kDTiles; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  bool timed_out = false;

  int j_fail = my_tiles;  // first tile whose wait gave up
  for (int j = 0; j < my_tiles; ++j) {
    const int s = j % kStages;
    if (!__all_sync(0xffffffffu, mbar_wait(&my_bars[s], (unsigned)((j / kStages) & 1), a.err, a.epoch))) {
      timed_out = true;
      j_fail = j;
      break;
    }
    const int blk = tile_block(j);
    const int64_t t0 = tile_t0(j);
    const int valid = (int)(t_end - t0 < kTile ? t_end - t0 : kTile);
    uint8_t* st = my_stages + s * kStageBytes;
    if (blk >= 0 && blk < a.num_blocks) {
      if (warp + kTcWarps * j == patch_tile) {
        // this step's token: row (len - 1) mod 16 of the tile, from k_new / v_new, into shared
        // memory and into the pool
        const int64_t src_off = ((int64_t)b * a.n_kv_heads + kvh) * D;
        const int64_t dst_off = new_row + (int64_t)kvh * D;
        patch_new_token<T, D>(st, (int)((len - 1) & (kTile - 1)), static_cast<const T*>(a.k_new) + src_off,
                              static_cast<const T*>(a.v_new) + src_off, static_cast<T*>(a.k_pool_w) + dst_off,
                              static_cast<T*>(a.v_pool_w) + dst_off, lane);
      }
      tile_update<T, D, G>(st, valid, qa, o, m_run, l_run, a.scale_log2, lane);
    }
    // release the stage and refill it with this warp's tile j + kStages
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0 && j + kStages < my_tiles) issue(j + kStages, tile_block(j + kStages));
  }
  if (timed_out && lane == 0) {
    raise_timeout(a.err, a.epoch);
    // leave no copy in flight: wait (bounded) for the tiles issued from j_fail on
    const int issued = j_fail + kStages < my_tiles ? j_fail + kStages : my_tiles;
    for (int j = j_fail; j < issued; ++j) mbar_wait(&my_bars[j % kStages], (unsigned)((j / kStages) & 1));
  }
  __syncwarp();

  // ---- combine: quad-reduce l, stage (m, l, o) per warp in the warp's own stages ----------------
  __syncwarp();
  float* wo = reinterpret_cast<float*>(my_stages);  // [G][D] floats, then m[G], l[G]
#pragma unroll
  for (int hh = 0; hh < kRows; ++hh) {
    float lr = l_run[hh];
    lr += __shfl_xor_sync(0xffffffffu, lr, 1);
    lr += __shfl_xor_sync(0xffffffffu, lr, 2);
    const int gr = g + 8 * hh;  // query head of this row
    if (gr < G) {
#pragma unroll
      for (int i = 0; i < kDTiles; ++i) {
        wo[gr * D + i * 8 + 2 * tig] = o[i][2 * hh];
        wo[gr * D + i * 8 + 2 * tig + 1] = o[i][2 * hh + 1];
      }
      if (tig == 0) {
        wo[G * D + gr] = m_run[hh];
        wo[G * D + G + gr] = my_tiles > 0 && !timed_out ? lr : 0.f;
      }
    }
  }
  __syncthreads();

  const bool direct = n_parts_row == 1;
  for (int i = threadIdx.x; i < G * D; i += kTcWarps * 32) {
    const int h = i / D;
    const int d = i - h * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kTcWarps; ++w) {
      const float* ww = reinterpret_cast<const float*>(stages + w * kStages * kStageBytes);
      if (ww[G * D + G + h] != 0.f) M = fmaxf(M, ww[G * D + h]);
    }
    float L = 0.f, A = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kTcWarps; ++w) {
        const float* ww = reinterpret_cast<const float*>(stages + w * kStages * kStageBytes);
        const float lw = ww[G * D + G + h];
        if (lw != 0.f) {
          const float f = fast_exp2(ww[G * D + h] - M);
          L = fmaf(lw, f, L);
          A = fmaf(ww[h * D + d], f, A);
        }
      }
    }
    const int64_t qh = row * a.n_q_heads + (int64_t)kvh * G + h;
    if (direct) {
      static_cast<T*>(a.out)[qh * D + d] = Elt<T>::from_float(L != 0.f ? A / L : 0.f);
    } else {
      const int64_t pi = qh * a.max_parts + part;
      a.ws_acc[pi * D + d] = A;
      if (d == 0) {
        a.ws_m[pi] = M;
        a.ws_l[pi] = L;
      }
    }
  }
}

// ------------------------------------------------------------------------------------------------
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

}  // namespace

// L2 promotion of the pool boxes' reads (build-time overridable: 0 none, 1 64 B, 2 128 B, 3 256 B)
#ifndef PA_POOL_L2_PROMOTION
#define PA_POOL_L2_PROMOTION 3
#endif

// Pool viewed as a 3-D tensor (column in [0, n_kv_heads * head_dim), token in block, block) with the
// pool's own block stride (so separate pools and unified K/V blocks share one code path); boxes of
// 64 columns x 16 tokens x 1 block.
bool encode_pool_map(CUtensorMap* map, const void* pool, pa_dtype dt, int64_t num_blocks, int block_size,
                     int n_kv_heads, int head_dim, int64_t block_stride) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)n_kv_heads * head_dim, (cuuint64_t)block_size, (cuuint64_t)num_blocks};
  const cuuint64_t strides[2] = {(cuuint64_t)n_kv_heads * head_dim * 2, (cuuint64_t)block_stride * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)kTile, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType ty = dt == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const CUtensorMapL2promotion promo = PA_POOL_L2_PROMOTION == 0   ? CU_TENSOR_MAP_L2_PROMOTION_NONE
                                       : PA_POOL_L2_PROMOTION == 1 ? CU_TENSOR_MAP_L2_PROMOTION_L2_64B
                                       : PA_POOL_L2_PROMOTION == 2 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B
                                                                   : CU_TENSOR_MAP_L2_PROMOTION_L2_256B;
  CUresult r = fn(map, ty, 3, const_cast<void*>(pool), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Queries [total_q][n_q_heads][head_dim] viewed as a 3-D tensor (column, head, token); boxes of 64
// columns x heads_box heads x tokens_box tokens with the 128-byte swizzle, so that one box lands as
// heads_box * tokens_box rows of 128 bytes ordered (token, head).  Rows past total_q read as zeros.
bool encode_q_map(CUtensorMap* map, const void* q, pa_dtype dt, int64_t total_q, int n_q_heads, int head_dim,
                  int heads_box, int tokens_box) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)n_q_heads, (cuuint64_t)total_q};
  const cuuint64_t strides[2] = {(cuuint64_t)head_dim * 2, (cuuint64_t)n_q_heads * head_dim * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)heads_box, (cuuint32_t)tokens_box};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType ty = dt == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUresult r = fn(map, ty, 3, const_cast<void*>(q), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool decode_tc_supported(pa_dtype dt, int block_size, int head_dim, int group, int64_t num_blocks) {
  if (dt != PA_BF16 && dt != PA_FP16) return false;
  if (block_size % kTile != 0) return false;
  if (head_dim != 64 && head_dim != 128) return false;
  if (group > 16) return false;
  if (num_blocks >= (int64_t(1) << 31)) return false;  // TMA block coordinate is int32
  return encode_fn() != nullptr;
}

template <typename T, int D, int G>
static cudaError_t launch_tc_g(const AttnArgs& a, const CUtensorMap& km, const CUtensorMap& vm, cudaStream_t s) {
  constexpr int smem = TcCfg<D>::kSmemBytes;
  static bool attr_set[64] = {};  // per instantiation and device; idempotent, so a race is harmless
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(decode_tc_kernel<T, D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  const int64_t grid = a.rows * (int64_t)a.max_parts * a.n_kv_heads;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kTcWarps * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  // programmatic dependent launch: the grid may start while the preceding kernel of the stream
  // (typically the previous step's merge) finishes; the kernel waits for it before any global access
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = PA_DECODE_PDL ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, decode_tc_kernel<T, D, G>, a, km, vm);
}

template <typename T, int D>
static cudaError_t launch_tc_d(const AttnArgs& a, const CUtensorMap& km, const CUtensorMap& vm, cudaStream_t s) {
  switch (a.group) {
    case 1: return launch_tc_g<T, D, 1>(a, km, vm, s);
    case 2: return launch_tc_g<T, D, 2>(a, km, vm, s);
    case 4: return launch_tc_g<T, D, 4>(a, km, vm, s);
    case 8: return launch_tc_g<T, D, 8>(a, km, vm, s);
    case 16: return launch_tc_g<T, D, 16>(a, km, vm, s);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T>
static cudaError_t launch_tc_t(const AttnArgs& a, const CUtensorMap& km, const CUtensorMap& vm, cudaStream_t s) {
  return a.head_dim == 64 ? launch_tc_d<T, 64>(a, km, vm, s) : launch_tc_d<T, 128>(a, km, vm, s);
}

cudaError_t launch_decode_tc(const AttnArgs& a, pa_dtype dt, cudaStream_t s, int* launches) {
  if (a.rows == 0) return cudaSuccess;
  CUtensorMap km, vm;
  if (!encode_pool_map(&km, a.k_pool, dt, a.num_blocks, a.block_size, a.n_kv_heads, a.head_dim, a.kv_block_stride) ||
      !encode_pool_map(&vm, a.v_pool, dt, a.num_blocks, a.block_size, a.n_kv_heads, a.head_dim, a.kv_block_stride))
    return cudaErrorInvalidValue;
  cudaError_t e = dt == PA_BF16 ? launch_tc_t<__nv_bfloat16>(a, km, vm, s) : launch_tc_t<__half>(a, km, vm, s);
  ++*launches;
  return e;
}

}  // namespace pa
