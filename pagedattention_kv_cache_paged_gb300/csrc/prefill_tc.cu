// Tensor-core causal chunked prefill over a paged history, bf16/fp16, block_size % 16 == 0.
//
// What it computes — JuliaPagedAttn README, "Features" (batched prefill: every prompt position in
// one call) with the online softmax of "Online Softmax": sequence b's chunk of m_b queries holds
// the last m_b positions of its context_lens[b] tokens and query r attends to positions
// 0 .. context_lens[b] - m_b + r through the block table (causal, inclusive).
//
// Work decomposition.  A CTA owns kRows = 16 * kPfWarps (query token, head) rows of one KV head:
// kRows / G consecutive query tokens of the flattened batch times the G query heads of the group,
// so every K/V tile fetched from HBM/L2 serves all heads of the group (read-time GQA, nanoserve
// Day 19 "What I learned" 4).  The token range may span several sequences; the CTA walks them as
// segments, each with its own keys, and a row's softmax state changes only during its own segment.
//
// Pipeline.  A producer warp streams 64-key tiles (K and V, boxes of 16 keys x 64 columns from the
// physical blocks the table names, 128-byte swizzle) into a ring of kPfStages stages; kPfWarps
// consumer warps compute S = Q K^T (mma.sync m16n8k16, fp32 accumulate), apply the causal mask,
// update the online softmax per row and accumulate O += P V, then release the stage.  Every
// mbarrier wait is bounded (PA_DEVERR_TIMEOUT).
#include <cudaTypedefs.h>

#include "pa_common.cuh"
#include "pa_internal.h"
#include "pa_ptx.cuh"

#ifndef PA_PF_WARPS
#define PA_PF_WARPS 8
#endif
#ifndef PA_PF_STAGES
#define PA_PF_STAGES 3
#endif

namespace pa {

constexpr int kPfWarps = PA_PF_WARPS;        // consumer warps
constexpr int kPfThreads = (kPfWarps + 1) * 32;
constexpr int kPfRows = 16 * kPfWarps;
constexpr int kKeyTile = 64;
constexpr int kSub = kKeyTile / 16;          // 16-key sub-tiles per tile
constexpr int kPfStages = PA_PF_STAGES;
constexpr int kBoxBytes = 16 * 128;          // one TMA box: 16 keys x 64 columns x 2 bytes

template <int D>
struct PfCfg {
  static constexpr int kHalves = D / 64;
  static constexpr int kOperandBytes = kSub * kHalves * kBoxBytes;  // one of K or V per stage
  static constexpr int kStageBytes = 2 * kOperandBytes;
  static constexpr int kQBytes = kPfRows * D * 2;                  // Q rows of the CTA, swizzled
  static constexpr int kSmemBytes = 1024 + 1024 + kPfStages * kStageBytes + kQBytes;
};

// Byte offset of (row r, 8-element chunk c) in the CTA's Q block: 16-row groups of head_dim/64
// swizzled 128-byte halves, laid out like one operand of a K/V stage.
template <int D>
__device__ __forceinline__ uint32_t q_offset(int r, int c) {
  const int grp = r >> 4, rr = r & 15;
  return (uint32_t)((grp * PfCfg<D>::kHalves + (c >> 3)) * kBoxBytes + rr * 128 + (((c & 7) ^ (rr & 7)) << 4));
}

// Byte offset of (key kk in 0..63, 8-element chunk c along head_dim) inside one operand of a stage.
template <int D>
__device__ __forceinline__ uint32_t pf_offset(int kk, int c) {
  const int sub = kk >> 4, r = kk & 15;
  return (uint32_t)((sub * PfCfg<D>::kHalves + (c >> 3)) * kBoxBytes + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

template <typename T, int D, int G>
__global__ void __launch_bounds__(kPfThreads, 1)
    prefill_tc_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap) {
  constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
  constexpr int kHalves = PfCfg<D>::kHalves;
  constexpr int kOpBytes = PfCfg<D>::kOperandBytes;
  constexpr int kStageBytes = PfCfg<D>::kStageBytes;
  constexpr int kKSteps = D / 16;
  constexpr int kDTiles = D / 8;
  constexpr int kQB = kPfRows / G;  // query tokens per CTA

  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(base);
  uint64_t* empty = full + kPfStages;
  uint8_t* stages = base + 1024;

  const int kvh = blockIdx.x % a.n_kv_heads;
  const int64_t T0 = (int64_t)(blockIdx.x / a.n_kv_heads) * kQB;
  const int64_t T1 = min(T0 + kQB, a.rows);  // a.rows = total_q
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int64_t max_len = a.bt_stride << a.block_shift;
  const int bmask = a.block_size - 1;

  if (threadIdx.x == 0) {
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
    for (int s = 0; s < kPfStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kPfWarps);
    }
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  __syncthreads();

  // Segment walk shared by producer and consumers: [seg0, seg1) tokens of sequence b, keys
  // [0, kv_end), context n, chunk start position pos0 = n - m (absolute position of the chunk's
  // first query).
  struct Seg {
    int b;
    int64_t seg0, seg1, n, pos0, q0, kv_end;
  };
  auto segment_at = [&](int64_t t, Seg& sg) -> bool {
    const int b = find_sequence(a.query_start_loc, a.batch, t);
    const int64_t q0 = __ldg(a.query_start_loc + b);
    const int64_t q1 = __ldg(a.query_start_loc + b + 1);
    int64_t n = __ldg(a.context_lens + b);
    sg.b = b;
    sg.seg0 = t;
    sg.seg1 = min(q1, T1);
    if (sg.seg1 <= t) sg.seg1 = t + 1;  // malformed locations: make progress, rows stay masked
    bool ok = q0 <= t && t < q1 && n >= q1 - q0 && n <= max_len;
    if (!ok) n = 0;
    sg.n = n;
    sg.q0 = q0;
    sg.pos0 = n - (q1 - q0);
    sg.kv_end = ok ? sg.pos0 + (sg.seg1 - 1 - q0) + 1 : 0;
    return ok;
  };

  if (warp == kPfWarps) {
    // ------------------------------- producer warp ------------------------------------------
    if (lane == 0) {
      int it = 0;
      bool alive = true;
      for (int64_t t = T0; t < T1 && alive;) {
        Seg sg;
        segment_at(t, sg);
        const int32_t* table = a.block_table + (int64_t)sg.b * a.bt_stride;
        const int n_tiles = (int)((sg.kv_end + kKeyTile - 1) / kKeyTile);
        for (int tile = 0; tile < n_tiles; ++tile, ++it) {
          const int s = it % kPfStages;
          const int round = it / kPfStages;
          if (round > 0 && !mbar_wait(&empty[s], (unsigned)((round - 1) & 1), a.err)) {
            raise_error(a.err, PA_DEVERR_TIMEOUT);
            alive = false;
            break;
          }
          uint32_t bytes = 0;
          int ys[kSub], yo[kSub];
#pragma unroll
          for (int sub = 0; sub < kSub; ++sub) {
            const int64_t k0 = (int64_t)tile * kKeyTile + sub * 16;
            ys[sub] = -1;
            if (k0 < sg.kv_end) {
              const int blk = __ldg(table + (k0 >> a.block_shift));
              if (blk < 0 || blk >= a.num_blocks) {
                raise_error(a.err, PA_DEVERR_BLOCK_ID);
              } else {
                ys[sub] = blk;
                yo[sub] = (int)(k0 & bmask);
                bytes += 2 * kHalves * kBoxBytes;
              }
            }
          }
          uint8_t* st = stages + s * kStageBytes;
          if (bytes == 0) {
            mbar_arrive(&full[s]);
          } else {
            mbar_arrive_expect_tx(&full[s], bytes);
#pragma unroll
            for (int sub = 0; sub < kSub; ++sub) {
              if (ys[sub] < 0) continue;
#pragma unroll
              for (int h = 0; h < kHalves; ++h) {
                const int off = (sub * kHalves + h) * kBoxBytes;
                tma_load_3d(st + off, &kmap, kvh * D + h * 64, yo[sub], ys[sub], &full[s]);
                tma_load_3d(st + kOpBytes + off, &vmap, kvh * D + h * 64, yo[sub], ys[sub], &full[s]);
              }
            }
          }
        }
        t = sg.seg1;
      }
    }
    return;
  }

  // --------------------------------- consumer warps -------------------------------------------
  const int g = lane >> 2, tig = lane & 3;
  // rows of this lane: r0 = 16 * warp + g, r1 = r0 + 8; row r <-> token T0 + r / G, head kvh*G + r % G
  const int r_lane[2] = {16 * warp + g, 16 * warp + g + 8};
  int64_t tok[2];
  int head[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    tok[i] = T0 + r_lane[i] / G;
    head[i] = kvh * G + r_lane[i] % G;
  }
  // Q rows of this warp into shared memory (swizzled), read back as A fragments by ldmatrix
  uint8_t* qs = stages + kPfStages * kStageBytes;
  {
    constexpr int kChunks = D / 8;
    for (int i = lane; i < 16 * kChunks; i += 32) {
      const int rr = i / kChunks, c = i % kChunks;
      const int r = 16 * warp + rr;
      const int64_t t = T0 + r / G;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (t < T1) {
        const T* qrow = static_cast<const T*>(a.q) + (t * a.n_q_heads + kvh * G + r % G) * D;
        v = __ldg(reinterpret_cast<const uint4*>(qrow + c * 8));
      }
      *reinterpret_cast<uint4*>(qs + q_offset<D>(r, c)) = v;
    }
    __syncwarp();
  }
  const uint32_t qb = smem_u32(qs);

  float o[kDTiles][4];
#pragma unroll
  for (int i = 0; i < kDTiles; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  int it = 0;
  bool alive = true;

  for (int64_t t = T0; t < T1 && alive;) {
    Seg sg;
    const bool seg_ok = segment_at(t, sg);
    if (!seg_ok && threadIdx.x == 0) raise_error(a.err, PA_DEVERR_QUERY_LOC);
    const int32_t* table = a.block_table + (int64_t)sg.b * a.bt_stride;
    // causal bound (inclusive) of this lane's two rows in this segment; -1 = row not in segment
    int64_t bound[2];
#pragma unroll
    for (int i = 0; i < 2; ++i)
      bound[i] = (seg_ok && tok[i] >= sg.seg0 && tok[i] < sg.seg1) ? sg.pos0 + (tok[i] - sg.q0) : -1;
    const int n_tiles = (int)((sg.kv_end + kKeyTile - 1) / kKeyTile);
    for (int tile = 0; tile < n_tiles; ++tile, ++it) {
      const int s = it % kPfStages;
      if (!mbar_wait(&full[s], (unsigned)((it / kPfStages) & 1), a.err)) {
        if (lane == 0) raise_error(a.err, PA_DEVERR_TIMEOUT);
        alive = false;
        break;
      }
      uint8_t* st = stages + s * kStageBytes;
      const int64_t kbase = (int64_t)tile * kKeyTile;
      // which 16-key sub-tiles hold data (present and with a valid block id)
      bool sub_ok[kSub];
#pragma unroll
      for (int sub = 0; sub < kSub; ++sub) {
        const int64_t k0 = kbase + sub * 16;
        bool okk = k0 < sg.kv_end;
        if (okk) {
          const int blk = __ldg(table + (k0 >> a.block_shift));
          okk = blk >= 0 && blk < a.num_blocks;
        }
        sub_ok[sub] = okk;
      }
      // V rows past the context (stale data of the last partial block) must not meet a zero
      // probability as NaN: zero them (every warp writes the same zeros before its own reads)
      if (kbase + kKeyTile > sg.n) {
        for (int i = lane; i < kKeyTile * 8 * kHalves; i += 32) {
          const int kk = i / (8 * kHalves);
          const int c = i % (8 * kHalves);
          const int64_t k0 = kbase + (kk & ~15);
          if (kbase + kk >= sg.n && k0 < sg.kv_end)
            *reinterpret_cast<uint4*>(st + kOpBytes + pf_offset<D>(kk, c)) = make_uint4(0, 0, 0, 0);
        }
        __syncwarp();
      }
      const uint32_t kb = smem_u32(st);
      const uint32_t vb = smem_u32(st + kOpBytes);
      // ---- S = Q K^T: 8 n-tiles of 8 keys, k-steps outermost (one Q fragment pair live) -------
      float sc[kKeyTile / 8][4];
#pragma unroll
      for (int nt = 0; nt < kKeyTile / 8; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < kKSteps; ks += 2) {
        uint32_t qf[2][4];
        const int mi = lane >> 3;
        const int qr = 16 * warp + (lane & 7) + 8 * (mi & 1);
#pragma unroll
        for (int j = 0; j < 2; ++j)
          ldsm_x4(qb + q_offset<D>(qr, 2 * (ks + j) + (mi >> 1)), qf[j][0], qf[j][1], qf[j][2], qf[j][3]);
#pragma unroll
        for (int nt = 0; nt < kKeyTile / 8; ++nt) {
          if (!sub_ok[nt >> 1]) continue;
          const int kk = nt * 8 + (lane & 7);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kb + pf_offset<D>(kk, 2 * ks + (lane >> 3)), b0, b1, b2, b3);
          mma_16816<kBf16>(sc[nt], qf[0][0], qf[0][1], qf[0][2], qf[0][3], b0, b1);
          mma_16816<kBf16>(sc[nt], qf[1][0], qf[1][1], qf[1][2], qf[1][3], b2, b3);
        }
      }
      // ---- causal mask, online softmax per row ------------------------------------------------
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int nt = 0; nt < kKeyTile / 8; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int i = e >> 1;
          const int64_t key = kbase + nt * 8 + 2 * tig + (e & 1);
          const bool keep = sub_ok[nt >> 1] && key <= bound[i];
          sc[nt][e] = keep ? sc[nt][e] * a.scale_log2 : -INFINITY;
          mx[i] = fmaxf(mx[i], sc[nt][e]);
        }
      }
      float corr[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 1));
        mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 2));
        const float m_new = fmaxf(m_run[i], mx[i]);
        const float m_use = m_new == -INFINITY ? 0.f : m_new;
        corr[i] = fast_exp2(m_run[i] - m_use);
        m_run[i] = m_new;
        mx[i] = m_use;
      }
      float rs[2] = {0.f, 0.f};
#pragma unroll
      for (int nt = 0; nt < kKeyTile / 8; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float p = fast_exp2(sc[nt][e] - mx[e >> 1]);
          sc[nt][e] = p;
          rs[e >> 1] += p;
        }
      }
#pragma unroll
      for (int i = 0; i < 2; ++i) l_run[i] = l_run[i] * corr[i] + rs[i];
      if (__any_sync(0xffffffffu, corr[0] != 1.f || corr[1] != 1.f)) {
#pragma unroll
        for (int d = 0; d < kDTiles; ++d) {
          o[d][0] *= corr[0];
          o[d][1] *= corr[0];
          o[d][2] *= corr[1];
          o[d][3] *= corr[1];
        }
      }
      // ---- O += P V: one k-step per 16-key sub-tile ------------------------------------------
#pragma unroll
      for (int sub = 0; sub < kSub; ++sub) {
        if (!sub_ok[sub]) continue;
        const uint32_t a0 = pack2<kBf16>(sc[2 * sub][0], sc[2 * sub][1]);
        const uint32_t a1 = pack2<kBf16>(sc[2 * sub][2], sc[2 * sub][3]);
        const uint32_t a2 = pack2<kBf16>(sc[2 * sub + 1][0], sc[2 * sub + 1][1]);
        const uint32_t a3 = pack2<kBf16>(sc[2 * sub + 1][2], sc[2 * sub + 1][3]);
        const int mi = lane >> 3;
        const int kk = sub * 16 + (lane & 7) + 8 * (mi & 1);
#pragma unroll
        for (int dt = 0; dt < kDTiles; dt += 2) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vb + pf_offset<D>(kk, dt + (mi >> 1)), b0, b1, b2, b3);
          mma_16816<kBf16>(o[dt], a0, a1, a2, a3, b0, b1);
          mma_16816<kBf16>(o[dt + 1], a0, a1, a2, a3, b2, b3);
        }
      }
      // release the stage to the producer
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    t = sg.seg1;
  }

  // ---- epilogue: normalise and store rows g and g+8 --------------------------------------------
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    l_run[i] += __shfl_xor_sync(0xffffffffu, l_run[i], 1);
    l_run[i] += __shfl_xor_sync(0xffffffffu, l_run[i], 2);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    if (tok[i] >= T1) continue;
    const float inv = l_run[i] != 0.f ? 1.f / l_run[i] : 0.f;
    T* orow = static_cast<T*>(a.out) + (tok[i] * a.n_q_heads + head[i]) * D;
#pragma unroll
    for (int d = 0; d < kDTiles; ++d) {
      const float v0 = o[d][2 * i] * inv, v1 = o[d][2 * i + 1] * inv;
      *reinterpret_cast<uint32_t*>(orow + d * 8 + 2 * tig) = pack2<kBf16>(v0, v1);
    }
  }
}

// ------------------------------------------------------------------------------------------------

bool prefill_tc_supported(pa_dtype dt, int block_size, int head_dim, int group, int64_t num_blocks) {
  return decode_tc_supported(dt, block_size, head_dim, group, num_blocks);
}

template <typename T, int D, int G>
static cudaError_t launch_pf_g(const AttnArgs& a, const CUtensorMap& km, const CUtensorMap& vm, cudaStream_t s) {
  constexpr int smem = PfCfg<D>::kSmemBytes;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(prefill_tc_kernel<T, D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  constexpr int qb = kPfRows / G;
  const int64_t grid = ((a.rows + qb - 1) / qb) * a.n_kv_heads;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  prefill_tc_kernel<T, D, G><<<(unsigned)grid, kPfThreads, smem, s>>>(a, km, vm);
  return cudaGetLastError();
}

template <typename T, int D>
static cudaError_t launch_pf_d(const AttnArgs& a, const CUtensorMap& km, const CUtensorMap& vm, cudaStream_t s) {
  switch (a.group) {
    case 1: return launch_pf_g<T, D, 1>(a, km, vm, s);
    case 2: return launch_pf_g<T, D, 2>(a, km, vm, s);
    case 4: return launch_pf_g<T, D, 4>(a, km, vm, s);
    case 8: return launch_pf_g<T, D, 8>(a, km, vm, s);
    case 16: return launch_pf_g<T, D, 16>(a, km, vm, s);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T>
static cudaError_t launch_pf_t(const AttnArgs& a, const CUtensorMap& km, const CUtensorMap& vm, cudaStream_t s) {
  return a.head_dim == 64 ? launch_pf_d<T, 64>(a, km, vm, s) : launch_pf_d<T, 128>(a, km, vm, s);
}

cudaError_t launch_prefill_tc(const AttnArgs& a, pa_dtype dt, cudaStream_t s, int* launches) {
  if (a.rows == 0) return cudaSuccess;
  CUtensorMap km, vm;
  if (!encode_pool_map(&km, a.k_pool, dt, a.num_blocks, a.block_size, a.n_kv_heads, a.head_dim, a.kv_block_stride) ||
      !encode_pool_map(&vm, a.v_pool, dt, a.num_blocks, a.block_size, a.n_kv_heads, a.head_dim, a.kv_block_stride))
    return cudaErrorInvalidValue;
  cudaError_t e = dt == PA_BF16 ? launch_pf_t<__nv_bfloat16>(a, km, vm, s) : launch_pf_t<__half>(a, km, vm, s);
  ++*launches;
  return e;
}

}  // namespace pa
