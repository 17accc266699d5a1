// tcgen05 causal chunked prefill over a paged history (bf16/fp16, block_size % 16 == 0).
//
// Computes the same thing as prefill_tc.cu — JuliaPagedAttn README "Features" (batched prefill)
// with the online softmax of "Online Softmax": the chunk of m_b queries holds the last m_b
// positions of sequence b's context and query r attends to positions 0 .. n_b - m_b + r through
// the block table — on the 5th-generation tensor cores with accumulators in tensor memory.
//
// CTA = 128 (query token, head) rows of one KV head (kRows / G tokens x the G heads of the group:
// read-time GQA, nanoserve Day 19 "What I learned" 4), 6 warps:
//   warps 0-3  softmax: thread t owns row t = TMEM lane t; loads its Q row to shared memory, turns
//              each S tile into probabilities, rescales O in TMEM when its running max grows,
//              writes P (bf16) to shared memory, and normalises O at the end;
//   warp 4     producer: TMA loads of 128-key K and V tiles (boxes of 16 keys x 64 columns from the
//              physical blocks the table names) into a 2-stage ring;
//   warp 5     MMA: allocates TMEM (S: 128 columns, O: head_dim columns) and issues
//              S = Q K^T (M 128, N 128) and O += P V (M 128, N head_dim, V as an MN-major operand)
//              with tcgen05.mma, signalling completion through tcgen05.commit.
// Handoffs: kv_full/kv_empty (producer <-> MMA), s_full (MMA -> softmax), p_full (softmax -> MMA),
// pv_done (MMA -> softmax).  Every wait is bounded (PA_DEVERR_TIMEOUT); TMEM is always released.
#include <cudaTypedefs.h>

#include "pa_common.cuh"
#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {

constexpr int kUmThreads = 192;
constexpr int kUmRows = 128;   // M of both products
constexpr int kUmKeys = 128;   // keys per tile
constexpr int kUmSub = kUmKeys / 16;
constexpr int kUmStages = 2;
constexpr int kUmTmemCols = 256;
constexpr int kUmHalf = 128 * 128;  // bytes of one 64-column half of a 128-row operand

template <int D>
struct UmCfg {
  static constexpr int kHalves = D / 64;
  static constexpr int kOpBytes = kUmKeys * D * 2;
  static constexpr int kStageBytes = 2 * kOpBytes;
  static constexpr int kQBytes = kUmRows * D * 2;
  static constexpr int kPBytes = kUmRows * kUmKeys * 2;
  static constexpr int kSmemBytes = 1024 + 1024 + kUmStages * kStageBytes + kQBytes + kPBytes;
};

// Byte offset of (row r in 0..127, 8-element chunk c) in a [half][row][128 B] swizzled operand.
__device__ __forceinline__ uint32_t um_off(int r, int c) {
  return (uint32_t)((c >> 3) * kUmHalf + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

template <typename T, int D, int G>
__global__ void __launch_bounds__(kUmThreads, 1)
    prefill_umma_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap) {
  constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
  constexpr int kHalves = UmCfg<D>::kHalves;
  constexpr int kOpBytes = UmCfg<D>::kOpBytes;
  constexpr int kStageBytes = UmCfg<D>::kStageBytes;
  constexpr int kQB = kUmRows / G;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(base);
  uint64_t* kv_full = bars;       // [2]
  uint64_t* kv_empty = bars + 2;  // [2]
  uint64_t* q_ready = bars + 4;
  uint64_t* s_full = bars + 5;
  uint64_t* p_full = bars + 6;
  uint64_t* pv_done = bars + 7;
  uint64_t* fin = bars + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + 512);
  uint8_t* stages = base + 1024;
  uint8_t* qs = stages + kUmStages * kStageBytes;
  uint8_t* ps = qs + UmCfg<D>::kQBytes;

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
    mbar_init(&kv_full[0], 1);
    mbar_init(&kv_full[1], 1);
    mbar_init(&kv_empty[0], 1);
    mbar_init(&kv_empty[1], 1);
    mbar_init(q_ready, 128);
    mbar_init(s_full, 1);
    mbar_init(p_full, 128);
    mbar_init(pv_done, 1);
    mbar_init(fin, 1);
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 5) tmem_alloc(tmem_slot, kUmTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem;
  const uint32_t tO = tmem + 128;

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

  if (warp == 4) {
    // --------------------------------------- producer -------------------------------------------
    if (lane == 0) {
      int i = 0;
      bool alive = true;
      for (int64_t t = T0; t < T1 && alive;) {
        const Seg sg = segment_at(t);
        const int32_t* table = a.block_table + (int64_t)sg.b * a.bt_stride;
        const int nt = tiles_of(sg);
        for (int tile = 0; tile < nt; ++tile, ++i) {
          const int s = i & 1;
          if (i >= 2 && !mbar_wait(&kv_empty[s], (unsigned)(((i >> 1) - 1) & 1), a.err)) {
            raise_error(a.err, PA_DEVERR_TIMEOUT);
            alive = false;
            break;
          }
          int ys[kUmSub];
          uint32_t bytes = 0;
#pragma unroll
          for (int sub = 0; sub < kUmSub; ++sub) {
            const int64_t k0 = (int64_t)tile * kUmKeys + sub * 16;
            ys[sub] = -1;
            if (k0 < sg.kv_end) {
              const int blk = __ldg(table + (k0 >> a.block_shift));
              if (blk < 0 || blk >= a.num_blocks) {
                raise_error(a.err, PA_DEVERR_BLOCK_ID);
              } else {
                ys[sub] = (int)(((int64_t)blk << a.block_shift) + (k0 & bmask));
                bytes += 2 * kHalves * 2048;
              }
            }
          }
          uint8_t* st = stages + s * kStageBytes;
          if (bytes == 0) {
            mbar_arrive(&kv_full[s]);
          } else {
            mbar_arrive_expect_tx(&kv_full[s], bytes);
#pragma unroll
            for (int sub = 0; sub < kUmSub; ++sub) {
              if (ys[sub] < 0) continue;
#pragma unroll
              for (int h = 0; h < kHalves; ++h) {
                const int off = h * kUmHalf + sub * 2048;
                tma_load_2d(st + off, &kmap, kvh * D + h * 64, ys[sub], &kv_full[s]);
                tma_load_2d(st + kOpBytes + off, &vmap, kvh * D + h * 64, ys[sub], &kv_full[s]);
              }
            }
          }
        }
        t = sg.seg1;
      }
    }
  } else if (warp == 5) {
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
      const uint32_t q_addr = smem_u32(qs), p_addr = smem_u32(ps);
      auto issue_s = [&](int i) {
        const uint32_t k_addr = smem_u32(stages + (i & 1) * kStageBytes);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = (ks >> 2) * kUmHalf + (ks & 3) * 32;
          umma_ss(tS, umma_desc_sw128(q_addr + off, 16, 1024), umma_desc_sw128(k_addr + off, 16, 1024), id_s,
                  ks > 0 ? 1u : 0u);
        }
        umma_commit(s_full);
      };
      bool alive = mbar_wait(q_ready, 0, a.err);
      if (alive && n_all > 0) {
        alive = mbar_wait(&kv_full[0], 0, a.err);
        if (alive) {
          tc_fence_after();
          issue_s(0);
        }
      }
      for (int i = 0; i < n_all && alive; ++i) {
        if (!mbar_wait(p_full, (unsigned)(i & 1), a.err)) {
          alive = false;
          break;
        }
        tc_fence_after();
        const uint32_t v_addr = smem_u32(stages + (i & 1) * kStageBytes + kOpBytes);
#pragma unroll
        for (int ks = 0; ks < kUmKeys / 16; ++ks) {
          const uint32_t aoff = (ks >> 2) * kUmHalf + (ks & 3) * 32;
          umma_ss(tO, umma_desc_sw128(p_addr + aoff, 16, 1024),
                  umma_desc_sw128(v_addr + ks * 2048, kUmHalf, 1024), id_pv, (i > 0 || ks > 0) ? 1u : 0u);
        }
        umma_commit(pv_done);
        umma_commit(&kv_empty[i & 1]);
        if (i + 1 < n_all) {
          if (!mbar_wait(&kv_full[(i + 1) & 1], (unsigned)(((i + 1) >> 1) & 1), a.err)) {
            alive = false;
            break;
          }
          tc_fence_after();
          issue_s(i + 1);
        }
      }
      if (!alive) raise_error(a.err, PA_DEVERR_TIMEOUT);
      if (n_all > 0) {
        umma_commit(fin);  // every MMA issued above has completed once this phase completes
        mbar_wait(fin, 0, a.err);
      }
    }
  } else {
    // ---------------------------------------- softmax -------------------------------------------
    const int r = threadIdx.x;  // row = TMEM lane
    const int64_t tok = T0 + r / G;
    const int head = kvh * G + r % G;
    {
      const uint4* qrow = reinterpret_cast<const uint4*>(static_cast<const T*>(a.q) + (tok * a.n_q_heads + head) * D);
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        const uint4 v = tok < T1 ? __ldg(qrow + c) : make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(qs + um_off(r, c)) = v;
      }
      fence_proxy_async_smem();
      mbar_arrive(q_ready);
    }
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
    float m_run = -INFINITY, l_run = 0.f;
    int i = 0;
    bool alive = true;
    for (int64_t t = T0; t < T1 && alive;) {
      const Seg sg = segment_at(t);
      if (!sg.ok && r == 0) raise_error(a.err, PA_DEVERR_QUERY_LOC);
      const int32_t* table = a.block_table + (int64_t)sg.b * a.bt_stride;
      const int64_t seg0 = t;
      const int64_t bound = (sg.ok && tok >= seg0 && tok < sg.seg1) ? sg.pos0 + (tok - sg.q0) : -1;
      const int nt = tiles_of(sg);
      for (int tile = 0; tile < nt; ++tile, ++i) {
        const int64_t kb = (int64_t)tile * kUmKeys;
        unsigned loaded = 0;  // bit per 16-key sub-tile holding data
#pragma unroll
        for (int sub = 0; sub < kUmSub; ++sub) {
          const int64_t k0 = kb + sub * 16;
          if (k0 < sg.kv_end) {
            const int blk = __ldg(table + (k0 >> a.block_shift));
            if (blk >= 0 && blk < a.num_blocks) loaded |= 1u << sub;
          }
        }
        if (!__all_sync(0xffffffffu, mbar_wait(s_full, (unsigned)(i & 1), a.err))) {
          alive = false;
          break;
        }
        tc_fence_after();
        // ---- S row -> masked, scaled scores (log2 domain) ------------------------------------
        float x[kUmKeys];
#pragma unroll
        for (int c0 = 0; c0 < kUmKeys; c0 += 32) {
          uint32_t v[32];
          tmem_ld32(tS + lane_base + c0, v);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) x[c0 + j] = __uint_as_float(v[j]);
        }
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < kUmKeys; ++c) {
          const bool keep = ((loaded >> (c >> 4)) & 1u) && (kb + c <= bound);
          x[c] = keep ? x[c] * a.scale_log2 : -INFINITY;
          mx = fmaxf(mx, x[c]);
        }
        const float m_new = fmaxf(m_run, mx);
        const float m_use = m_new == -INFINITY ? 0.f : m_new;
        const float corr = fast_exp2(m_run - m_use);
        m_run = m_new;
        float rs = 0.f;
#pragma unroll
        for (int c = 0; c < kUmKeys; ++c) {
          x[c] = fast_exp2(x[c] - m_use);
          rs += x[c];
        }
        l_run = l_run * corr + rs;
        // ---- wait for the previous P V (O stable, P buffer free), then rescale O -------------------
        if (i > 0) {
          if (!__all_sync(0xffffffffu, mbar_wait(pv_done, (unsigned)((i - 1) & 1), a.err))) {
            alive = false;
            break;
          }
          tc_fence_after();
          if (__any_sync(0xffffffffu, corr != 1.f)) {
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
              uint32_t v[32];
              tmem_ld32(tO + lane_base + c0, v);
              tmem_wait_ld();
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * corr);
              tmem_st32(tO + lane_base + c0, v);
            }
            tmem_wait_st();
          }
        }
        // ---- V rows that hold no data or lie past the context become zeros ------------------------
        if (kb + kUmKeys > sg.n || loaded != (1u << kUmSub) - 1u) {
          if (!__all_sync(0xffffffffu, mbar_wait(&kv_full[i & 1], (unsigned)((i >> 1) & 1), a.err))) {
            alive = false;
            break;
          }
          uint8_t* vst = stages + (i & 1) * kStageBytes + kOpBytes;
          for (int e = r; e < kUmKeys * 8 * kHalves; e += 128) {
            const int key = e / (8 * kHalves);
            const int c = e % (8 * kHalves);
            if (kb + key >= sg.n || !((loaded >> (key >> 4)) & 1u))
              *reinterpret_cast<uint4*>(vst + um_off(key, c)) = make_uint4(0, 0, 0, 0);
          }
        }
        // ---- P row (bf16/fp16) into shared memory --------------------------------------------------
#pragma unroll
        for (int c = 0; c < kUmKeys / 8; ++c) {
          uint4 w;
          w.x = pack2<kBf16>(x[8 * c + 0], x[8 * c + 1]);
          w.y = pack2<kBf16>(x[8 * c + 2], x[8 * c + 3]);
          w.z = pack2<kBf16>(x[8 * c + 4], x[8 * c + 5]);
          w.w = pack2<kBf16>(x[8 * c + 6], x[8 * c + 7]);
          *reinterpret_cast<uint4*>(ps + um_off(r, c)) = w;
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(p_full);
      }
      t = sg.seg1;
    }
    if (!alive && lane == 0) raise_error(a.err, PA_DEVERR_TIMEOUT);
    // ---- epilogue: O / l for this row ----------------------------------------------------------------
    if (alive && i > 0) {
      alive = __all_sync(0xffffffffu, mbar_wait(pv_done, (unsigned)((i - 1) & 1), a.err));
      tc_fence_after();
    }
    const float inv = (alive && l_run != 0.f) ? 1.f / l_run : 0.f;
    T* orow = static_cast<T*>(a.out) + (tok * a.n_q_heads + head) * D;
#pragma unroll
    for (int c0 = 0; c0 < D; c0 += 32) {
      uint32_t v[32];
      tmem_ld32(tO + lane_base + c0, v);
      tmem_wait_ld();
      if (tok < T1) {
#pragma unroll
        for (int j = 0; j < 32; j += 8) {
          uint4 w;
          w.x = pack2<kBf16>(__uint_as_float(v[j]) * inv, __uint_as_float(v[j + 1]) * inv);
          w.y = pack2<kBf16>(__uint_as_float(v[j + 2]) * inv, __uint_as_float(v[j + 3]) * inv);
          w.z = pack2<kBf16>(__uint_as_float(v[j + 4]) * inv, __uint_as_float(v[j + 5]) * inv);
          w.w = pack2<kBf16>(__uint_as_float(v[j + 6]) * inv, __uint_as_float(v[j + 7]) * inv);
          *reinterpret_cast<uint4*>(orow + c0 + j) = w;
        }
      }
    }
    // rows that saw no key (l = 0) were never written by P V: O holds no data, write zeros
    if (tok < T1 && i == 0) {
#pragma unroll
      for (int c = 0; c < D / 8; ++c) reinterpret_cast<uint4*>(orow)[c] = make_uint4(0, 0, 0, 0);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kUmTmemCols);
  }
}

// ------------------------------------------------------------------------------------------------
bool encode_pool_map(CUtensorMap* map, const void* pool, pa_dtype dt, int64_t num_blocks, int block_size,
                     int n_kv_heads, int head_dim);

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
  if (!encode_pool_map(&km, a.k_pool, dt, a.num_blocks, a.block_size, a.n_kv_heads, a.head_dim) ||
      !encode_pool_map(&vm, a.v_pool, dt, a.num_blocks, a.block_size, a.n_kv_heads, a.head_dim))
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
