// CUDA-core paged attention: decode rows (one query token per sequence) and prefill rows (one
// query token of a causal chunk), for every dtype and supported shape.
//
// What it computes — JuliaPagedAttn README, "Online Softmax": one pass over the context with a
// running maximum, a running sum and an accumulator rescaled when the maximum grows; output =
// accumulator / running sum.  The context is read through the block table (JuliaPagedAttn
// "Architecture": block-table indirection; "Block Layout"), the GQA repeat happens at read time
// (nanoserve Day 19, "What I learned" 4): one CTA serves the whole query group of a KV head, so
// each K/V row is loaded from HBM once per (row, KV head) and reused by the G query heads.
//
// Grid (1-D): blockIdx.x = (row * max_parts + part) * n_kv_heads + kv_head.  KV heads of the same
// (row, partition) are adjacent so that CTAs touching the same physical blocks run together.
// A row's tokens [0, len) are cut into partitions of part_tokens; a row with one partition writes
// its output directly, otherwise the CTA stores its partial state (max, sum, accumulator; log2
// domain) in the workspace for the log-sum-exp merge kernel.
//
// Inside a CTA each warp streams its own chunks of kRowsPerLoad * kUnroll tokens: a 16-byte vector
// per lane per token row (kLanesPerRow lanes cover one row of head_dim), kUnroll K and V loads in
// flight per lane, dot products reduced across the row's lanes with xor-shuffles, and one online
// softmax update per chunk.  The warps' states are merged through shared memory at the end.
#include <float.h>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

constexpr int kSimtWarps = 4;
constexpr int kSimtUnroll = 4;

template <typename T, int D, int G>
__global__ void __launch_bounds__(kSimtWarps * 32) attn_simt_kernel(const AttnArgs a) {
  constexpr int kVec = Elt<T>::kVec;          // elements per 16-byte vector
  constexpr int kLanesPerRow = D / kVec;      // lanes covering one K/V row
  constexpr int kRowsPerLoad = 32 / kLanesPerRow;
  constexpr int kChunk = kRowsPerLoad * kSimtUnroll;
  static_assert(kLanesPerRow <= 32 && 32 % kLanesPerRow == 0, "head_dim / vector width");

  __shared__ float sm_m[kSimtWarps][G];
  __shared__ float sm_l[kSimtWarps][G];
  __shared__ float sm_acc[kSimtWarps][G][D];

  const int kvh = blockIdx.x % a.n_kv_heads;
  const int64_t rest = blockIdx.x / a.n_kv_heads;
  const int part = (int)(rest % a.max_parts);
  const int64_t row = rest / a.max_parts;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int dsub = lane % kLanesPerRow;
  const int rsub = lane / kLanesPerRow;

  pdl_launch_dependents();  // the split-K merge may begin launching; it waits for this grid's results

  // ---- which sequence and how many keys this row sees --------------------------------------
  const int64_t max_len = a.bt_stride << a.block_shift;
  int b;
  int64_t len;
  if (a.query_start_loc == nullptr) {
    b = (int)row;
    len = __ldg(a.context_lens + b);
  } else {
    b = find_sequence(a.query_start_loc, a.batch, row);
    const int64_t q0 = __ldg(a.query_start_loc + b);
    const int64_t q1 = __ldg(a.query_start_loc + b + 1);
    const int64_t n = __ldg(a.context_lens + b);
    len = n - (q1 - q0) + (row - q0) + 1;  // causal bound of query r = row - q0
    if (row < q0 || row >= q1 || len < 1) {
      if (threadIdx.x == 0) raise_error(a.err, PA_DEVERR_QUERY_LOC);
      len = 0;
    }
  }
  if (len < 0 || len > max_len) {
    if (threadIdx.x == 0) raise_error(a.err, PA_DEVERR_CONTEXT_LEN);
    len = len < 0 ? 0 : max_len;
  }
  const int n_parts_row = len == 0 ? 1 : (int)((len + a.part_tokens - 1) / a.part_tokens);
  if (part >= n_parts_row) return;
  const int64_t t_begin = (int64_t)part * a.part_tokens;
  const int64_t t_end = min(t_begin + a.part_tokens, len);

  // ---- the query group, pre-scaled into the log2 domain ---------------------------------------
  const T* qrow = static_cast<const T*>(a.q) + (row * a.n_q_heads + (int64_t)kvh * G) * D;
  float qf[G][kVec];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(qrow + h * D + dsub * kVec));
    Elt<T>::unpack(v, qf[h]);
#pragma unroll
    for (int e = 0; e < kVec; ++e) qf[h][e] *= a.scale_log2;
  }

  float m[G], l[G], acc[G][kVec];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.f;
#pragma unroll
    for (int e = 0; e < kVec; ++e) acc[h][e] = 0.f;
  }

  const int32_t* table = a.block_table + (int64_t)b * a.bt_stride;
  const int64_t row_elems = (int64_t)a.n_kv_heads * D;  // elements per pool slot
  // fused write (decode rows only): the partition holding the last context position writes this
  // step's K/V row there and takes it straight from k_new / v_new
  int64_t new_row = -1, patch_pos = -1;  // new_row: element offset of the new token's pool row
  if (a.k_new != nullptr && a.query_start_loc == nullptr && len > 0 && part == n_parts_row - 1) {
    const int64_t last = len - 1;
    const int64_t s_new = __ldg(a.slot_mapping + b);
    const int blk_last = __ldg(table + (last >> a.block_shift));
    const int64_t expect = (blk_last >= 0 && blk_last < a.num_blocks)
                               ? ((int64_t)blk_last << a.block_shift) + (last & (a.block_size - 1)) : -2;
    if (s_new >= 0) {
      if (s_new == expect) {
        new_row = (int64_t)blk_last * a.kv_block_stride + (last & (a.block_size - 1)) * row_elems;
        patch_pos = last;
      } else if (threadIdx.x == 0) {
        raise_error(a.err, PA_DEVERR_SLOT);
      }
    }
  }
  const T* kbase = static_cast<const T*>(a.k_pool) + (int64_t)kvh * D + dsub * kVec;
  const T* vbase = static_cast<const T*>(a.v_pool) + (int64_t)kvh * D + dsub * kVec;
  const int bmask = a.block_size - 1;

  for (int64_t c0 = t_begin + (int64_t)warp * kChunk; c0 < t_end; c0 += (int64_t)kSimtWarps * kChunk) {
    uint4 kr[kSimtUnroll], vr[kSimtUnroll];
    bool valid[kSimtUnroll];
#pragma unroll
    for (int u = 0; u < kSimtUnroll; ++u) {
      const int64_t t = c0 + u * kRowsPerLoad + rsub;
      valid[u] = t < t_end;
      kr[u] = make_uint4(0, 0, 0, 0);
      vr[u] = make_uint4(0, 0, 0, 0);
      if (valid[u]) {
        const int blk = __ldg(table + (t >> a.block_shift));
        if (blk < 0 || blk >= a.num_blocks) {
          raise_error(a.err, PA_DEVERR_BLOCK_ID);
          valid[u] = false;
        } else if (t == patch_pos) {
          const int64_t off = ((int64_t)b * a.n_kv_heads + kvh) * D + dsub * kVec;
          kr[u] = __ldg(reinterpret_cast<const uint4*>(static_cast<const T*>(a.k_new) + off));
          vr[u] = __ldg(reinterpret_cast<const uint4*>(static_cast<const T*>(a.v_new) + off));
          const int64_t poff = new_row + (int64_t)kvh * D + dsub * kVec;
          *reinterpret_cast<uint4*>(static_cast<T*>(a.k_pool_w) + poff) = kr[u];
          *reinterpret_cast<uint4*>(static_cast<T*>(a.v_pool_w) + poff) = vr[u];
        } else {
          const int64_t off = (int64_t)blk * a.kv_block_stride + (t & bmask) * row_elems;
          kr[u] = ld_stream16(kbase + off);
          vr[u] = ld_stream16(vbase + off);
        }
      }
    }
    // scores s[u][h] (log2 domain) for this lane's token of each load
    float s[kSimtUnroll][G];
#pragma unroll
    for (int u = 0; u < kSimtUnroll; ++u) {
      float kf[kVec];
      Elt<T>::unpack(kr[u], kf);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float d = 0.f;
#pragma unroll
        for (int e = 0; e < kVec; ++e) d = fmaf(qf[h][e], kf[e], d);
#pragma unroll
        for (int off = kLanesPerRow / 2; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
        s[u][h] = valid[u] ? d : -INFINITY;
      }
    }
    // one online-softmax update per chunk, with a warp-uniform maximum per head
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float mx = s[0][h];
#pragma unroll
      for (int u = 1; u < kSimtUnroll; ++u) mx = fmaxf(mx, s[u][h]);
#pragma unroll
      for (int off = kLanesPerRow; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float m_new = fmaxf(m[h], mx);
      if (m_new == -INFINITY) continue;  // nothing valid yet (all ids in this chunk were bad)
      const float corr = fast_exp2(m[h] - m_new);  // m = -inf -> 0
      l[h] *= corr;
#pragma unroll
      for (int e = 0; e < kVec; ++e) acc[h][e] *= corr;
      m[h] = m_new;
    }
#pragma unroll
    for (int u = 0; u < kSimtUnroll; ++u) {
      float vf[kVec];
      Elt<T>::unpack(vr[u], vf);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float p = valid[u] ? fast_exp2(s[u][h] - m[h]) : 0.f;
        l[h] += p;
#pragma unroll
        for (int e = 0; e < kVec; ++e) acc[h][e] = fmaf(p, vf[e], acc[h][e]);
      }
    }
  }

  // ---- reduce the row groups of the warp, then the warps of the CTA -------------------------
#pragma unroll
  for (int h = 0; h < G; ++h) {
#pragma unroll
    for (int off = kLanesPerRow; off < 32; off <<= 1) {
      l[h] += __shfl_xor_sync(0xffffffffu, l[h], off);
#pragma unroll
      for (int e = 0; e < kVec; ++e) acc[h][e] += __shfl_xor_sync(0xffffffffu, acc[h][e], off);
    }
  }
  if (rsub == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
#pragma unroll
      for (int e = 0; e < kVec; ++e) sm_acc[warp][h][dsub * kVec + e] = acc[h][e];
    }
  }
  if (lane == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      sm_m[warp][h] = m[h];
      sm_l[warp][h] = l[h];
    }
  }
  __syncthreads();

  const bool direct = n_parts_row == 1;
  for (int i = threadIdx.x; i < G * D; i += kSimtWarps * 32) {
    const int h = i / D;
    const int d = i - h * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kSimtWarps; ++w)
      if (sm_l[w][h] != 0.f) M = fmaxf(M, sm_m[w][h]);
    float L = 0.f, A = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kSimtWarps; ++w) {
        if (sm_l[w][h] != 0.f) {
          const float f = fast_exp2(sm_m[w][h] - M);
          L = fmaf(sm_l[w][h], f, L);
          A = fmaf(sm_acc[w][h][d], f, A);
        }
      }
    }
    const int64_t qh = row * a.n_q_heads + (int64_t)kvh * G + h;  // global (row, query head)
    if (direct) {
      T* o = static_cast<T*>(a.out) + qh * D + d;
      *o = Elt<T>::from_float(L != 0.f ? A / L : 0.f);
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

template <typename T, int D>
static cudaError_t launch_simt_g(const AttnArgs& a, cudaStream_t s) {
  const int64_t grid = a.rows * (int64_t)a.max_parts * a.n_kv_heads;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const dim3 blk(kSimtWarps * 32);
  switch (a.group) {
    case 1: attn_simt_kernel<T, D, 1><<<(unsigned)grid, blk, 0, s>>>(a); break;
    case 2: attn_simt_kernel<T, D, 2><<<(unsigned)grid, blk, 0, s>>>(a); break;
    case 4: attn_simt_kernel<T, D, 4><<<(unsigned)grid, blk, 0, s>>>(a); break;
    case 8: attn_simt_kernel<T, D, 8><<<(unsigned)grid, blk, 0, s>>>(a); break;
    case 16: attn_simt_kernel<T, D, 16><<<(unsigned)grid, blk, 0, s>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

template <typename T>
static cudaError_t launch_simt_t(const AttnArgs& a, cudaStream_t s) {
  switch (a.head_dim) {
    case 64: return launch_simt_g<T, 64>(a, s);
    case 128: return launch_simt_g<T, 128>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_attn_simt(const AttnArgs& a, pa_dtype dt, cudaStream_t s, int* launches) {
  if (a.rows == 0) return cudaSuccess;
  cudaError_t e;
  switch (dt) {
    case PA_BF16: e = launch_simt_t<__nv_bfloat16>(a, s); break;
    case PA_FP16: e = launch_simt_t<__half>(a, s); break;
    case PA_FP32: e = launch_simt_t<float>(a, s); break;
    default: return cudaErrorInvalidValue;
  }
  ++*launches;
  return e;
}

}  // namespace pa
