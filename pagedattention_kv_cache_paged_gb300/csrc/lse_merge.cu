// Log-sum-exp merge of split-K partials.
//
// Partition p of a row holds m_p (maximum score, log2 domain), l_p = sum 2^(s - m_p) and the
// unnormalised accumulator acc_p = sum 2^(s - m_p) v.  Rescaling every partition to the common
// maximum M = max_p m_p gives the exact softmax over the union:
//   out = sum_p acc_p 2^(m_p - M) / sum_p l_p 2^(m_p - M).
// This is the correction step of the single-pass softmax (JuliaPagedAttn README, "Online
// Softmax") applied to whole partitions instead of single tokens.  Partitions with l_p = 0 hold no
// token and are skipped; a row with none left is written as zeros.  A NaN anywhere in a partition
// propagates to the output, as it does in the two-pass definition.
//
// Few partitions per row (n_parts < kWideParts): one warp per output row; lanes own head_dim / 32
// consecutive elements.  Many (long contexts): one CTA of kWideWarps warps per row, the warps
// taking every kWideWarps-th partition with several 16-byte loads in flight each, then summing
// their shares in shared memory; the result is the same identity, summed in another order.
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

#ifndef PA_MERGE_WARPS
#define PA_MERGE_WARPS 4
#endif
constexpr int kMergeWarps = PA_MERGE_WARPS;  // rows (warps) per CTA of the one-warp-per-row merge

template <typename T, int D>
__global__ void __launch_bounds__(kMergeWarps * 32) lse_merge_kernel(const MergeArgs a) {
  constexpr int kPer = D / 32;
  constexpr int kSpec = 4;  // partitions whose accumulators are loaded before the count is known
  const int64_t row = (int64_t)blockIdx.x * kMergeWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  pdl_launch_dependents();  // the next step's decode grid may begin launching (it waits for this grid)
  pdl_wait_primary();       // partials of the partition kernel are complete and visible
  if (row >= a.rows) return;
  const float* pm = a.part_m + row * a.n_parts;
  const float* pl = a.part_l + row * a.n_parts;
  const float* pacc = a.part_acc + row * a.n_parts * (int64_t)D + lane * kPer;
  // Every load that does not depend on the partition count goes out at once (one round trip to
  // memory instead of three): the row's length, (max, sum) of partition `lane`, and this lane's
  // head_dim slice of the first kSpec partitions' accumulators.
  const int64_t seq = a.context_lens != nullptr ? row / a.heads_per_seq : 0;
  int64_t len = a.context_lens != nullptr ? __ldg(a.context_lens + seq) : 0;
  const float m_l = lane < a.n_parts ? pm[lane] : -INFINITY;
  const float l_l = lane < a.n_parts ? pl[lane] : 0.f;
  float accs[kSpec][kPer];
#pragma unroll
  for (int j = 0; j < kSpec; ++j)
#pragma unroll
    for (int i = 0; i < kPer; ++i) accs[j][i] = j < a.n_parts ? pacc[(int64_t)j * D + i] : 0.f;

  int parts = a.n_parts;
  if (a.context_lens != nullptr) {
    len = len < 0 ? 0 : (len > a.max_len ? a.max_len : len);
    parts = len == 0 ? 1 : (int)((len + a.part_tokens - 1) / a.part_tokens);
    if (parts <= 1) return;  // written directly by the partition kernel
  }
  // the row maximum over partitions that hold tokens: lane p looks at partitions p, p + 32, ...
  float M = lane < parts && l_l != 0.f ? m_l : -INFINITY;
  for (int p = lane + 32; p < parts; p += 32)
    if (pl[p] != 0.f) M = fmaxf(M, pm[p]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float L = 0.f;
  float acc[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) acc[i] = 0.f;
  if (M != -INFINITY) {
    for (int p0 = 0; p0 < parts; p0 += 32) {
      // weight of partition p0 + lane, then every lane accumulates its head_dim slice over the chunk
      const int p = p0 + lane;
      float w = 0.f;
      if (p < parts) {
        const float lp = p0 == 0 ? l_l : pl[p];
        if (lp != 0.f) {
          w = fast_exp2((p0 == 0 ? m_l : pm[p]) - M);
          L = fmaf(lp, w, L);
        }
      }
      const int n = parts - p0 < 32 ? parts - p0 : 32;
      if (p0 == 0) {
#pragma unroll
        for (int j = 0; j < kSpec; ++j) {
          const float wj = __shfl_sync(0xffffffffu, w, j);
          if (j < n && wj != 0.f) {
#pragma unroll
            for (int i = 0; i < kPer; ++i) acc[i] = fmaf(accs[j][i], wj, acc[i]);
          }
        }
      }
#pragma unroll 4
      for (int j = p0 == 0 ? kSpec : 0; j < n; ++j) {
        const float wj = __shfl_sync(0xffffffffu, w, j);
        if (wj != 0.f) {
          const float* src = pacc + (int64_t)(p0 + j) * D;
#pragma unroll
          for (int i = 0; i < kPer; ++i) acc[i] = fmaf(src[i], wj, acc[i]);
        }
      }
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
  const float inv = L != 0.f ? 1.f / L : 0.f;
  T* o = static_cast<T*>(a.out) + row * D + lane * kPer;
#pragma unroll
  for (int i = 0; i < kPer; ++i) o[i] = Elt<T>::from_float(acc[i] * inv);
}

constexpr int kWideParts = 16;
constexpr int kWideWarps = 8;

// Number of partitions of row `row` that hold partial states (1: the row was written directly by
// the partition kernel).
__device__ __forceinline__ int merge_parts(const MergeArgs& a, int64_t row) {
  if (a.context_lens == nullptr) return a.n_parts;
  const int64_t seq = row / a.heads_per_seq;
  int64_t len = __ldg(a.context_lens + seq);
  len = len < 0 ? 0 : (len > a.max_len ? a.max_len : len);
  return len == 0 ? 1 : (int)((len + a.part_tokens - 1) / a.part_tokens);
}

template <typename T, int D>
__global__ void __launch_bounds__(kWideWarps * 32) lse_merge_wide_kernel(const MergeArgs a) {
  constexpr int kPer = D / 32;  // elements per lane: 4 (one 16-byte load) or 2 (8 bytes)
  __shared__ float s_red[kWideWarps];
  __shared__ float s_acc[kWideWarps][D];
  __shared__ float s_l[kWideWarps];
  const int64_t row = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_launch_dependents();  // the next step's decode grid may begin launching (it waits for this grid)
  pdl_wait_primary();       // partials of the partition kernel are complete and visible
  const int parts = merge_parts(a, row);  // uniform over the CTA
  if (parts <= 1) return;
  const float* pm = a.part_m + row * a.n_parts;
  const float* pl = a.part_l + row * a.n_parts;
  const float* pacc = a.part_acc + row * a.n_parts * (int64_t)D + lane * kPer;
  // the row maximum over partitions that hold tokens
  float M = -INFINITY;
  for (int p = threadIdx.x; p < parts; p += kWideWarps * 32)
    if (pl[p] != 0.f) M = fmaxf(M, pm[p]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  if (lane == 0) s_red[warp] = M;
  __syncthreads();
  M = s_red[0];
#pragma unroll
  for (int w = 1; w < kWideWarps; ++w) M = fmaxf(M, s_red[w]);
  // warp w: partitions w, w + kWideWarps, ...
  float L = 0.f;
  float acc[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) acc[i] = 0.f;
  if (M != -INFINITY) {
#pragma unroll 4
    for (int p = warp; p < parts; p += kWideWarps) {
      const float lp = pl[p];
      if (lp != 0.f) {
        const float wp = fast_exp2(pm[p] - M);
        L = fmaf(lp, wp, L);
        const float* src = pacc + (int64_t)p * D;
        if constexpr (kPer == 4) {
          const float4 v = *reinterpret_cast<const float4*>(src);
          acc[0] = fmaf(v.x, wp, acc[0]);
          acc[1] = fmaf(v.y, wp, acc[1]);
          acc[2] = fmaf(v.z, wp, acc[2]);
          acc[3] = fmaf(v.w, wp, acc[3]);
        } else {
#pragma unroll
          for (int i = 0; i < kPer; ++i) acc[i] = fmaf(src[i], wp, acc[i]);
        }
      }
    }
  }
#pragma unroll
  for (int i = 0; i < kPer; ++i) s_acc[warp][lane * kPer + i] = acc[i];
  if (lane == 0) s_l[warp] = L;  // every lane of the warp holds the same L
  __syncthreads();
  float Lt = 0.f;
#pragma unroll
  for (int w = 0; w < kWideWarps; ++w) Lt += s_l[w];
  const float inv = Lt != 0.f ? 1.f / Lt : 0.f;
  T* o = static_cast<T*>(a.out) + row * D;
  for (int d = threadIdx.x; d < D; d += kWideWarps * 32) {
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < kWideWarps; ++w) v += s_acc[w][d];
    o[d] = Elt<T>::from_float(v * inv);
  }
}

template <typename T, int D>
static cudaError_t launch_merge_d(const MergeArgs& a, cudaStream_t s, unsigned blocks, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(kMergeWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  // (the wide kernel reads each lane's slice with one 16-byte load: needs a 16-byte aligned base)
  if (a.n_parts >= kWideParts && (reinterpret_cast<uintptr_t>(a.part_acc) & 15u) == 0) {
    cfg.gridDim = dim3((unsigned)a.rows);
    cfg.blockDim = dim3(kWideWarps * 32);
    return cudaLaunchKernelEx(&cfg, lse_merge_wide_kernel<T, D>, a);
  }
  return cudaLaunchKernelEx(&cfg, lse_merge_kernel<T, D>, a);
}

template <typename T>
static cudaError_t launch_merge_t(const MergeArgs& a, cudaStream_t s) {
  const int64_t blocks = (a.rows + kMergeWarps - 1) / kMergeWarps;
  if (blocks > 0x7fffffffLL || (a.n_parts >= kWideParts && a.rows > 0x7fffffffLL)) return cudaErrorInvalidConfiguration;
  const bool pdl = a.context_lens != nullptr;  // internal merge right after the partition kernel
  switch (a.head_dim) {
    case 64: return launch_merge_d<T, 64>(a, s, (unsigned)blocks, pdl);
    case 128: return launch_merge_d<T, 128>(a, s, (unsigned)blocks, pdl);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_lse_merge(const MergeArgs& a, pa_dtype dt, cudaStream_t s, int* launches) {
  if (a.rows == 0) return cudaSuccess;
  cudaError_t e;
  switch (dt) {
    case PA_BF16: e = launch_merge_t<__nv_bfloat16>(a, s); break;
    case PA_FP16: e = launch_merge_t<__half>(a, s); break;
    case PA_FP32: e = launch_merge_t<float>(a, s); break;
    default: return cudaErrorInvalidValue;
  }
  ++*launches;
  return e;
}

}  // namespace pa
