// copy_blocks: the copy step of a copy-on-write fork (JuliaPagedAttn README, "Copy-on-Write":
// allocate a new block, copy the data, update the table, decrement the refcount — the table and
// refcount bookkeeping stay on the host).
//
// Grid: x = pair, y = slice of the block.  Each thread moves up to kUnroll 16-byte vectors of K
// and of V, issuing all loads before the stores.  Pairs with an id outside the pool are skipped and
// recorded in the device error word.
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;

__global__ void __launch_bounds__(kCopyThreads) copy_blocks_kernel(uint4* __restrict__ k_pool,
                                                                   uint4* __restrict__ v_pool,
                                                                   const int64_t* __restrict__ pairs,
                                                                   int64_t num_blocks, int64_t block_vecs,
                                                                   int64_t block_stride_vecs, unsigned* err) {
  const int64_t p = blockIdx.x;
  const int64_t src = __ldg(pairs + 2 * p);
  const int64_t dst = __ldg(pairs + 2 * p + 1);
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (blockIdx.y == 0 && threadIdx.x == 0) raise_error(err, PA_DEVERR_COPY_PAIR);
    return;
  }
  const int64_t slice = (int64_t)kCopyThreads * kCopyUnroll;
  const int64_t base = (int64_t)blockIdx.y * slice + threadIdx.x;
  const uint4* ks = k_pool + src * block_stride_vecs;
  const uint4* vs = v_pool + src * block_stride_vecs;
  uint4* kd = k_pool + dst * block_stride_vecs;
  uint4* vd = v_pool + dst * block_stride_vecs;
  uint4 kb[kCopyUnroll], vb[kCopyUnroll];
#pragma unroll
  for (int u = 0; u < kCopyUnroll; ++u) {
    const int64_t i = base + (int64_t)u * kCopyThreads;
    if (i < block_vecs) {
      kb[u] = ld_stream16(ks + i);
      vb[u] = ld_stream16(vs + i);
    }
  }
#pragma unroll
  for (int u = 0; u < kCopyUnroll; ++u) {
    const int64_t i = base + (int64_t)u * kCopyThreads;
    if (i < block_vecs) {
      kd[i] = kb[u];
      vd[i] = vb[u];
    }
  }
}

cudaError_t launch_copy_blocks(const CopyBlocksArgs& a, cudaStream_t s, int* launches) {
  if (a.n_pairs == 0) return cudaSuccess;
  const int64_t slice = (int64_t)kCopyThreads * kCopyUnroll;
  const int64_t ny = (a.block_vecs + slice - 1) / slice;
  if (ny > 65535 || a.n_pairs > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  dim3 grid((unsigned)a.n_pairs, (unsigned)ny);
  copy_blocks_kernel<<<grid, kCopyThreads, 0, s>>>(static_cast<uint4*>(a.k_pool),
                                                   static_cast<uint4*>(a.v_pool), a.pairs,
                                                   a.num_blocks, a.block_vecs, a.block_stride_vecs, a.err);
  ++*launches;
  return cudaGetLastError();
}

}  // namespace pa

// ------------------------------------------------------------------------------------------------
// swap_blocks: copy blocks between two pools that may live in different memories — the device pool
// and a pinned host pool mapped into the device address space (Pico-vLLM dev log #5 "Paged
// Attention", swap_out / swap_in between the GPU pool and the pinned CPU pool).  One launch moves
// every (src, dst) pair; each thread keeps kSwapUnroll 16-byte vectors in flight, enough to cover
// the latency of the host link.
// ------------------------------------------------------------------------------------------------
namespace pa {

constexpr int kSwapThreads = 256;
constexpr int kSwapUnroll = 8;

__global__ void __launch_bounds__(kSwapThreads) swap_blocks_kernel(const SwapArgs a) {
  const int64_t p = blockIdx.x;
  const int64_t src = __ldg(a.pairs + 2 * p);
  const int64_t dst = __ldg(a.pairs + 2 * p + 1);
  if (src < 0 || src >= a.src_num_blocks || dst < 0 || dst >= a.dst_num_blocks) {
    if (blockIdx.y == 0 && threadIdx.x == 0) raise_error(a.err, PA_DEVERR_COPY_PAIR);
    return;
  }
  const int64_t slice = (int64_t)kSwapThreads * kSwapUnroll;
  const int64_t base = (int64_t)blockIdx.y * slice + threadIdx.x;
  const uint4* ks = static_cast<const uint4*>(a.src_k) + src * a.block_stride_vecs;
  const uint4* vs = static_cast<const uint4*>(a.src_v) + src * a.block_stride_vecs;
  uint4* kd = static_cast<uint4*>(a.dst_k) + dst * a.block_stride_vecs;
  uint4* vd = static_cast<uint4*>(a.dst_v) + dst * a.block_stride_vecs;
  uint4 kb[kSwapUnroll], vb[kSwapUnroll];
#pragma unroll
  for (int u = 0; u < kSwapUnroll; ++u) {
    const int64_t i = base + (int64_t)u * kSwapThreads;
    if (i < a.block_vecs) {
      kb[u] = ld_stream16(ks + i);
      vb[u] = ld_stream16(vs + i);
    }
  }
#pragma unroll
  for (int u = 0; u < kSwapUnroll; ++u) {
    const int64_t i = base + (int64_t)u * kSwapThreads;
    if (i < a.block_vecs) {
      kd[i] = kb[u];
      vd[i] = vb[u];
    }
  }
}

cudaError_t launch_swap_blocks(const SwapArgs& a, cudaStream_t s, int* launches) {
  if (a.n_pairs == 0) return cudaSuccess;
  const int64_t slice = (int64_t)kSwapThreads * kSwapUnroll;
  const int64_t ny = (a.block_vecs + slice - 1) / slice;
  if (ny > 65535 || a.n_pairs > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  swap_blocks_kernel<<<dim3((unsigned)a.n_pairs, (unsigned)ny), kSwapThreads, 0, s>>>(a);
  ++*launches;
  return cudaGetLastError();
}

}  // namespace pa
