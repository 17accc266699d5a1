// paged_kv_write: scatter this step's K/V rows into pool slots through slot_mapping.
// nanoserve "Day 19: the fused paged read wired into attention", "What I learned" 2 — the shared
// write scatters the K/V to this step's slots; "Diagram" — the write goes through slot_mapping.
//
// One thread moves one 16-byte vector of K and the matching vector of V.  The copy is a bit copy
// (no conversion), so the result is exact for every dtype.  A negative slot writes nothing; a slot
// past the pool is skipped and recorded in the device error word.
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

__global__ void __launch_bounds__(256) kv_write_kernel(const uint4* __restrict__ k_new,
                                                       const uint4* __restrict__ v_new,
                                                       const int64_t* __restrict__ slots,
                                                       int64_t n_tokens, uint4* __restrict__ k_pool,
                                                       uint4* __restrict__ v_pool, int64_t total_slots,
                                                       int row_vecs, int block_size, int64_t block_stride_vecs,
                                                       unsigned* err) {
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t total = n_tokens * row_vecs;
  if (idx >= total) return;
  const int64_t t = idx / row_vecs;
  const int c = (int)(idx - t * row_vecs);
  const int64_t slot = __ldg(slots + t);
  if (slot < 0) return;
  if (slot >= total_slots) {
    if (c == 0) raise_error(err, PA_DEVERR_SLOT);
    return;
  }
  const uint4 kv = __ldg(k_new + idx);
  const uint4 vv = __ldg(v_new + idx);
  const int64_t blk = slot / block_size;
  const int64_t row = blk * block_stride_vecs + (slot - blk * block_size) * row_vecs;
  k_pool[row + c] = kv;
  v_pool[row + c] = vv;
}

cudaError_t launch_kv_write(const KvWriteArgs& a, pa_dtype, cudaStream_t s, int* launches) {
  const int64_t total = a.n_tokens * a.row_vecs;
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  const int64_t blocks = (total + threads - 1) / threads;
  kv_write_kernel<<<(unsigned)blocks, threads, 0, s>>>(
      static_cast<const uint4*>(a.k_new), static_cast<const uint4*>(a.v_new), a.slot_mapping,
      a.n_tokens, static_cast<uint4*>(a.k_pool), static_cast<uint4*>(a.v_pool), a.total_slots,
      a.row_vecs, a.block_size, a.block_stride_vecs, a.err);
  ++*launches;
  return cudaGetLastError();
}

}  // namespace pa
