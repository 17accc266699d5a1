// Internal launch interface between the C ABI layer (abi.cu) and the kernel translation units.
// Host-only declarations; no torch types, no device code.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pagedattn.h"

namespace pa {

// Element size of an I/O dtype in bytes.
inline int dtype_bytes(pa_dtype dt) { return dt == PA_FP32 ? 4 : 2; }

// Record a CUDA error for pa_last_cuda_error() on this thread and return PA_ECUDA.
int fail_cuda(cudaError_t e);

// The calling thread's current CUDA context (identifies a device's context across resets).
int current_context(void** ctx);

struct KvWriteArgs {
  const void* k_new;
  const void* v_new;
  const int64_t* slot_mapping;
  int64_t n_tokens;
  void* k_pool;
  void* v_pool;
  int64_t total_slots;   // num_blocks * block_size
  int row_vecs;          // n_kv_heads * head_dim * elt / 16 (16-byte vectors per token row)
  int block_size;
  int64_t block_stride_vecs;  // 16-byte vectors from one block of a pool to the next
  unsigned* err;         // device error word
};

struct CopyBlocksArgs {
  void* k_pool;
  void* v_pool;
  const int64_t* pairs;
  int64_t n_pairs;
  int64_t num_blocks;
  int64_t block_vecs;    // block_bytes / 16
  int64_t block_stride_vecs;  // 16-byte vectors from one block of a pool to the next
  unsigned* err;
};

// Block transfer between two pools (either may be mapped pinned host memory).
struct SwapArgs {
  void* dst_k;
  void* dst_v;
  const void* src_k;
  const void* src_v;
  const int64_t* pairs;  // (src, dst)
  int64_t n_pairs;
  int64_t src_num_blocks;
  int64_t dst_num_blocks;
  int64_t block_vecs;    // block_bytes / 16
  int64_t block_stride_vecs;  // 16-byte vectors from one block of a pool to the next (both pools)
  unsigned* err;
};

// One attention launch over "rows": a decode row is a sequence, a prefill row is a query token.
struct AttnArgs {
  void* out;
  const void* q;
  const void* k_pool;
  const void* v_pool;
  const int32_t* block_table;
  int64_t bt_stride;
  const int32_t* context_lens;
  const int32_t* query_start_loc;  // nullptr for decode
  int batch;
  int64_t rows;                    // batch (decode) or total_q (prefill)
  int64_t num_blocks;
  int block_size;
  int block_shift;                 // log2(block_size)
  int64_t kv_block_stride;         // elements from one block of a pool to the next (separate pools:
                                   // block_size * n_kv_heads * head_dim; unified K/V blocks: twice that)
  float scale_log2;                // scale * log2(e)
  int n_q_heads;
  int n_kv_heads;
  int group;                       // n_q_heads / n_kv_heads
  int head_dim;
  // split-K (decode only)
  int part_tokens;                 // tokens per partition (multiple of block_size)
  int max_parts;                   // partitions per row in the grid (1 = no split)
  float* ws_m;                     // [rows * n_q_heads][max_parts]
  float* ws_l;                     // [rows * n_q_heads][max_parts]
  float* ws_acc;                   // [rows * n_q_heads][max_parts][head_dim]
  unsigned* err;                   // device error word pair ([0] bits, [1] epoch of a launch that gave up)
  unsigned epoch;                  // this launch's epoch (never 0): its bounded waits abort only on it
  // fused K/V write (decode only; all nullptr otherwise): sequence b's new token k_new[b], v_new[b]
  // ([batch][n_kv_heads][head_dim]) goes to pool row slot_mapping[b], which must be the slot of its
  // last context position; the CTA reading that position takes the row from k_new/v_new directly.
  const void* k_new;
  const void* v_new;
  const int64_t* slot_mapping;
  void* k_pool_w;                  // the pools again, writable
  void* v_pool_w;
};

struct MergeArgs {
  void* out;
  const float* part_m;
  const float* part_l;
  const float* part_acc;
  int64_t rows;                    // rows of [rows][n_parts]
  int n_parts;
  int head_dim;
  // when context_lens != nullptr, row r belongs to sequence r / heads_per_seq and only its first
  // ceil(len / part_tokens) partitions exist; rows with a single partition are skipped (the
  // partition kernel wrote them directly).
  const int32_t* context_lens;
  int heads_per_seq;
  int part_tokens;
  int64_t max_len;                 // clamp for context_lens (bt_stride * block_size)
};

// Launchers: return cudaSuccess or the launch error.  `launches` is incremented per kernel.
cudaError_t launch_kv_write(const KvWriteArgs& a, pa_dtype dt, cudaStream_t s, int* launches);
cudaError_t launch_copy_blocks(const CopyBlocksArgs& a, cudaStream_t s, int* launches);
cudaError_t launch_swap_blocks(const SwapArgs& a, cudaStream_t s, int* launches);
cudaError_t launch_attn_simt(const AttnArgs& a, pa_dtype dt, cudaStream_t s, int* launches);
cudaError_t launch_lse_merge(const MergeArgs& a, pa_dtype dt, cudaStream_t s, int* launches);

// TMA view of a pool: 3-D tensor (column = n_kv_heads * head_dim, token in block, block) with the
// pool's block stride, boxes of 64 columns x 16 tokens x 1 block, 128-byte swizzle.
bool encode_pool_map(CUtensorMap* map, const void* pool, pa_dtype dt, int64_t num_blocks, int block_size,
                     int n_kv_heads, int head_dim, int64_t block_stride);

// TMA view of the queries [total_q][n_q_heads][head_dim]: 3-D tensor (column, head, token), boxes of
// 64 columns x heads_box heads x tokens_box tokens, 128-byte swizzle, rows past total_q read as zeros.
bool encode_q_map(CUtensorMap* map, const void* q, pa_dtype dt, int64_t total_q, int n_q_heads, int head_dim,
                  int heads_box, int tokens_box);

// Tensor-core decode (TMA + mma.sync) for bf16/fp16 pools with block_size % 16 == 0.
bool decode_tc_supported(pa_dtype dt, int block_size, int head_dim, int group, int64_t num_blocks);
cudaError_t launch_decode_tc(const AttnArgs& a, pa_dtype dt, cudaStream_t s, int* launches);

// tcgen05 causal prefill (TMEM accumulators, TMA rings, warp-specialised) for bf16/fp16 pools with
// block_size % 16 == 0 (the support set of the tensor-core decode).
cudaError_t launch_prefill_umma(const AttnArgs& a, pa_dtype dt, cudaStream_t s, int* launches);

// Bounded-wait self-test (selftest.cu): one CTA whose two waits run out; see pa_selftest_bounded_wait.
cudaError_t launch_selftest_wait(unsigned* err, unsigned epoch, uint64_t limit_ns, unsigned long long* elapsed_ns,
                                 cudaStream_t s, int* launches);

}  // namespace pa
