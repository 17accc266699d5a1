/*
 * pagedattn.h — C ABI of the paged KV-cache attention library (libpagedattn.so).
 *
 * The library implements the device hot path of PagedAttention over a block-table-indexed KV cache
 * on one GPU (sm_103a): the slot-mapped K/V write, decode attention straight from scattered
 * physical blocks (read-time GQA, single-pass online softmax, split-K with an exact log-sum-exp
 * merge), causal chunked prefill over a paged history, and the block copy used by copy-on-write
 * forks.
 *
 * Conventions shared by every call
 * --------------------------------
 * Memory.  Every pointer argument is a DEVICE pointer unless stated otherwise.  The caller owns all
 *   buffers (pools, tables, outputs, workspace); the library allocates nothing and frees nothing.
 *   Each call is asynchronous on `stream` (a cudaStream_t passed as void*; NULL = legacy default
 *   stream) and returns after enqueueing its kernels.
 * Pools.  A K pool and a V pool are each a contiguous array [num_blocks][block_size][n_kv_heads]
 *   [head_dim] of the I/O dtype (Pico-vLLM dev log #5 "Paged Attention", core data structures:
 *   the device cache tensor is indexed block, token-in-block, kv head, head dim; JuliaPagedAttn
 *   README, "Block Layout": a block holds block_size consecutive tokens for every KV head).
 *   Pool base pointers must be 16-byte aligned.
 * Block stride and unified K/V blocks.  The calls above take contiguous pools: block b of a pool
 *   starts b * block bytes after its base (block bytes = block_size * n_kv_heads * head_dim *
 *   element size).  Each has an `_ex` twin whose optional pa_opts says how far apart the blocks
 *   of each pool lie (kv_block_stride_bytes), so the same kernels also read pools whose blocks are
 *   interleaved with other data.  The case the pages name is unified K/V blocks (JuliaPagedAttn
 *   README, "Features": keys and values of a token in one block, a single block table and pool):
 *   one pool [num_blocks][2][block_size][n_kv_heads][head_dim] where physical block b holds the
 *   keys of its block_size tokens followed by their values.  Pass k_pool = the pool's base,
 *   v_pool = k_pool + block bytes and kv_block_stride_bytes = 2 * block bytes.  Slots, tables,
 *   block ids and results are the same as with separate pools.  The stride is a per-call argument:
 *   calls with different layouts may run concurrently from any number of threads.
 * Slots.  Logical position j of sequence b lives in slot
 *   block_table[b * block_table_stride + j / block_size] * block_size + j % block_size,
 *   i.e. row `slot` of the pool viewed as [num_blocks * block_size][n_kv_heads][head_dim].
 * Tables.  block_table is int32 [batch][block_table_stride] (Pico-vLLM dev log #5,
 *   get_block_table: int32 physical ids); entries past ceil(context_lens[b] / block_size) are never
 *   read.  context_lens is int32 [batch] and counts the token(s) just written (Pico-vLLM dev log
 *   #5: the current token's K/V already exist in every layer, hence the +1 correction).
 * GQA.  n_q_heads must be a multiple of n_kv_heads; query head i reads KV head
 *   i / (n_q_heads / n_kv_heads).  The cache stores only the KV heads and the repeat happens at
 *   read time (nanoserve "Day 19: the fused paged read wired into attention", "What I learned" 4).
 * Dtypes.  q, pools and out share one dtype (PA_BF16, PA_FP16 or PA_FP32); scores, softmax
 *   statistics and accumulators are fp32; outputs are rounded to nearest-even.
 * Supported shapes.  head_dim in {64, 128}; block_size a power of two in [1, 256];
 *   n_q_heads / n_kv_heads in {1, 2, 4, 8, 16}.  Other shapes return PA_EUNSUPPORTED.
 * Errors.  0 = success.  Negative values (PA_E*) mean nothing was launched, except PA_ECUDA,
 *   which reports a launch failure (pa_last_cuda_error() gives the cudaError_t).  Device code never
 *   traps: an out-of-range block id, slot or copy pair met on the device is skipped (treated as
 *   masked) and recorded in a device error word that pa_device_error_flags() reads back.  With
 *   checked mode on (pa_set_checked_mode(1)) each call first copies its index arrays to the host,
 *   synchronizing `stream`, and returns PA_ERANGE without launching if any index, length or
 *   duplicate is invalid.
 * State.  The library keeps no state that changes what a call computes other than the checked-mode
 *   flag.  It also holds, per device, the device error word and the address lookups it needs to
 *   launch (tensor-map encoder, SM count), none of which alters results.
 */
#ifndef PAGEDATTN_H_
#define PAGEDATTN_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PA_API __attribute__((visibility("default")))
#else
#define PA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { PA_BF16 = 0, PA_FP16 = 1, PA_FP32 = 2 } pa_dtype;

enum {
  PA_OK = 0,
  PA_EINVAL = -1,        /* null pointer, negative or inconsistent size, heads not divisible */
  PA_EDTYPE = -2,        /* dtype not one of pa_dtype */
  PA_ERANGE = -3,        /* checked mode: block id / slot / length / pair out of range or duplicate */
  PA_EWORKSPACE = -4,    /* workspace given but smaller than required or not 16-byte aligned */
  PA_ECUDA = -5,         /* a CUDA launch failed; see pa_last_cuda_error() */
  PA_EUNSUPPORTED = -6   /* shape outside the supported set (see "Supported shapes") */
};

/* Bits of the device error word (pa_device_error_flags). */
enum {
  PA_DEVERR_BLOCK_ID = 1,     /* a table entry inside a context was < 0 or >= num_blocks */
  PA_DEVERR_SLOT = 2,         /* a slot >= num_blocks * block_size */
  PA_DEVERR_CONTEXT_LEN = 4,  /* context_lens[b] < 0 or > block_table_stride * block_size */
  PA_DEVERR_COPY_PAIR = 8,    /* a copy pair with src or dst outside [0, num_blocks) */
  PA_DEVERR_QUERY_LOC = 16,   /* query_start_loc not non-decreasing, or a chunk longer than its context */
  PA_DEVERR_TIMEOUT = 32      /* a bounded wait in a pipelined kernel gave up (the kernel returned early) */
};

/* Options for pa_set_option / pa_get_option.  The only process-wide option is the checked mode. */
enum {
  PA_OPT_CHECKED = 1           /* 0 (default) or 1: host-side validation before each launch */
};

/*
 * Per-call options of the `_ex` entry points.  A NULL pointer, or a zero-filled struct, means the
 * defaults; nothing here outlives the call.  Invalid values return PA_EINVAL.
 *   kv_block_stride_bytes  distance between consecutive blocks of each pool, a multiple of 16 and
 *                          at least the block bytes; 0 = the block bytes (contiguous pools).  See
 *                          "Block stride and unified K/V blocks".
 *   decode_kernel          0 auto (tensor cores for bf16/fp16 pools with block_size % 16 == 0, else
 *                          CUDA cores), 1 CUDA cores, 2 tensor cores (PA_EUNSUPPORTED if the shape
 *                          does not allow them)
 *   prefill_kernel         0 auto (tcgen05 tensor cores where the shape allows, else CUDA cores),
 *                          1 CUDA cores, 2 tcgen05 (PA_EUNSUPPORTED if the shape does not allow it)
 *   partition_tokens       split-K partition length in tokens, rounded up to block_size, at most
 *                          2^30; 0 = automatic (see paged_attention_decode_workspace_size)
 *   reserved               must be 0
 */
typedef struct pa_opts {
  int64_t kv_block_stride_bytes;
  int32_t decode_kernel;
  int32_t prefill_kernel;
  int32_t partition_tokens;
  int32_t reserved;
} pa_opts;

/*
 * paged_kv_write — scatter this step's K/V into the pools through slot_mapping.
 * Source: nanoserve Day 19, "What I learned" 2 (the shared write scatters the K/V to this step's
 * slots) and "Diagram" (the write goes through slot_mapping); JuliaPagedAttn README, API
 * "write_kv_cache!".
 *   k_new, v_new   [n_tokens][n_kv_heads][head_dim], dtype, contiguous (read only)
 *   slot_mapping   int64 [n_tokens]; token t is written to pool row slot_mapping[t]; a negative
 *                  slot writes nothing for that token.  Slots must be distinct (duplicates race;
 *                  checked mode rejects them).
 *   k_pool, v_pool pools as above (written in place).  The copy is bit-exact.
 * n_tokens == 0 is a no-op returning PA_OK.
 */
PA_API int paged_kv_write(const void* k_new, const void* v_new, const int64_t* slot_mapping, int64_t n_tokens,
                   void* k_pool, void* v_pool, int64_t num_blocks, int block_size, int n_kv_heads,
                   int head_dim, pa_dtype dtype, void* stream);
/* paged_kv_write with per-call options (opts may be NULL; only kv_block_stride_bytes applies). */
PA_API int paged_kv_write_ex(const void* k_new, const void* v_new, const int64_t* slot_mapping, int64_t n_tokens,
                             void* k_pool, void* v_pool, int64_t num_blocks, int block_size, int n_kv_heads,
                             int head_dim, pa_dtype dtype, const pa_opts* opts, void* stream);

/*
 * paged_attention_decode — one query token per sequence attends over its whole paged context.
 * Source: JuliaPagedAttn README, API "paged_attention_cpu!(O, Q, K_cache, V_cache, block_table,
 * context_lengths, layer, scale)" and "Online Softmax"; nanoserve Day 19 "What I added today"
 * (paged_attention(layer, k, v, q, n_rep, scale)).
 *   out            [batch][n_q_heads][head_dim], dtype (written)
 *   q              [batch][n_q_heads][head_dim], dtype
 *   block_table    int32 [batch][block_table_stride]; context_lens int32 [batch]
 *   scale          multiplies q.k (callers usually pass 1/sqrt(head_dim))
 *   out[b][i] = sum_j softmax_j(scale * q[b][i] . K_j) V_j over the context_lens[b] tokens of
 *   sequence b, reading KV head i / (n_q_heads / n_kv_heads).  An empty context gives zeros.
 *   workspace      optional fp32 scratch for split-K (long contexts are cut into partitions whose
 *                  partial softmax states are merged exactly by log-sum-exp).  Pass at least
 *                  paged_attention_decode_workspace_size(...) bytes, 16-byte aligned.  With
 *                  workspace == NULL every (sequence, KV head) runs as one partition (correct, but
 *                  slower for long or uneven contexts).  The contents need no initialisation.
 */
PA_API int paged_attention_decode(void* out, const void* q, const void* k_pool, const void* v_pool,
                           const int32_t* block_table, int64_t block_table_stride,
                           const int32_t* context_lens, int batch, int64_t num_blocks, int block_size,
                           float scale, int n_q_heads, int n_kv_heads, int head_dim, pa_dtype dtype,
                           void* workspace, size_t workspace_bytes, void* stream);
/* paged_attention_decode with per-call options (opts may be NULL).  The workspace must be at least
 * paged_attention_decode_workspace_size_ex(..., opts) bytes for the same opts. */
PA_API int paged_attention_decode_ex(void* out, const void* q, const void* k_pool, const void* v_pool,
                                     const int32_t* block_table, int64_t block_table_stride,
                                     const int32_t* context_lens, int batch, int64_t num_blocks, int block_size,
                                     float scale, int n_q_heads, int n_kv_heads, int head_dim, pa_dtype dtype,
                                     void* workspace, size_t workspace_bytes, const pa_opts* opts, void* stream);

/*
 * paged_attention_decode_fused — paged_kv_write of each sequence's new token followed by
 * paged_attention_decode, in one launch (nanoserve Day 19, "What I added today": the fused paged
 * read writes this step's K/V into the block pool and then attends over the whole history through
 * the block table, without rebuilding it).
 *   k_new, v_new   [batch][n_kv_heads][head_dim], dtype: the new token of sequence b is row b
 *   slot_mapping   int64 [batch]: slot of that token, which must be the slot of position
 *                  context_lens[b] - 1 (the decode convention) or negative (no write).  Any other
 *                  slot is neither written nor used: the device records PA_DEVERR_SLOT, checked
 *                  mode returns PA_ERANGE.
 *   k_pool, v_pool written in place (the new rows), then read.
 * Every other argument, the output and the workspace rules are those of paged_attention_decode; the
 * result (output and pools) is bit-identical to the two separate calls.
 */
PA_API int paged_attention_decode_fused(void* out, const void* q, const void* k_new, const void* v_new,
                                        const int64_t* slot_mapping, void* k_pool, void* v_pool,
                                        const int32_t* block_table, int64_t block_table_stride,
                                        const int32_t* context_lens, int batch, int64_t num_blocks, int block_size,
                                        float scale, int n_q_heads, int n_kv_heads, int head_dim, pa_dtype dtype,
                                        void* workspace, size_t workspace_bytes, void* stream);
/* paged_attention_decode_fused with per-call options (opts may be NULL). */
PA_API int paged_attention_decode_fused_ex(void* out, const void* q, const void* k_new, const void* v_new,
                                           const int64_t* slot_mapping, void* k_pool, void* v_pool,
                                           const int32_t* block_table, int64_t block_table_stride,
                                           const int32_t* context_lens, int batch, int64_t num_blocks,
                                           int block_size, float scale, int n_q_heads, int n_kv_heads, int head_dim,
                                           pa_dtype dtype, void* workspace, size_t workspace_bytes,
                                           const pa_opts* opts, void* stream);

/*
 * Workspace bytes paged_attention_decode needs for split-K with these sizes on the current device
 * (0 if it never splits).  The split-K plan: a row (sequence, KV head) as long as its table allows
 * is cut into partitions of P tokens, P chosen so that the grid holds at most one wave of decode
 * CTAs on this device (W = its SM count x 3 resident CTAs, x 2 for groups of 16 query heads): with
 * R = batch x n_kv_heads rows, P = ceil(capacity / max(1, floor(W / R))), clamped to [256, 1024]
 * tokens and rounded up to block_size; rows no longer than P are not split.  The
 * `_ex` form applies opts->partition_tokens instead when it is non-zero.  Invalid sizes give 0.
 */
PA_API size_t paged_attention_decode_workspace_size(int batch, int64_t block_table_stride, int block_size,
                                             int n_q_heads, int n_kv_heads, int head_dim);
PA_API size_t paged_attention_decode_workspace_size_ex(int batch, int64_t block_table_stride, int block_size,
                                                       int n_q_heads, int n_kv_heads, int head_dim,
                                                       const pa_opts* opts);

/* The split-K plan above for a device with sm_count SMs, computed on the host without touching a
 * device: *part_tokens (partition length), *max_parts (partitions of a row as long as its table
 * allows; 1 = no split) and *workspace_bytes.  partition_tokens as in pa_opts (0 = automatic).
 * Returns PA_EINVAL for invalid sizes or a null output pointer. */
PA_API int pa_decode_split_plan(int batch, int64_t block_table_stride, int block_size, int n_q_heads, int n_kv_heads,
                                int head_dim, int partition_tokens, int sm_count, int* part_tokens, int* max_parts,
                                size_t* workspace_bytes);

/*
 * paged_attention_prefill — causal chunked prefill over a paged history.
 * Source: JuliaPagedAttn README, "Features" (batched prefill: all prompt positions in one kernel
 * call) and API "prefill!".
 *   q, out          [total_q][n_q_heads][head_dim], dtype
 *   query_start_loc int32 [batch + 1], non-decreasing, query_start_loc[0] = 0,
 *                   query_start_loc[batch] = total_q.  Sequence b owns the m_b = qsl[b+1] - qsl[b]
 *                   queries qsl[b] .. qsl[b+1]-1; an empty chunk (m_b = 0) is allowed.
 *   context_lens    int32 [batch], history + chunk (the chunk's K/V must already be written).
 *   The chunk occupies the last m_b positions of the context; its query r (0-based) attends to
 *   positions 0 .. context_lens[b] - m_b + r inclusive.
 */
PA_API int paged_attention_prefill(void* out, const void* q, const int32_t* query_start_loc, int64_t total_q,
                            const void* k_pool, const void* v_pool, const int32_t* block_table,
                            int64_t block_table_stride, const int32_t* context_lens, int batch,
                            int64_t num_blocks, int block_size, float scale, int n_q_heads,
                            int n_kv_heads, int head_dim, pa_dtype dtype, void* stream);
/* paged_attention_prefill with per-call options (opts may be NULL). */
PA_API int paged_attention_prefill_ex(void* out, const void* q, const int32_t* query_start_loc, int64_t total_q,
                                      const void* k_pool, const void* v_pool, const int32_t* block_table,
                                      int64_t block_table_stride, const int32_t* context_lens, int batch,
                                      int64_t num_blocks, int block_size, float scale, int n_q_heads,
                                      int n_kv_heads, int head_dim, pa_dtype dtype, const pa_opts* opts,
                                      void* stream);

/*
 * copy_blocks — make physical block dst a bit copy of block src, in both pools, for each pair.
 * Source: JuliaPagedAttn README, "Copy-on-Write" (allocate a new block, copy the data, update the
 * table, decrement the refcount; the table update and refcount stay with the caller) and API
 * "cow_fork!".
 *   block_pairs  int64 [n_pairs][2] = (src, dst).  A dst must not appear twice nor as a src of
 *                another pair (checked mode rejects both); block_bytes = block_size * n_kv_heads *
 *                head_dim * element size, a multiple of 16 (the bytes of one block of one pool).
 */
PA_API int copy_blocks(void* k_pool, void* v_pool, const int64_t* block_pairs, int64_t n_pairs,
                int64_t num_blocks, int64_t block_bytes, void* stream);
/* copy_blocks with per-call options (opts may be NULL; only kv_block_stride_bytes applies). */
PA_API int copy_blocks_ex(void* k_pool, void* v_pool, const int64_t* block_pairs, int64_t n_pairs,
                          int64_t num_blocks, int64_t block_bytes, const pa_opts* opts, void* stream);

/*
 * swap_blocks — move blocks between two pools in one launch: the device pool and a pinned host pool
 * (Pico-vLLM dev log #5 "Paged Attention", core data structures: swap_out copies GPU blocks to the
 * pinned CPU pool, swap_in copies them back; the table and free-list bookkeeping stay with the
 * caller), or two device pools.
 *   dst_k_pool, dst_v_pool  destination pools, dst_num_blocks blocks each
 *   src_k_pool, src_v_pool  source pools, src_num_blocks blocks each
 *   Each pool is device memory or pinned host memory (cudaHostAlloc / cudaHostRegister, reachable
 *   from the device); pageable host memory returns PA_EINVAL.
 *   block_pairs  int64 [n_pairs][2] = (src block, dst block), device memory or pinned host memory.
 *                A dst must not appear twice (checked mode rejects it); out-of-range ids are
 *                skipped on the device and recorded as PA_DEVERR_COPY_PAIR.
 *   block_bytes  bytes of one block of one pool (block_size * n_kv_heads * head_dim * element size),
 *                a multiple of 16.  The copy is bit-exact and ordered on `stream`.
 */
PA_API int swap_blocks(void* dst_k_pool, void* dst_v_pool, int64_t dst_num_blocks, const void* src_k_pool,
                       const void* src_v_pool, int64_t src_num_blocks, const int64_t* block_pairs, int64_t n_pairs,
                       int64_t block_bytes, void* stream);
/* swap_blocks with per-call options (opts may be NULL; only kv_block_stride_bytes applies, to both
 * sides: for unified K/V blocks on both sides pass each v pointer = its k pointer + block_bytes
 * and kv_block_stride_bytes = 2 * block_bytes). */
PA_API int swap_blocks_ex(void* dst_k_pool, void* dst_v_pool, int64_t dst_num_blocks, const void* src_k_pool,
                          const void* src_v_pool, int64_t src_num_blocks, const int64_t* block_pairs,
                          int64_t n_pairs, int64_t block_bytes, const pa_opts* opts, void* stream);

/*
 * paged_attention_lse_merge — merge split-K partials exactly (the partition-combining identity of
 * the online softmax in JuliaPagedAttn README "Online Softmax", applied to whole partitions).
 *   part_max   fp32 [rows][n_parts]   running maxima in the log2 domain (score * log2(e))
 *   part_sum   fp32 [rows][n_parts]   sums of 2^(s - max)
 *   part_acc   fp32 [rows][n_parts][head_dim]  unnormalised accumulators
 *   out        [rows][head_dim], dtype: sum_p acc_p 2^(m_p - M) / sum_p l_p 2^(m_p - M), M = max_p m_p;
 *              partitions with part_sum == 0 are skipped; a row with none left gives zeros.
 */
PA_API int paged_attention_lse_merge(void* out, const float* part_max, const float* part_sum,
                              const float* part_acc, int64_t rows, int n_parts, int head_dim,
                              pa_dtype dtype, void* stream);

/*
 * paged_attention_decode_static_scratch — paged_attention_decode for callers that cannot allocate
 * device memory.  (The pages have no counterpart: this is a property of the library, not of the
 * method.)
 *
 * Who needs it: code that receives only the buffers it was handed and has no way to obtain more
 * device memory — a plugin or custom-op interface whose host owns the allocator and offers no
 * scratch, a serving loop that fixes its whole memory plan at start-up and forbids cudaMalloc on
 * the hot path (cudaMalloc may synchronize the device), or a foreign-language caller that only
 * holds raw device pointers.  Such callers cannot provide the split-K workspace.
 *
 * Arguments and results are exactly those of paged_attention_decode without the workspace pair
 * (contiguous pools, default options); the output is bit-identical to paged_attention_decode with
 * a caller workspace.  The split-K scratch lives instead in a file-scope device array of
 * PA_STATIC_SCRATCH_BYTES that every GPU loading this library holds until the process exits.  No
 * call allocates or frees anything.
 *   - The first call on a device (in each CUDA context: again after a device reset) looks up the
 *     array's device address with that device current, a one-time host set-up; make that first
 *     call before any stream capture.
 *   - Arguments are validated first, exactly as by paged_attention_decode; then problems whose
 *     split-K scratch (paged_attention_decode_workspace_size) exceeds PA_STATIC_SCRATCH_BYTES are
 *     rejected with PA_EWORKSPACE before anything is launched.
 *   - All calls on a device share the one array and it keeps the last call's contents; nothing in
 *     it needs to start at zero.  Calls whose kernels overlap on the GPU (other streams, other
 *     threads) race on the array: serialize them on one stream.
 */
#define PA_STATIC_SCRATCH_BYTES (32u * 1024u * 1024u)
PA_API int paged_attention_decode_static_scratch(void* out, const void* q, const void* k_pool, const void* v_pool,
                                                 const int32_t* block_table, int64_t block_table_stride,
                                                 const int32_t* context_lens, int batch, int64_t num_blocks,
                                                 int block_size, float scale, int n_q_heads, int n_kv_heads,
                                                 int head_dim, pa_dtype dtype, void* stream);

/* Checked mode on (1) or off (0, the default): the library's one process-wide setting.
 * pa_set_checked_mode(on) is pa_set_option(PA_OPT_CHECKED, on); any other option or value returns
 * PA_EINVAL, and pa_get_option of an unknown option returns PA_EINVAL. */
PA_API int pa_set_checked_mode(int on);
PA_API int pa_set_option(int option, int64_t value);
PA_API int64_t pa_get_option(int option);

/* The cudaError_t of the last PA_ECUDA on this thread (0 if none). */
PA_API int pa_last_cuda_error(void);

/* Short static description of a status code. */
PA_API const char* pa_status_string(int status);

/* Read (and, if clear != 0, reset) the device error word of the current device.  Synchronizes
 * `stream`.  Returns the PA_DEVERR_* bits, or a negative status on a CUDA failure.  The word
 * accumulates over launches until cleared; clearing is only for reporting: a timeout recorded by one
 * launch never shortens the waits of a later one (see pa_selftest_bounded_wait). */
PA_API int pa_device_error_flags(int clear, void* stream);

/*
 * pa_selftest_bounded_wait — run the failure path of the library's bounded waits on the device.
 * The pages have no counterpart: this is a test hook for the library itself.  Every pipelined kernel
 * (TMA rings, tensor-memory hand-offs) waits on mbarriers with a time limit and, when one runs out,
 * records PA_DEVERR_TIMEOUT and returns instead of hanging; the other waiting warps and CTAs of
 * the same launch see that and leave too.  The abort is scoped to the launch: each launch carries
 * its own epoch number and a wait leaves early only when the launch that gave up was its own, so a
 * later, healthy launch runs to completion even while PA_DEVERR_TIMEOUT is still set.  (A launch
 * captured in a CUDA graph keeps its epoch on every replay: after a replay gave up, clear the word
 * with pa_device_error_flags(1, ...) before replaying the graph again.)  This call launches one CTA
 * that does exactly that on barriers nothing completes: warp 0 gives up after limit_ns and records
 * the timeout, warp 1 (limit 1 s) must leave as soon as it sees it.  Nothing faults and the context
 * stays usable.
 *   limit_ns     warp 0's limit, 1000 .. 1000000000 (else PA_EINVAL)
 *   elapsed_ns   optional device uint64_t[2]: how long warp 0's and warp 1's waits took
 * Read the outcome with pa_device_error_flags(clear, stream).
 */
PA_API int pa_selftest_bounded_wait(int64_t limit_ns, void* elapsed_ns, void* stream);

/* Number of kernels this library has launched in this process (all devices). */
PA_API uint64_t pa_launch_count(void);

/* Library version string. */
PA_API const char* pa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDATTN_H_ */
