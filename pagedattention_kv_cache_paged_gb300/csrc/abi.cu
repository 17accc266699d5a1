// The C ABI (include/pagedattn.h): argument validation, the optional checked mode, split-K
// planning and dispatch to the kernels.  Holds no arithmetic of the method itself.
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdio>
#include <mutex>
#include <unordered_set>
#include <vector>

#include "pa_internal.h"

// Device error word pair, one per device context.  [0] accumulates the PA_DEVERR_* bits; [1] holds
// the epoch of the last launch whose bounded wait gave up, so that the other waits of that launch
// (and only of that launch) leave early.  Kernels receive the pair's address as an argument.
__device__ unsigned g_pa_device_error[2] = {0u, 0u};

namespace pa {

namespace {
thread_local int t_last_cuda_error = 0;
}  // namespace

int fail_cuda(cudaError_t e) {
  t_last_cuda_error = (int)e;
  return PA_ECUDA;
}

int current_context(void** ctx) {
  static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
  });
  if (fn == nullptr) return PA_ECUDA;
  CUcontext c = nullptr;
  if (fn(&c) != CUDA_SUCCESS) return PA_ECUDA;
  *ctx = static_cast<void*>(c);
  return PA_OK;
}

namespace {

constexpr int kMaxDevices = 64;
std::atomic<int> g_checked{0};
std::atomic<uint64_t> g_launches{0};
std::atomic<unsigned> g_epoch{0};
std::mutex g_dev_mutex;
// per device: the CUDA context the cached values below belong to, the error word's address there
// and the SM count (looked up again when the device's current context changes, e.g. after a reset)
void* g_ctx[kMaxDevices] = {};
unsigned* g_err_ptr[kMaxDevices] = {};
int g_sm_count[kMaxDevices] = {};

// Epoch of a new launch: never 0, the error word's initial (and cleared) value.
unsigned next_epoch() {
  unsigned e;
  do {
    e = g_epoch.fetch_add(1u, std::memory_order_relaxed) + 1u;
  } while (e == 0u);
  return e;
}

// Address of this device's error word pair and its SM count, looked up once per device context.
int device_info(unsigned** err, int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e);
  if (dev < 0 || dev >= kMaxDevices) return PA_EINVAL;
  void* ctx = nullptr;
  int rc = current_context(&ctx);
  if (rc) return rc;
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  if (g_err_ptr[dev] == nullptr || g_ctx[dev] != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_pa_device_error);
    if (e != cudaSuccess) return fail_cuda(e);
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return fail_cuda(e);
    g_err_ptr[dev] = static_cast<unsigned*>(p);
    g_sm_count[dev] = n;
    g_ctx[dev] = ctx;
  }
  if (err) *err = g_err_ptr[dev];
  if (sms) *sms = g_sm_count[dev];
  return PA_OK;
}

int finish(cudaError_t e, int launches) {
  g_launches.fetch_add((uint64_t)launches, std::memory_order_relaxed);
  if (e != cudaSuccess) return fail_cuda(e);
  return PA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool is_pow2(int64_t x) { return x > 0 && (x & (x - 1)) == 0; }
int log2i(int64_t x) {
  int r = 0;
  while ((int64_t(1) << r) < x) ++r;
  return r;
}
bool checked() { return g_checked.load() != 0; }

// Per-call options, validated; a null pointer means all defaults.
int read_opts(const pa_opts* o, pa_opts* out) {
  pa_opts d{};
  if (o != nullptr) d = *o;
  if (d.kv_block_stride_bytes < 0 || d.reserved != 0) return PA_EINVAL;
  if (d.decode_kernel < 0 || d.decode_kernel > 2 || d.prefill_kernel < 0 || d.prefill_kernel > 2) return PA_EINVAL;
  if (d.partition_tokens < 0 || d.partition_tokens > (1 << 30)) return PA_EINVAL;
  *out = d;
  return PA_OK;
}

// Distance in bytes from one block of a pool to the next: the call's kv_block_stride_bytes, or one
// block when it is 0.  An explicit stride is a multiple of 16 and at least one block.
int pool_block_stride(const pa_opts& o, int64_t block_bytes, int64_t* stride_bytes) {
  if (o.kv_block_stride_bytes == 0) {
    *stride_bytes = block_bytes;
    return PA_OK;
  }
  if (o.kv_block_stride_bytes < block_bytes || o.kv_block_stride_bytes % 16 != 0) return PA_EINVAL;
  *stride_bytes = o.kv_block_stride_bytes;
  return PA_OK;
}

int check_dtype(pa_dtype dt) { return (dt == PA_BF16 || dt == PA_FP16 || dt == PA_FP32) ? PA_OK : PA_EDTYPE; }

int check_heads(int n_q_heads, int n_kv_heads, int head_dim) {
  if (n_q_heads <= 0 || n_kv_heads <= 0 || head_dim <= 0) return PA_EINVAL;
  if (n_q_heads % n_kv_heads != 0) return PA_EINVAL;
  const int g = n_q_heads / n_kv_heads;
  if (g != 1 && g != 2 && g != 4 && g != 8 && g != 16) return PA_EUNSUPPORTED;
  if (head_dim != 64 && head_dim != 128) return PA_EUNSUPPORTED;
  return PA_OK;
}

template <typename T>
int copy_to_host(std::vector<T>& dst, const T* src, int64_t n, cudaStream_t s) {
  dst.resize((size_t)n);
  if (n == 0) return PA_OK;
  cudaError_t e = cudaMemcpyAsync(dst.data(), src, sizeof(T) * (size_t)n, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return e == cudaSuccess ? PA_OK : fail_cuda(e);
}

// Checked mode: every table entry a context reaches must name a pool block.
int validate_tables(const int32_t* block_table, int64_t bt_stride, const int32_t* context_lens, int batch,
                    int64_t num_blocks, int block_size, cudaStream_t s, std::vector<int32_t>* lens_out) {
  std::vector<int32_t> lens, table;
  int rc = copy_to_host(lens, context_lens, batch, s);
  if (rc) return rc;
  rc = copy_to_host(table, block_table, (int64_t)batch * bt_stride, s);
  if (rc) return rc;
  for (int b = 0; b < batch; ++b) {
    const int64_t n = lens[b];
    if (n < 0 || n > bt_stride * block_size) return PA_ERANGE;
    const int64_t nb = (n + block_size - 1) / block_size;
    for (int64_t j = 0; j < nb; ++j) {
      const int64_t id = table[(size_t)(b * bt_stride + j)];
      if (id < 0 || id >= num_blocks) return PA_ERANGE;
    }
  }
  if (lens_out) *lens_out = std::move(lens);
  return PA_OK;
}

// Split-K plan: partition length in tokens and partitions per row.  The automatic length gives the
// grid at most one wave of the tensor-core decode (3 resident CTAs per SM, 2 for groups of 16 query
// heads, times the device's SM count) when every row is as long as the table allows: each row gets
// floor(wave / rows) partitions (at least one), so that rounding never spills a few CTAs into a
// second wave that would take as long as the first.  The length stays between 256
// tokens (four 16-token tiles per warp: below that the merge launch costs more than the shorter
// partitions save) and 1024 (measured best at the serving shape, where rows are long and many:
// shorter partitions there lose to per-CTA start-up and merge traffic).  Small batches of long rows
// get short partitions and so enough CTAs to keep loads in flight; a batch that fills the GPU
// anyway is not split further.
int64_t split_target_ctas(int sms, int group) { return (int64_t)(sms > 0 ? sms : 1) * (group > 8 ? 2 : 3); }

// Longest context a table row can describe; context lengths are int32, so longer rows are capped.
int64_t table_capacity(int64_t bt_stride, int block_size) {
  const int64_t cap = bt_stride * block_size;
  return cap < (int64_t)INT32_MAX ? cap : (int64_t)INT32_MAX;
}

void plan_split(int batch, int n_kv_heads, int group, int sms, int64_t bt_stride, int block_size,
                int64_t partition_tokens, int* part_tokens, int* max_parts) {
  const int64_t max_len = table_capacity(bt_stride, block_size);
  int64_t p = partition_tokens;
  if (p <= 0) {
    const int64_t target = split_target_ctas(sms, group);
    const int64_t rows = (int64_t)(batch > 0 ? batch : 1) * (n_kv_heads > 0 ? n_kv_heads : 1);
    const int64_t parts = target / rows > 1 ? target / rows : 1;
    p = (max_len + parts - 1) / parts;
    p = p < 256 ? 256 : (p > 1024 ? 1024 : p);
  }
  p = ((p + block_size - 1) / block_size) * block_size;
  if (p >= max_len) {
    *part_tokens = (int)(max_len > 0 ? max_len : block_size);
    *max_parts = 1;
    return;
  }
  *part_tokens = (int)p;
  *max_parts = (int)((max_len + p - 1) / p);
}

struct WsLayout {
  size_t bytes;
  size_t off_m, off_l;
};

// Split-K workspace when rows split into up to max_parts partitions: acc[rows_heads][max_parts]
// [head_dim], then m[rows_heads][max_parts] and l[rows_heads][max_parts], each section 16-byte
// aligned.
WsLayout workspace_layout(int64_t rows_heads, int max_parts, int head_dim) {
  WsLayout w{};
  if (max_parts <= 1) return w;
  const size_t n = (size_t)rows_heads * (size_t)max_parts;
  auto up16 = [](size_t x) { return (x + 15) & ~size_t(15); };
  w.off_m = n * (size_t)head_dim * sizeof(float);
  w.off_l = w.off_m + up16(n * sizeof(float));
  w.bytes = w.off_l + up16(n * sizeof(float));
  return w;
}

}  // namespace
}  // namespace pa

using namespace pa;

namespace {

int kv_write_impl(const void* k_new, const void* v_new, const int64_t* slot_mapping, int64_t n_tokens, void* k_pool,
                  void* v_pool, int64_t num_blocks, int block_size, int n_kv_heads, int head_dim, pa_dtype dtype,
                  const pa_opts* opts, void* stream) {
  int rc = check_dtype(dtype);
  if (rc) return rc;
  pa_opts o;
  if ((rc = read_opts(opts, &o))) return rc;
  if (n_tokens < 0 || num_blocks <= 0 || block_size <= 0 || n_kv_heads <= 0 || head_dim <= 0) return PA_EINVAL;
  if (n_tokens == 0) return PA_OK;
  if (!k_new || !v_new || !slot_mapping || !k_pool || !v_pool) return PA_EINVAL;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pool) || !aligned16(v_pool)) return PA_EINVAL;
  const int64_t row_bytes = (int64_t)n_kv_heads * head_dim * dtype_bytes(dtype);
  if (row_bytes % 16 != 0) return PA_EUNSUPPORTED;
  int64_t stride_bytes = 0;
  if ((rc = pool_block_stride(o, row_bytes * block_size, &stride_bytes))) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned* err = nullptr;
  if ((rc = device_info(&err, nullptr))) return rc;
  const int64_t total_slots = num_blocks * block_size;
  if (checked()) {
    std::vector<int64_t> slots;
    if ((rc = copy_to_host(slots, slot_mapping, n_tokens, s))) return rc;
    std::unordered_set<int64_t> seen;
    for (int64_t v : slots) {
      if (v < 0) continue;
      if (v >= total_slots || !seen.insert(v).second) return PA_ERANGE;
    }
  }
  KvWriteArgs a{k_new,        v_new,     slot_mapping,      n_tokens, k_pool, v_pool, total_slots,
                (int)(row_bytes / 16), block_size, stride_bytes / 16, err};
  int launches = 0;
  cudaError_t e = launch_kv_write(a, dtype, s, &launches);
  return finish(e, launches);
}

size_t workspace_size_impl(int batch, int64_t block_table_stride, int block_size, int n_q_heads, int n_kv_heads,
                           int head_dim, const pa_opts* opts) {
  if (batch <= 0 || block_table_stride <= 0 || block_size <= 0 || n_q_heads <= 0 || n_kv_heads <= 0 ||
      head_dim <= 0 || n_q_heads % n_kv_heads != 0)
    return 0;
  pa_opts o;
  if (read_opts(opts, &o)) return 0;
  int sms = 0;
  if (device_info(nullptr, &sms)) return 0;
  int part = 0, max_parts = 1;
  plan_split(batch, n_kv_heads, n_q_heads / n_kv_heads, sms, block_table_stride, block_size, o.partition_tokens,
             &part, &max_parts);
  return workspace_layout((int64_t)batch * n_q_heads, max_parts, head_dim).bytes;
}

int decode_impl(void* out, const void* q, const void* k_pool, const void* v_pool, const int32_t* block_table,
                int64_t block_table_stride, const int32_t* context_lens, int batch, int64_t num_blocks, int block_size,
                float scale, int n_q_heads, int n_kv_heads, int head_dim, pa_dtype dtype, void* workspace,
                size_t workspace_bytes, const pa_opts* opts, void* stream, const void* k_new, const void* v_new,
                const int64_t* slot_mapping) {
  int rc = check_dtype(dtype);
  if (rc) return rc;
  pa_opts o;
  if ((rc = read_opts(opts, &o))) return rc;
  rc = check_heads(n_q_heads, n_kv_heads, head_dim);
  if (rc) return rc;
  if (batch < 0 || num_blocks <= 0 || block_table_stride <= 0 || !is_pow2(block_size) || block_size > 256)
    return block_size > 256 || (block_size > 0 && !is_pow2(block_size)) ? PA_EUNSUPPORTED : PA_EINVAL;
  if (batch == 0) return PA_OK;
  if (!out || !q || !k_pool || !v_pool || !block_table || !context_lens) return PA_EINVAL;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool)) return PA_EINVAL;
  const bool fused = k_new != nullptr || v_new != nullptr || slot_mapping != nullptr;
  if (fused && (!k_new || !v_new || !slot_mapping || !aligned16(k_new) || !aligned16(v_new))) return PA_EINVAL;
  const int64_t block_elems = (int64_t)block_size * n_kv_heads * head_dim;
  int64_t stride_bytes = 0;
  if ((rc = pool_block_stride(o, block_elems * dtype_bytes(dtype), &stride_bytes))) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned* err = nullptr;
  int sms = 0;
  if ((rc = device_info(&err, &sms))) return rc;
  const int group = n_q_heads / n_kv_heads;
  const bool tc_ok = decode_tc_supported(dtype, block_size, head_dim, group, num_blocks);
  if (o.decode_kernel == 2 && !tc_ok) return PA_EUNSUPPORTED;
  const bool use_tc = o.decode_kernel == 2 || (o.decode_kernel == 0 && tc_ok);

  int part_tokens = 0, max_parts = 1;
  plan_split(batch, n_kv_heads, group, sms, block_table_stride, block_size, o.partition_tokens, &part_tokens,
             &max_parts);
  const WsLayout ws = workspace_layout((int64_t)batch * n_q_heads, max_parts, head_dim);
  if (max_parts > 1) {
    if (workspace == nullptr) {
      max_parts = 1;
      part_tokens = (int)table_capacity(block_table_stride, block_size);
    } else if (workspace_bytes < ws.bytes || !aligned16(workspace)) {
      return PA_EWORKSPACE;
    }
  }
  if (checked()) {
    std::vector<int32_t> lens;
    rc = validate_tables(block_table, block_table_stride, context_lens, batch, num_blocks, block_size, s, &lens);
    if (rc) return rc;
    if (fused) {
      std::vector<int64_t> slots;
      std::vector<int32_t> table;
      if ((rc = copy_to_host(slots, slot_mapping, batch, s))) return rc;
      if ((rc = copy_to_host(table, block_table, (int64_t)batch * block_table_stride, s))) return rc;
      for (int b = 0; b < batch; ++b) {
        if (slots[(size_t)b] < 0) continue;
        const int64_t last = (int64_t)lens[(size_t)b] - 1;
        if (last < 0) return PA_ERANGE;
        const int64_t expect = (int64_t)table[(size_t)(b * block_table_stride + last / block_size)] * block_size +
                               last % block_size;
        if (slots[(size_t)b] != expect) return PA_ERANGE;
      }
    }
  }
  AttnArgs a{};
  a.out = out;
  a.q = q;
  a.k_pool = k_pool;
  a.v_pool = v_pool;
  a.block_table = block_table;
  a.bt_stride = block_table_stride;
  a.context_lens = context_lens;
  a.query_start_loc = nullptr;
  a.batch = batch;
  a.rows = batch;
  a.num_blocks = num_blocks;
  a.block_size = block_size;
  a.block_shift = log2i(block_size);
  a.kv_block_stride = stride_bytes / dtype_bytes(dtype);
  a.scale_log2 = scale * 1.4426950408889634f;
  a.n_q_heads = n_q_heads;
  a.n_kv_heads = n_kv_heads;
  a.group = group;
  a.head_dim = head_dim;
  a.part_tokens = part_tokens;
  a.max_parts = max_parts;
  if (max_parts > 1) {
    char* base = static_cast<char*>(workspace);
    a.ws_acc = reinterpret_cast<float*>(base);
    a.ws_m = reinterpret_cast<float*>(base + ws.off_m);
    a.ws_l = reinterpret_cast<float*>(base + ws.off_l);
  }
  a.err = err;
  a.epoch = next_epoch();
  if (fused) {
    a.k_new = k_new;
    a.v_new = v_new;
    a.slot_mapping = slot_mapping;
    a.k_pool_w = const_cast<void*>(k_pool);
    a.v_pool_w = const_cast<void*>(v_pool);
  }
  int launches = 0;
  cudaError_t e = use_tc ? launch_decode_tc(a, dtype, s, &launches) : launch_attn_simt(a, dtype, s, &launches);
  if (e == cudaSuccess && max_parts > 1) {
    MergeArgs m{};
    m.out = out;
    m.part_m = a.ws_m;
    m.part_l = a.ws_l;
    m.part_acc = a.ws_acc;
    m.rows = (int64_t)batch * n_q_heads;
    m.n_parts = max_parts;
    m.head_dim = head_dim;
    m.context_lens = context_lens;
    m.heads_per_seq = n_q_heads;
    m.part_tokens = part_tokens;
    m.max_len = block_table_stride * block_size;
    e = launch_lse_merge(m, dtype, s, &launches);
  }
  return finish(e, launches);
}

int prefill_impl(void* out, const void* q, const int32_t* query_start_loc, int64_t total_q, const void* k_pool,
                 const void* v_pool, const int32_t* block_table, int64_t block_table_stride,
                 const int32_t* context_lens, int batch, int64_t num_blocks, int block_size, float scale,
                 int n_q_heads, int n_kv_heads, int head_dim, pa_dtype dtype, const pa_opts* opts, void* stream) {
  int rc = check_dtype(dtype);
  if (rc) return rc;
  pa_opts o;
  if ((rc = read_opts(opts, &o))) return rc;
  rc = check_heads(n_q_heads, n_kv_heads, head_dim);
  if (rc) return rc;
  if (batch < 0 || total_q < 0 || num_blocks <= 0 || block_table_stride <= 0) return PA_EINVAL;
  if (!is_pow2(block_size) || block_size > 256) return block_size <= 0 ? PA_EINVAL : PA_EUNSUPPORTED;
  if (batch == 0 || total_q == 0) return PA_OK;
  if (total_q > INT32_MAX) return PA_EINVAL;  // query rows are int32 (query_start_loc is int32)
  if (!out || !q || !query_start_loc || !k_pool || !v_pool || !block_table || !context_lens) return PA_EINVAL;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool)) return PA_EINVAL;
  int64_t stride_bytes = 0;
  if ((rc = pool_block_stride(o, (int64_t)block_size * n_kv_heads * head_dim * dtype_bytes(dtype), &stride_bytes)))
    return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned* err = nullptr;
  if ((rc = device_info(&err, nullptr))) return rc;
  const int group = n_q_heads / n_kv_heads;
  // the tcgen05 kernel has the tensor-core decode's support set
  const bool tc_ok = decode_tc_supported(dtype, block_size, head_dim, group, num_blocks);
  if (o.prefill_kernel == 2 && !tc_ok) return PA_EUNSUPPORTED;
  const bool use_tc = o.prefill_kernel == 2 || (o.prefill_kernel == 0 && tc_ok);
  if (checked()) {
    std::vector<int32_t> lens, qsl;
    rc = validate_tables(block_table, block_table_stride, context_lens, batch, num_blocks, block_size, s, &lens);
    if (rc) return rc;
    if ((rc = copy_to_host(qsl, query_start_loc, (int64_t)batch + 1, s))) return rc;
    if (qsl[0] != 0 || qsl[(size_t)batch] != total_q) return PA_ERANGE;
    for (int b = 0; b < batch; ++b) {
      const int64_t m = (int64_t)qsl[(size_t)b + 1] - qsl[(size_t)b];
      if (m < 0 || m > lens[(size_t)b]) return PA_ERANGE;
    }
  }
  AttnArgs a{};
  a.out = out;
  a.q = q;
  a.k_pool = k_pool;
  a.v_pool = v_pool;
  a.block_table = block_table;
  a.bt_stride = block_table_stride;
  a.context_lens = context_lens;
  a.query_start_loc = query_start_loc;
  a.batch = batch;
  a.rows = total_q;
  a.num_blocks = num_blocks;
  a.block_size = block_size;
  a.block_shift = log2i(block_size);
  a.kv_block_stride = stride_bytes / dtype_bytes(dtype);
  a.scale_log2 = scale * 1.4426950408889634f;
  a.n_q_heads = n_q_heads;
  a.n_kv_heads = n_kv_heads;
  a.group = group;
  a.head_dim = head_dim;
  a.part_tokens = (int)table_capacity(block_table_stride, block_size);
  a.max_parts = 1;
  a.err = err;
  a.epoch = next_epoch();
  int launches = 0;
  cudaError_t e = use_tc ? launch_prefill_umma(a, dtype, s, &launches) : launch_attn_simt(a, dtype, s, &launches);
  return finish(e, launches);
}

int copy_blocks_impl(void* k_pool, void* v_pool, const int64_t* block_pairs, int64_t n_pairs, int64_t num_blocks,
                     int64_t block_bytes, const pa_opts* opts, void* stream) {
  pa_opts o;
  int rc = read_opts(opts, &o);
  if (rc) return rc;
  if (n_pairs < 0 || num_blocks <= 0 || block_bytes <= 0 || block_bytes % 16 != 0) return PA_EINVAL;
  if (n_pairs == 0) return PA_OK;
  if (!k_pool || !v_pool || !block_pairs) return PA_EINVAL;
  if (!aligned16(k_pool) || !aligned16(v_pool)) return PA_EINVAL;
  int64_t stride_bytes = 0;
  if ((rc = pool_block_stride(o, block_bytes, &stride_bytes))) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned* err = nullptr;
  if ((rc = device_info(&err, nullptr))) return rc;
  if (checked()) {
    std::vector<int64_t> pairs;
    if ((rc = copy_to_host(pairs, block_pairs, 2 * n_pairs, s))) return rc;
    std::unordered_set<int64_t> dsts, srcs;
    for (int64_t i = 0; i < n_pairs; ++i) {
      const int64_t src = pairs[(size_t)(2 * i)], dst = pairs[(size_t)(2 * i + 1)];
      if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) return PA_ERANGE;
      if (!dsts.insert(dst).second) return PA_ERANGE;
      srcs.insert(src);
    }
    for (int64_t d : dsts)
      if (srcs.count(d)) return PA_ERANGE;
  }
  CopyBlocksArgs a{k_pool, v_pool, block_pairs, n_pairs, num_blocks, block_bytes / 16, stride_bytes / 16, err};
  int launches = 0;
  cudaError_t e = launch_copy_blocks(a, s, &launches);
  return finish(e, launches);
}

// Device-accessible address of a pool: device memory as is, pinned host memory through its mapping.
int device_address(const void* p, void** out) {
  cudaPointerAttributes at{};
  cudaError_t e = cudaPointerGetAttributes(&at, p);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return PA_EINVAL;
  }
  if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) {
    *out = const_cast<void*>(p);
    return PA_OK;
  }
  if (at.type == cudaMemoryTypeHost && at.devicePointer != nullptr) {
    *out = at.devicePointer;
    return PA_OK;
  }
  return PA_EINVAL;  // pageable host memory: not reachable from the device
}

int swap_blocks_impl(void* dst_k_pool, void* dst_v_pool, int64_t dst_num_blocks, const void* src_k_pool,
                     const void* src_v_pool, int64_t src_num_blocks, const int64_t* block_pairs, int64_t n_pairs,
                     int64_t block_bytes, const pa_opts* opts, void* stream) {
  pa_opts o;
  int rc = read_opts(opts, &o);
  if (rc) return rc;
  if (n_pairs < 0 || dst_num_blocks <= 0 || src_num_blocks <= 0 || block_bytes <= 0 || block_bytes % 16 != 0)
    return PA_EINVAL;
  if (n_pairs == 0) return PA_OK;
  if (!dst_k_pool || !dst_v_pool || !src_k_pool || !src_v_pool || !block_pairs) return PA_EINVAL;
  if (!aligned16(dst_k_pool) || !aligned16(dst_v_pool) || !aligned16(src_k_pool) || !aligned16(src_v_pool))
    return PA_EINVAL;
  int64_t stride_bytes = 0;
  if ((rc = pool_block_stride(o, block_bytes, &stride_bytes))) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned* err = nullptr;
  if ((rc = device_info(&err, nullptr))) return rc;
  SwapArgs a{};
  void* p = nullptr;
  if ((rc = device_address(dst_k_pool, &p))) return rc;
  a.dst_k = p;
  if ((rc = device_address(dst_v_pool, &p))) return rc;
  a.dst_v = p;
  if ((rc = device_address(src_k_pool, &p))) return rc;
  a.src_k = p;
  if ((rc = device_address(src_v_pool, &p))) return rc;
  a.src_v = p;
  if ((rc = device_address(block_pairs, &p))) return rc;
  a.pairs = static_cast<const int64_t*>(p);
  if (checked()) {
    std::vector<int64_t> pairs;
    if ((rc = copy_to_host(pairs, a.pairs, 2 * n_pairs, s))) return rc;
    std::unordered_set<int64_t> dsts;
    for (int64_t i = 0; i < n_pairs; ++i) {
      const int64_t src = pairs[(size_t)(2 * i)], dst = pairs[(size_t)(2 * i + 1)];
      if (src < 0 || src >= src_num_blocks || dst < 0 || dst >= dst_num_blocks) return PA_ERANGE;
      if (!dsts.insert(dst).second) return PA_ERANGE;
    }
  }
  a.n_pairs = n_pairs;
  a.src_num_blocks = src_num_blocks;
  a.dst_num_blocks = dst_num_blocks;
  a.block_vecs = block_bytes / 16;
  a.block_stride_vecs = stride_bytes / 16;
  a.err = err;
  int launches = 0;
  cudaError_t e = launch_swap_blocks(a, s, &launches);
  return finish(e, launches);
}

}  // namespace

extern "C" {

int pa_set_option(int option, int64_t value) {
  if (option != PA_OPT_CHECKED || (value != 0 && value != 1)) return PA_EINVAL;
  g_checked.store((int)value);
  return PA_OK;
}

int pa_set_checked_mode(int on) { return pa_set_option(PA_OPT_CHECKED, on); }

int64_t pa_get_option(int option) {
  if (option != PA_OPT_CHECKED) return PA_EINVAL;
  return g_checked.load();
}

int pa_last_cuda_error(void) { return t_last_cuda_error; }

const char* pa_status_string(int status) {
  switch (status) {
    case PA_OK: return "ok";
    case PA_EINVAL: return "invalid argument";
    case PA_EDTYPE: return "unsupported dtype";
    case PA_ERANGE: return "index, length or pair out of range (checked mode)";
    case PA_EWORKSPACE: return "workspace too small or misaligned";
    case PA_ECUDA: return "CUDA launch failed";
    case PA_EUNSUPPORTED: return "unsupported shape";
    default: return "unknown status";
  }
}

uint64_t pa_launch_count(void) { return g_launches.load(); }

const char* pa_version(void) { return "pagedattn 0.2 (sm_103a)"; }

int pa_device_error_flags(int clear, void* stream) {
  unsigned* err = nullptr;
  int rc = device_info(&err, nullptr);
  if (rc) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, err, sizeof(v), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess && clear) e = cudaMemsetAsync(err, 0, 2 * sizeof(unsigned), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail_cuda(e);
  return (int)v;
}

int pa_selftest_bounded_wait(int64_t limit_ns, void* elapsed_ns, void* stream) {
  if (limit_ns < 1000 || limit_ns > 1000000000) return PA_EINVAL;
  if (elapsed_ns != nullptr && (reinterpret_cast<uintptr_t>(elapsed_ns) & 7u) != 0) return PA_EINVAL;
  unsigned* err = nullptr;
  int rc = device_info(&err, nullptr);
  if (rc) return rc;
  int launches = 0;
  cudaError_t e = launch_selftest_wait(err, next_epoch(), (uint64_t)limit_ns,
                                       static_cast<unsigned long long*>(elapsed_ns),
                                       static_cast<cudaStream_t>(stream), &launches);
  return finish(e, launches);
}

int paged_kv_write(const void* k_new, const void* v_new, const int64_t* slot_mapping, int64_t n_tokens,
                   void* k_pool, void* v_pool, int64_t num_blocks, int block_size, int n_kv_heads,
                   int head_dim, pa_dtype dtype, void* stream) {
  return kv_write_impl(k_new, v_new, slot_mapping, n_tokens, k_pool, v_pool, num_blocks, block_size, n_kv_heads,
                       head_dim, dtype, nullptr, stream);
}

int paged_kv_write_ex(const void* k_new, const void* v_new, const int64_t* slot_mapping, int64_t n_tokens,
                      void* k_pool, void* v_pool, int64_t num_blocks, int block_size, int n_kv_heads, int head_dim,
                      pa_dtype dtype, const pa_opts* opts, void* stream) {
  return kv_write_impl(k_new, v_new, slot_mapping, n_tokens, k_pool, v_pool, num_blocks, block_size, n_kv_heads,
                       head_dim, dtype, opts, stream);
}

int pa_decode_split_plan(int batch, int64_t block_table_stride, int block_size, int n_q_heads, int n_kv_heads,
                         int head_dim, int partition_tokens, int sm_count, int* part_tokens, int* max_parts,
                         size_t* workspace_bytes) {
  if (batch <= 0 || block_table_stride <= 0 || block_size <= 0 || n_q_heads <= 0 || n_kv_heads <= 0 ||
      head_dim <= 0 || n_q_heads % n_kv_heads != 0 || partition_tokens < 0 || partition_tokens > (1 << 30) ||
      sm_count <= 0 || !part_tokens || !max_parts || !workspace_bytes)
    return PA_EINVAL;
  plan_split(batch, n_kv_heads, n_q_heads / n_kv_heads, sm_count, block_table_stride, block_size, partition_tokens,
             part_tokens, max_parts);
  *workspace_bytes = workspace_layout((int64_t)batch * n_q_heads, *max_parts, head_dim).bytes;
  return PA_OK;
}

size_t paged_attention_decode_workspace_size(int batch, int64_t block_table_stride, int block_size,
                                             int n_q_heads, int n_kv_heads, int head_dim) {
  return workspace_size_impl(batch, block_table_stride, block_size, n_q_heads, n_kv_heads, head_dim, nullptr);
}

size_t paged_attention_decode_workspace_size_ex(int batch, int64_t block_table_stride, int block_size,
                                                int n_q_heads, int n_kv_heads, int head_dim, const pa_opts* opts) {
  return workspace_size_impl(batch, block_table_stride, block_size, n_q_heads, n_kv_heads, head_dim, opts);
}

int paged_attention_decode(void* out, const void* q, const void* k_pool, const void* v_pool,
                           const int32_t* block_table, int64_t block_table_stride,
                           const int32_t* context_lens, int batch, int64_t num_blocks, int block_size,
                           float scale, int n_q_heads, int n_kv_heads, int head_dim, pa_dtype dtype,
                           void* workspace, size_t workspace_bytes, void* stream) {
  return decode_impl(out, q, k_pool, v_pool, block_table, block_table_stride, context_lens, batch, num_blocks,
                     block_size, scale, n_q_heads, n_kv_heads, head_dim, dtype, workspace, workspace_bytes, nullptr,
                     stream, nullptr, nullptr, nullptr);
}

int paged_attention_decode_ex(void* out, const void* q, const void* k_pool, const void* v_pool,
                              const int32_t* block_table, int64_t block_table_stride, const int32_t* context_lens,
                              int batch, int64_t num_blocks, int block_size, float scale, int n_q_heads,
                              int n_kv_heads, int head_dim, pa_dtype dtype, void* workspace, size_t workspace_bytes,
                              const pa_opts* opts, void* stream) {
  return decode_impl(out, q, k_pool, v_pool, block_table, block_table_stride, context_lens, batch, num_blocks,
                     block_size, scale, n_q_heads, n_kv_heads, head_dim, dtype, workspace, workspace_bytes, opts,
                     stream, nullptr, nullptr, nullptr);
}

int paged_attention_decode_fused(void* out, const void* q, const void* k_new, const void* v_new,
                                 const int64_t* slot_mapping, void* k_pool, void* v_pool,
                                 const int32_t* block_table, int64_t block_table_stride,
                                 const int32_t* context_lens, int batch, int64_t num_blocks, int block_size,
                                 float scale, int n_q_heads, int n_kv_heads, int head_dim, pa_dtype dtype,
                                 void* workspace, size_t workspace_bytes, void* stream) {
  if (batch > 0 && (!k_new || !v_new || !slot_mapping)) return PA_EINVAL;
  return decode_impl(out, q, k_pool, v_pool, block_table, block_table_stride, context_lens, batch, num_blocks,
                     block_size, scale, n_q_heads, n_kv_heads, head_dim, dtype, workspace, workspace_bytes, nullptr,
                     stream, k_new, v_new, slot_mapping);
}

int paged_attention_decode_fused_ex(void* out, const void* q, const void* k_new, const void* v_new,
                                    const int64_t* slot_mapping, void* k_pool, void* v_pool,
                                    const int32_t* block_table, int64_t block_table_stride,
                                    const int32_t* context_lens, int batch, int64_t num_blocks, int block_size,
                                    float scale, int n_q_heads, int n_kv_heads, int head_dim, pa_dtype dtype,
                                    void* workspace, size_t workspace_bytes, const pa_opts* opts, void* stream) {
  if (batch > 0 && (!k_new || !v_new || !slot_mapping)) return PA_EINVAL;
  return decode_impl(out, q, k_pool, v_pool, block_table, block_table_stride, context_lens, batch, num_blocks,
                     block_size, scale, n_q_heads, n_kv_heads, head_dim, dtype, workspace, workspace_bytes, opts,
                     stream, k_new, v_new, slot_mapping);
}

int paged_attention_prefill(void* out, const void* q, const int32_t* query_start_loc, int64_t total_q,
                            const void* k_pool, const void* v_pool, const int32_t* block_table,
                            int64_t block_table_stride, const int32_t* context_lens, int batch,
                            int64_t num_blocks, int block_size, float scale, int n_q_heads,
                            int n_kv_heads, int head_dim, pa_dtype dtype, void* stream) {
  return prefill_impl(out, q, query_start_loc, total_q, k_pool, v_pool, block_table, block_table_stride,
                      context_lens, batch, num_blocks, block_size, scale, n_q_heads, n_kv_heads, head_dim, dtype,
                      nullptr, stream);
}

int paged_attention_prefill_ex(void* out, const void* q, const int32_t* query_start_loc, int64_t total_q,
                               const void* k_pool, const void* v_pool, const int32_t* block_table,
                               int64_t block_table_stride, const int32_t* context_lens, int batch,
                               int64_t num_blocks, int block_size, float scale, int n_q_heads, int n_kv_heads,
                               int head_dim, pa_dtype dtype, const pa_opts* opts, void* stream) {
  return prefill_impl(out, q, query_start_loc, total_q, k_pool, v_pool, block_table, block_table_stride,
                      context_lens, batch, num_blocks, block_size, scale, n_q_heads, n_kv_heads, head_dim, dtype,
                      opts, stream);
}

int copy_blocks(void* k_pool, void* v_pool, const int64_t* block_pairs, int64_t n_pairs,
                int64_t num_blocks, int64_t block_bytes, void* stream) {
  return copy_blocks_impl(k_pool, v_pool, block_pairs, n_pairs, num_blocks, block_bytes, nullptr, stream);
}

int copy_blocks_ex(void* k_pool, void* v_pool, const int64_t* block_pairs, int64_t n_pairs, int64_t num_blocks,
                   int64_t block_bytes, const pa_opts* opts, void* stream) {
  return copy_blocks_impl(k_pool, v_pool, block_pairs, n_pairs, num_blocks, block_bytes, opts, stream);
}

int swap_blocks(void* dst_k_pool, void* dst_v_pool, int64_t dst_num_blocks, const void* src_k_pool,
                const void* src_v_pool, int64_t src_num_blocks, const int64_t* block_pairs, int64_t n_pairs,
                int64_t block_bytes, void* stream) {
  return swap_blocks_impl(dst_k_pool, dst_v_pool, dst_num_blocks, src_k_pool, src_v_pool, src_num_blocks, block_pairs,
                          n_pairs, block_bytes, nullptr, stream);
}

int swap_blocks_ex(void* dst_k_pool, void* dst_v_pool, int64_t dst_num_blocks, const void* src_k_pool,
                   const void* src_v_pool, int64_t src_num_blocks, const int64_t* block_pairs, int64_t n_pairs,
                   int64_t block_bytes, const pa_opts* opts, void* stream) {
  return swap_blocks_impl(dst_k_pool, dst_v_pool, dst_num_blocks, src_k_pool, src_v_pool, src_num_blocks, block_pairs,
                          n_pairs, block_bytes, opts, stream);
}

int paged_attention_lse_merge(void* out, const float* part_max, const float* part_sum,
                              const float* part_acc, int64_t rows, int n_parts, int head_dim,
                              pa_dtype dtype, void* stream) {
  int rc = check_dtype(dtype);
  if (rc) return rc;
  if (rows < 0 || n_parts <= 0) return PA_EINVAL;
  if (head_dim != 64 && head_dim != 128) return PA_EUNSUPPORTED;
  if (rows == 0) return PA_OK;
  if (!out || !part_max || !part_sum || !part_acc) return PA_EINVAL;
  MergeArgs m{};
  m.out = out;
  m.part_m = part_max;
  m.part_l = part_sum;
  m.part_acc = part_acc;
  m.rows = rows;
  m.n_parts = n_parts;
  m.head_dim = head_dim;
  m.context_lens = nullptr;
  int launches = 0;
  cudaError_t e = launch_lse_merge(m, dtype, static_cast<cudaStream_t>(stream), &launches);
  return finish(e, launches);
}

}  // extern "C"
