// paged_attention_decode_static_scratch: paged decode for callers that cannot allocate device
// memory.  The split-K scratch that paged_attention_decode takes from the caller lives here in a
// file-scope device array instead; this entry point only looks up its address and hands it to
// the regular decode path, which validates every argument and rejects problems whose scratch
// would not fit the array.
#include <mutex>

#include "pa_internal.h"

// The scratch itself: one per device that loads the library, held until the process exits.
static __device__ __align__(256) unsigned char g_pa_static_scratch[PA_STATIC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};
void* g_scratch_ctx[kMaxDevices] = {};  // the CUDA context g_scratch_ptr[dev] was looked up in

// Device address of the scratch on the current device.  In host code the array's name is only a
// stand-in; the address comes from the runtime, once per device and CUDA context, with that device
// current (a new context after a device reset reloads the module and moves the array).
int scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return pa::fail_cuda(e);
  if (dev < 0 || dev >= kMaxDevices) return PA_EINVAL;
  void* ctx = nullptr;
  const int rc = pa::current_context(&ctx);
  if (rc != PA_OK) return rc;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_ptr[dev] == nullptr || g_scratch_ctx[dev] != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_pa_static_scratch);
    if (e != cudaSuccess) return pa::fail_cuda(e);
    if (p == nullptr) return pa::fail_cuda(cudaErrorInvalidSymbol);
    g_scratch_ptr[dev] = p;
    g_scratch_ctx[dev] = ctx;
  }
  *out = g_scratch_ptr[dev];
  return PA_OK;
}

}  // namespace

extern "C" int paged_attention_decode_static_scratch(void* out, const void* q, const void* k_pool,
                                                     const void* v_pool, const int32_t* block_table,
                                                     int64_t block_table_stride, const int32_t* context_lens,
                                                     int batch, int64_t num_blocks, int block_size, float scale,
                                                     int n_q_heads, int n_kv_heads, int head_dim, pa_dtype dtype,
                                                     void* stream) {
  void* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != PA_OK) return rc;
  // paged_attention_decode checks the arguments first, then returns PA_EWORKSPACE without launching
  // when the split-K plan needs more than the array holds
  return paged_attention_decode(out, q, k_pool, v_pool, block_table, block_table_stride, context_lens, batch,
                                num_blocks, block_size, scale, n_q_heads, n_kv_heads, head_dim, dtype, scratch,
                                (size_t)PA_STATIC_SCRATCH_BYTES, stream);
}
