// pa_attention_varlen_static: attention for callers that cannot allocate
// device memory. The workspace is a scratch array compiled into this library;
// the call forwards to pa_attention_varlen with that array's device address.
#include <mutex>

#include "pa_common.cuh"
#include "pa_launch.h"

// The scratch array. Every GPU that loads the library holds one copy of
// PA_STATIC_WORKSPACE_BYTES until the process exits. In host code this name
// is only a handle: its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_pa_static_scratch[PA_STATIC_WORKSPACE_BYTES];

namespace {

constexpr int kMaxStaticDevices = 64;

std::mutex g_static_lock;
void *g_static_ptr[kMaxStaticDevices] = {};

// Device address of the scratch array on the current device, looked up with
// that device current. A successful lookup is cached; a failed one (for
// instance a first call made during stream capture) is not, so a later call
// tries again. NULL on failure, with the CUDA error recorded for
// pa_last_cuda_error().
void *static_scratch() {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) {
    pa::set_last_cuda_error(err);
    return nullptr;
  }
  if (dev < 0 || dev >= kMaxStaticDevices) return nullptr;
  std::lock_guard<std::mutex> guard(g_static_lock);
  if (!g_static_ptr[dev]) {
    void *ptr = nullptr;
    err = cudaGetSymbolAddress(&ptr, g_pa_static_scratch);
    if (err != cudaSuccess) {
      pa::set_last_cuda_error(err);
      return nullptr;
    }
    g_static_ptr[dev] = ptr;
  }
  return g_static_ptr[dev];
}

}  // namespace

extern "C" pa_status pa_attention_varlen_static(const void *q, int64_t q_token_stride, const void *key_cache,
                                                const void *value_cache, const int32_t *block_tables,
                                                int32_t max_blocks_per_seq, const int32_t *seq_lens,
                                                const int32_t *query_start_loc, int32_t num_seqs,
                                                int32_t total_q_tokens, int32_t max_query_len, int32_t max_seq_len,
                                                int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                                                int32_t block_size, int64_t num_blocks, float scale, void *out,
                                                int32_t dtype, void *stream) {
  // The workspace this call's plan needs: the 16-bit-cache layout, which is
  // what pa_attention_varlen checks (0 when the sizes are invalid; the
  // regular entry point then reports which, before launching anything).
  size_t need = 0;
  if (pa_attention_workspace_size(num_seqs, total_q_tokens, max_query_len, max_seq_len, num_heads, num_kv_heads,
                                  head_dim, block_size) > 0) {
    pa::WorkspaceLayout w16;
    if (pa::workspace_layout(num_seqs, total_q_tokens, max_seq_len, num_heads, num_kv_heads, head_dim, false, w16))
      need = w16.total;
  }
  if (need > PA_STATIC_WORKSPACE_BYTES) return PA_ERR_WORKSPACE;
  void *scratch = nullptr;
  if (num_seqs > 0 && total_q_tokens > 0 && need > 0) {
    scratch = static_scratch();
    if (!scratch) return PA_ERR_CUDA;
  }
  return pa_attention_varlen(q, q_token_stride, key_cache, value_cache, block_tables, max_blocks_per_seq, seq_lens,
                             query_start_loc, num_seqs, total_q_tokens, max_query_len, max_seq_len, num_heads,
                             num_kv_heads, head_dim, block_size, num_blocks, scale, out, scratch,
                             scratch ? PA_STATIC_WORKSPACE_BYTES : 0, dtype, stream);
}
