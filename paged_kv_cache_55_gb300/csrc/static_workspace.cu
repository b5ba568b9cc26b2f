// pa_attention_varlen_static: attention for callers that cannot allocate
// device memory. The workspace is a scratch array compiled into this library;
// the call forwards to pa_attention_varlen with that array's device address.
#include <mutex>

#include "pa_common.cuh"

// The scratch array. Every GPU that loads the library holds one copy of
// PA_STATIC_WORKSPACE_BYTES until the process exits. In host code this name
// is only a handle: its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_pa_static_scratch[PA_STATIC_WORKSPACE_BYTES];

namespace {

constexpr int kMaxStaticDevices = 64;

struct StaticScratch {
  std::once_flag once;
  void *ptr = nullptr;
  cudaError_t err = cudaSuccess;
};
StaticScratch g_static[kMaxStaticDevices];

// Device address of the scratch array on the current device, looked up once
// per device (with that device current) and cached. NULL on failure.
void *static_scratch() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxStaticDevices) return nullptr;
  StaticScratch &s = g_static[dev];
  std::call_once(s.once, [&]() {
    void *ptr = nullptr;
    s.err = cudaGetSymbolAddress(&ptr, g_pa_static_scratch);
    s.ptr = (s.err == cudaSuccess) ? ptr : nullptr;
  });
  return s.ptr;
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
  const size_t need = pa_attention_workspace_size(num_seqs, total_q_tokens, max_query_len, max_seq_len, num_heads,
                                                  num_kv_heads, head_dim, block_size);
  if (need > PA_STATIC_WORKSPACE_BYTES) return PA_ERR_WORKSPACE;
  void *scratch = nullptr;
  if (num_seqs > 0 && total_q_tokens > 0 && need > 0) {
    scratch = static_scratch();
    if (!scratch) return PA_ERR_CUDA;
  }
  // need == 0 means the sizes are invalid (or there is nothing to do): the
  // regular entry point reports which, before launching anything.
  return pa_attention_varlen(q, q_token_stride, key_cache, value_cache, block_tables, max_blocks_per_seq, seq_lens,
                             query_start_loc, num_seqs, total_q_tokens, max_query_len, max_seq_len, num_heads,
                             num_kv_heads, head_dim, block_size, num_blocks, scale, out, scratch,
                             scratch ? PA_STATIC_WORKSPACE_BYTES : 0, dtype, stream);
}
