// C ABI of libpagedattn.so (declared in include/pagedattn.h): argument
// validation, per-device state, and dispatch to the kernels' launchers.
#include <atomic>
#include <climits>
#include <cmath>
#include <mutex>

#include "pa_common.cuh"
#include "pa_launch.h"


// Device status word: kernels OR PA_FLAG_* bits into it when they skip work
// because an index is out of range.
__device__ unsigned int g_pa_status_word;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceState {
  std::once_flag once;
  unsigned int *status = nullptr;
  int sm_count = 0;
  cudaError_t err = cudaSuccess;
};
DeviceState g_devices[kMaxDevices];
std::atomic<uint64_t> g_launches{0};
thread_local cudaEvent_t t_ev_start = nullptr;
thread_local cudaEvent_t t_ev_stop = nullptr;
thread_local cudaEvent_t t_tile_start = nullptr;
thread_local cudaEvent_t t_tile_stop = nullptr;
thread_local cudaError_t t_last_cuda_error = cudaSuccess;

// Record the CUDA error behind a PA_ERR_LAUNCH / PA_ERR_CUDA return.
pa_status cuda_failure(pa_status status, cudaError_t err) {
  t_last_cuda_error = err;
  return status;
}

// Per-device set-up on first use: the status word's device address and the
// SM count (both fixed for the life of the process).
DeviceState *device_state() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  DeviceState &s = g_devices[dev];
  std::call_once(s.once, [&]() {
    void *ptr = nullptr;
    s.err = cudaGetSymbolAddress(&ptr, g_pa_status_word);
    if (s.err == cudaSuccess) s.err = cudaDeviceGetAttribute(&s.sm_count, cudaDevAttrMultiProcessorCount, dev);
    s.status = static_cast<unsigned int *>(ptr);
  });
  if (s.err != cudaSuccess) t_last_cuda_error = s.err;
  return s.err == cudaSuccess ? &s : nullptr;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool valid_cache_scale(float s) { return std::isfinite(s) && s > 0.0f; }

// Head dims with built kernels: 64 and 128, 80 and 96 (rows padded to whole
// 64-element swizzle atoms in shared memory), and 256.
bool supported_head_dim(int32_t d) { return d == 64 || d == 80 || d == 96 || d == 128 || d == 256; }

// Bytes of one cache element: 2 for the 16-bit types, 1 for E4M3 codes; 0 if unknown.
int cache_elem_bytes(int32_t dtype) {
  return (dtype == PA_BF16 || dtype == PA_FP16) ? 2 : (dtype == PA_FP8_E4M3 ? 1 : 0);
}

bool supported_dims(int32_t num_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size) {
  if (!supported_head_dim(head_dim)) return false;
  if (block_size != 8 && block_size != 16 && block_size != 32) return false;
  if (num_kv_heads <= 0 || num_heads % num_kv_heads != 0) return false;
  const int G = num_heads / num_kv_heads;
  return G == 1 || G == 2 || G == 4 || G == 8;
}

}  // namespace

void pa::set_last_cuda_error(cudaError_t err) { t_last_cuda_error = err; }

extern "C" {

const char *pa_status_string(int32_t status) {
  switch (status) {
    case PA_OK: return "ok";
    case PA_ERR_NULL: return "a required pointer is NULL";
    case PA_ERR_DIMS: return "invalid or inconsistent sizes";
    case PA_ERR_UNSUPPORTED: return "unsupported dtype, head_dim, block_size or group size";
    case PA_ERR_ALIGN: return "pointer or stride not aligned for 16-byte vectors";
    case PA_ERR_WORKSPACE: return "workspace missing or too small";
    case PA_ERR_LAUNCH: return "kernel launch failed";
    case PA_ERR_DEVICE_BOUNDS: return "a kernel met an out-of-range index (see status flags)";
    case PA_ERR_CUDA: return "CUDA runtime call failed";
    default: return "unknown status";
  }
}

const char *pa_last_cuda_error(void) { return cudaGetErrorName(t_last_cuda_error); }

uint64_t pa_launch_count(void) { return g_launches.load(); }

pa_status pa_attention_set_timing_events(void *start, void *stop) {
  if ((start == nullptr) != (stop == nullptr)) return PA_ERR_NULL;
  t_ev_start = static_cast<cudaEvent_t>(start);
  t_ev_stop = static_cast<cudaEvent_t>(stop);
  return PA_OK;
}

pa_status pa_attention_set_tile_timing_events(void *start, void *stop) {
  if ((start == nullptr) != (stop == nullptr)) return PA_ERR_NULL;
  t_tile_start = static_cast<cudaEvent_t>(start);
  t_tile_stop = static_cast<cudaEvent_t>(stop);
  return PA_OK;
}

pa_status pa_reshape_and_cache(const void *key, const void *value, int64_t key_token_stride,
                               int64_t value_token_stride, void *key_cache, void *value_cache,
                               const int64_t *slot_mapping, int32_t num_tokens, int32_t num_kv_heads,
                               int32_t head_dim, int32_t block_size, int64_t num_blocks, int32_t dtype,
                               void *stream) {
  if (dtype != PA_BF16 && dtype != PA_FP16) return PA_ERR_UNSUPPORTED;
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks < 0)
    return PA_ERR_DIMS;
  if (!supported_head_dim(head_dim)) return PA_ERR_UNSUPPORTED;
  if (block_size != 8 && block_size != 16 && block_size != 32) return PA_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PA_OK;
  if (!key || !value || !key_cache || !value_cache || !slot_mapping) return PA_ERR_NULL;
  const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
  if (row > INT32_MAX) return PA_ERR_UNSUPPORTED;  // a token row's element count is an int32 in the kernel
  if (key_token_stride < row || value_token_stride < row) return PA_ERR_DIMS;
  if (key_token_stride % 8 || value_token_stride % 8) return PA_ERR_ALIGN;
  if (!aligned(key, 16) || !aligned(value, 16) || !aligned(key_cache, 16) || !aligned(value_cache, 16) ||
      !aligned(slot_mapping, 8))
    return PA_ERR_ALIGN;
  DeviceState *ds = device_state();
  if (!ds) return PA_ERR_CUDA;
  cudaError_t err = pa::launch_reshape_and_cache(
      key, value, key_token_stride, value_token_stride, key_cache, value_cache, slot_mapping, num_tokens,
      static_cast<int32_t>(row), num_blocks * block_size, ds->status, ds->sm_count,
      static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_failure(PA_ERR_LAUNCH, err);
  g_launches.fetch_add(1);
  return PA_OK;
}

pa_status pa_reshape_and_cache_fp8(const void *key, const void *value, int64_t key_token_stride,
                                   int64_t value_token_stride, void *key_cache, void *value_cache,
                                   const int64_t *slot_mapping, int32_t num_tokens, int32_t num_kv_heads,
                                   int32_t head_dim, int32_t block_size, int64_t num_blocks, float k_scale,
                                   float v_scale, int32_t dtype, void *stream) {
  if (dtype != PA_BF16 && dtype != PA_FP16) return PA_ERR_UNSUPPORTED;
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks < 0)
    return PA_ERR_DIMS;
  if (!valid_cache_scale(k_scale) || !valid_cache_scale(v_scale)) return PA_ERR_DIMS;
  if (!supported_head_dim(head_dim)) return PA_ERR_UNSUPPORTED;
  if (block_size != 8 && block_size != 16 && block_size != 32) return PA_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PA_OK;
  if (!key || !value || !key_cache || !value_cache || !slot_mapping) return PA_ERR_NULL;
  const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
  if (row > INT32_MAX) return PA_ERR_UNSUPPORTED;  // a token row's element count is an int32 in the kernel
  if (key_token_stride < row || value_token_stride < row) return PA_ERR_DIMS;
  if (key_token_stride % 8 || value_token_stride % 8) return PA_ERR_ALIGN;
  if (!aligned(key, 16) || !aligned(value, 16) || !aligned(key_cache, 16) || !aligned(value_cache, 16) ||
      !aligned(slot_mapping, 8))
    return PA_ERR_ALIGN;
  DeviceState *ds = device_state();
  if (!ds) return PA_ERR_CUDA;
  cudaError_t err = pa::launch_reshape_and_cache_fp8(
      key, value, key_token_stride, value_token_stride, key_cache, value_cache, slot_mapping, num_tokens,
      static_cast<int32_t>(row), num_blocks * block_size, k_scale, v_scale, dtype, ds->status, ds->sm_count,
      static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_failure(PA_ERR_LAUNCH, err);
  g_launches.fetch_add(1);
  return PA_OK;
}

size_t pa_attention_workspace_size(int32_t num_seqs, int32_t total_q_tokens, int32_t max_query_len,
                                   int32_t max_seq_len, int32_t num_heads, int32_t num_kv_heads,
                                   int32_t head_dim, int32_t block_size) {
  if (max_query_len < 0 || max_seq_len < max_query_len) return 0;
  if (!supported_dims(num_heads, num_kv_heads, head_dim, block_size)) return 0;
  // one size for either cache type: the larger of the two plans
  pa::WorkspaceLayout w16, w8;
  if (!pa::workspace_layout(num_seqs, total_q_tokens, max_seq_len, num_heads, num_kv_heads, head_dim, false, w16) ||
      !pa::workspace_layout(num_seqs, total_q_tokens, max_seq_len, num_heads, num_kv_heads, head_dim, true, w8))
    return 0;
  return w16.total > w8.total ? w16.total : w8.total;
}

pa_status pa_attention_plan_info(int32_t num_seqs, int32_t max_seq_len, int32_t num_heads,
                                 int32_t num_kv_heads, int32_t *partition_tokens, int32_t *max_partitions) {
  pa::WorkspaceLayout w;
  if (!pa::workspace_layout(num_seqs, 0, max_seq_len, num_heads, num_kv_heads, 128, false, w)) return PA_ERR_DIMS;
  if (partition_tokens) *partition_tokens = w.part_tokens;
  if (max_partitions) *max_partitions = w.max_parts;
  return PA_OK;
}

}  // extern "C"

namespace {

// pa_attention_varlen and pa_attention_varlen_fp8: validation, then the launch.
pa_status attention_call(const void *q, int64_t q_token_stride, const void *key_cache, const void *value_cache,
                         const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *seq_lens,
                         const int32_t *query_start_loc, int32_t num_seqs, int32_t total_q_tokens,
                         int32_t max_query_len, int32_t max_seq_len, int32_t num_heads, int32_t num_kv_heads,
                         int32_t head_dim, int32_t block_size, int64_t num_blocks, float scale, bool kv_fp8,
                         float k_scale, float v_scale, void *out, void *workspace, size_t workspace_bytes,
                         int32_t dtype, void *stream) {
  cudaEvent_t ev_start = t_ev_start, ev_stop = t_ev_stop, tile_start = t_tile_start, tile_stop = t_tile_stop;
  t_ev_start = t_ev_stop = t_tile_start = t_tile_stop = nullptr;
  if (dtype != PA_BF16 && dtype != PA_FP16) return PA_ERR_UNSUPPORTED;
  if (kv_fp8 && (!valid_cache_scale(k_scale) || !valid_cache_scale(v_scale))) return PA_ERR_DIMS;
  if (num_seqs < 0 || total_q_tokens < 0 || max_query_len < 0 || max_seq_len < max_query_len ||
      max_blocks_per_seq < 0 || num_blocks < 0 || num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0)
    return PA_ERR_DIMS;
  if (!supported_dims(num_heads, num_kv_heads, head_dim, block_size)) {
    if (num_heads % num_kv_heads != 0) return PA_ERR_DIMS;
    return PA_ERR_UNSUPPORTED;
  }
  if (!std::isfinite(scale)) return PA_ERR_DIMS;
  if (num_seqs == 0 || total_q_tokens == 0) return PA_OK;
  if (max_query_len == 0 || max_blocks_per_seq == 0 || num_blocks == 0) return PA_ERR_DIMS;
  if (num_blocks > INT32_MAX / block_size) return PA_ERR_UNSUPPORTED;  // cache rows are int32 TMA coordinates
  if (static_cast<int64_t>(max_query_len) > total_q_tokens) return PA_ERR_DIMS;
  if (!q || !key_cache || !value_cache || !block_tables || !seq_lens || !query_start_loc || !out)
    return PA_ERR_NULL;
  if (q_token_stride < static_cast<int64_t>(num_heads) * head_dim) return PA_ERR_DIMS;
  if (q_token_stride % 2 || !aligned(q, 4)) return PA_ERR_ALIGN;
  if (!aligned(key_cache, 16) || !aligned(value_cache, 16) || !aligned(out, 16) || !aligned(block_tables, 4) ||
      !aligned(seq_lens, 4) || !aligned(query_start_loc, 4))
    return PA_ERR_ALIGN;
  pa::WorkspaceLayout w;
  if (!pa::workspace_layout(num_seqs, total_q_tokens, max_seq_len, num_heads, num_kv_heads, head_dim, kv_fp8, w))
    return PA_ERR_DIMS;
  if (!workspace || workspace_bytes < w.total) return PA_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return PA_ERR_ALIGN;
  DeviceState *ds = device_state();
  if (!ds) return PA_ERR_CUDA;

  pa::AttnLaunch a;
  a.q = q;
  a.q_stride = q_token_stride;
  a.key_cache = key_cache;
  a.value_cache = value_cache;
  a.block_tables = block_tables;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.seq_lens = seq_lens;
  a.query_start_loc = query_start_loc;
  a.num_seqs = num_seqs;
  a.total_q = total_q_tokens;
  a.max_query_len = max_query_len;
  a.max_seq_len = max_seq_len;
  a.num_heads = num_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.block_size = block_size;
  a.num_blocks = num_blocks;
  a.scale = scale;
  a.dtype = dtype;
  a.kv_fp8 = kv_fp8;
  a.k_scale = kv_fp8 ? k_scale : 1.0f;
  a.v_scale = kv_fp8 ? v_scale : 1.0f;
  a.out = out;
  a.workspace = workspace;
  a.status = ds->status;
  a.sm_count = ds->sm_count;
  a.ev_start = ev_start;
  a.ev_stop = ev_stop;
  a.tile_start = tile_start;
  a.tile_stop = tile_stop;
  int launched = 0;
  cudaError_t err = pa::launch_attention(a, static_cast<cudaStream_t>(stream), &launched);
  g_launches.fetch_add(static_cast<uint64_t>(launched));
  if (err != cudaSuccess) return cuda_failure(PA_ERR_LAUNCH, err);
  return PA_OK;
}

}  // namespace

extern "C" {

pa_status pa_attention_varlen(const void *q, int64_t q_token_stride, const void *key_cache,
                              const void *value_cache, const int32_t *block_tables, int32_t max_blocks_per_seq,
                              const int32_t *seq_lens, const int32_t *query_start_loc, int32_t num_seqs,
                              int32_t total_q_tokens, int32_t max_query_len, int32_t max_seq_len,
                              int32_t num_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                              int64_t num_blocks, float scale, void *out, void *workspace,
                              size_t workspace_bytes, int32_t dtype, void *stream) {
  return attention_call(q, q_token_stride, key_cache, value_cache, block_tables, max_blocks_per_seq, seq_lens,
                        query_start_loc, num_seqs, total_q_tokens, max_query_len, max_seq_len, num_heads,
                        num_kv_heads, head_dim, block_size, num_blocks, scale, false, 1.0f, 1.0f, out, workspace,
                        workspace_bytes, dtype, stream);
}

pa_status pa_attention_varlen_fp8(const void *q, int64_t q_token_stride, const void *key_cache,
                                  const void *value_cache, const int32_t *block_tables, int32_t max_blocks_per_seq,
                                  const int32_t *seq_lens, const int32_t *query_start_loc, int32_t num_seqs,
                                  int32_t total_q_tokens, int32_t max_query_len, int32_t max_seq_len,
                                  int32_t num_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                  int64_t num_blocks, float scale, float k_scale, float v_scale, void *out,
                                  void *workspace, size_t workspace_bytes, int32_t dtype, void *stream) {
  return attention_call(q, q_token_stride, key_cache, value_cache, block_tables, max_blocks_per_seq, seq_lens,
                        query_start_loc, num_seqs, total_q_tokens, max_query_len, max_seq_len, num_heads,
                        num_kv_heads, head_dim, block_size, num_blocks, scale, true, k_scale, v_scale, out,
                        workspace, workspace_bytes, dtype, stream);
}

}  // extern "C"

namespace {

pa_status rope_call(void *q, int64_t q_token_stride, const void *key, const void *value, int64_t key_token_stride,
                    int64_t value_token_stride, void *key_cache, void *value_cache, const int64_t *slot_mapping,
                    const int64_t *positions, const float *cos_sin_cache, int32_t max_position, int32_t rotary_dim,
                    int32_t is_neox, int32_t num_tokens, int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                    int32_t block_size, int64_t num_blocks, bool kv8, float k_scale, float v_scale, int32_t dtype,
                    void *stream) {
  if (dtype != PA_BF16 && dtype != PA_FP16) return PA_ERR_UNSUPPORTED;
  if (num_tokens < 0 || num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
      num_blocks < 0 || max_position <= 0 || rotary_dim <= 0 || rotary_dim > head_dim)
    return PA_ERR_DIMS;
  if (kv8 && (!valid_cache_scale(k_scale) || !valid_cache_scale(v_scale))) return PA_ERR_DIMS;
  // 16-byte vectors of elements; 8-bit caches: 8-byte vectors of codes, rows of whole 16-byte vectors
  if (head_dim % (kv8 ? 16 : 8) || rotary_dim % 16) return PA_ERR_ALIGN;
  if (rotary_dim > 512) return PA_ERR_UNSUPPORTED;  // the table row is staged in shared memory
  // a token's q, K and V rows, counted in 16-byte chunks, are an int32 in the kernel
  if ((static_cast<int64_t>(num_heads) + 2 * static_cast<int64_t>(num_kv_heads)) * (head_dim / 8) > INT32_MAX)
    return PA_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PA_OK;
  if (!q || !key || !value || !key_cache || !value_cache || !slot_mapping || !positions || !cos_sin_cache)
    return PA_ERR_NULL;
  const int64_t kv_row = static_cast<int64_t>(num_kv_heads) * head_dim;
  if (q_token_stride < static_cast<int64_t>(num_heads) * head_dim || key_token_stride < kv_row ||
      value_token_stride < kv_row)
    return PA_ERR_DIMS;
  if (q_token_stride % 8 || key_token_stride % 8 || value_token_stride % 8) return PA_ERR_ALIGN;
  if (!aligned(q, 16) || !aligned(key, 16) || !aligned(value, 16) || !aligned(key_cache, 16) ||
      !aligned(value_cache, 16) || !aligned(cos_sin_cache, 16) || !aligned(slot_mapping, 8) || !aligned(positions, 8))
    return PA_ERR_ALIGN;
  DeviceState *ds = device_state();
  if (!ds) return PA_ERR_CUDA;
  cudaError_t err = pa::launch_rope_reshape_and_cache(
      q, q_token_stride, key, value, key_token_stride, value_token_stride, key_cache, value_cache, slot_mapping,
      positions, cos_sin_cache, max_position, rotary_dim, is_neox != 0, num_tokens, num_heads, num_kv_heads,
      head_dim, num_blocks * block_size, dtype, kv8, k_scale, v_scale, ds->status, ds->sm_count,
      static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_failure(PA_ERR_LAUNCH, err);
  g_launches.fetch_add(1);
  return PA_OK;
}

}  // namespace

extern "C" {

pa_status pa_rope_reshape_and_cache(void *q, int64_t q_token_stride, const void *key, const void *value,
                                    int64_t key_token_stride, int64_t value_token_stride, void *key_cache,
                                    void *value_cache, const int64_t *slot_mapping, const int64_t *positions,
                                    const float *cos_sin_cache, int32_t max_position, int32_t rotary_dim,
                                    int32_t is_neox, int32_t num_tokens, int32_t num_heads, int32_t num_kv_heads,
                                    int32_t head_dim, int32_t block_size, int64_t num_blocks, int32_t dtype,
                                    void *stream) {
  return rope_call(q, q_token_stride, key, value, key_token_stride, value_token_stride, key_cache, value_cache,
                   slot_mapping, positions, cos_sin_cache, max_position, rotary_dim, is_neox, num_tokens, num_heads,
                   num_kv_heads, head_dim, block_size, num_blocks, false, 1.0f, 1.0f, dtype, stream);
}

pa_status pa_rope_reshape_and_cache_fp8(void *q, int64_t q_token_stride, const void *key, const void *value,
                                        int64_t key_token_stride, int64_t value_token_stride, void *key_cache,
                                        void *value_cache, const int64_t *slot_mapping, const int64_t *positions,
                                        const float *cos_sin_cache, int32_t max_position, int32_t rotary_dim,
                                        int32_t is_neox, int32_t num_tokens, int32_t num_heads,
                                        int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                        int64_t num_blocks, float k_scale, float v_scale, int32_t dtype,
                                        void *stream) {
  return rope_call(q, q_token_stride, key, value, key_token_stride, value_token_stride, key_cache, value_cache,
                   slot_mapping, positions, cos_sin_cache, max_position, rotary_dim, is_neox, num_tokens, num_heads,
                   num_kv_heads, head_dim, block_size, num_blocks, true, k_scale, v_scale, dtype, stream);
}

pa_status pa_copy_blocks(void *key_cache, void *value_cache, const int64_t *block_mapping, int32_t num_pairs,
                         int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int64_t num_blocks,
                         int32_t dtype, void *stream) {
  const int esize = cache_elem_bytes(dtype);
  if (!esize) return PA_ERR_UNSUPPORTED;
  if (num_pairs < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks < 0) return PA_ERR_DIMS;
  if ((head_dim * esize) % 16) return PA_ERR_ALIGN;  // a block is a whole number of 16-byte vectors
  if (num_pairs == 0) return PA_OK;
  if (!key_cache || !value_cache || !block_mapping) return PA_ERR_NULL;
  if (!aligned(key_cache, 16) || !aligned(value_cache, 16) || !aligned(block_mapping, 8)) return PA_ERR_ALIGN;
  DeviceState *ds = device_state();
  if (!ds) return PA_ERR_CUDA;
  const int64_t block_bytes = static_cast<int64_t>(block_size) * num_kv_heads * head_dim * esize;
  cudaError_t err = pa::launch_copy_blocks(key_cache, value_cache, block_mapping, num_pairs, block_bytes, num_blocks,
                                           ds->status, ds->sm_count, static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_failure(PA_ERR_LAUNCH, err);
  g_launches.fetch_add(1);
  return PA_OK;
}

pa_status pa_gather_kv(const void *key_cache, const void *value_cache, const int32_t *block_table_row,
                       int32_t seq_len, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                       int64_t num_blocks, void *key_out, void *value_out, int32_t dtype, void *stream) {
  const int esize = cache_elem_bytes(dtype);
  if (!esize) return PA_ERR_UNSUPPORTED;
  if (seq_len < 0 || num_kv_heads <= 0 || head_dim <= 0 || num_blocks < 0) return PA_ERR_DIMS;
  if (!supported_head_dim(head_dim)) return PA_ERR_UNSUPPORTED;
  if (block_size != 8 && block_size != 16 && block_size != 32) return PA_ERR_UNSUPPORTED;
  if (seq_len == 0) return PA_OK;
  if (!key_cache || !value_cache || !block_table_row || !key_out || !value_out) return PA_ERR_NULL;
  if (!aligned(key_cache, 16) || !aligned(value_cache, 16) || !aligned(key_out, 16) || !aligned(value_out, 16) ||
      !aligned(block_table_row, 4))
    return PA_ERR_ALIGN;
  const int64_t row_bytes = static_cast<int64_t>(num_kv_heads) * head_dim * esize;
  if (row_bytes > INT32_MAX) return PA_ERR_UNSUPPORTED;  // a cache row's byte count is an int32 in the kernel
  DeviceState *ds = device_state();
  if (!ds) return PA_ERR_CUDA;
  cudaError_t err = pa::launch_gather_kv(key_cache, value_cache, block_table_row, seq_len,
                                         static_cast<int32_t>(row_bytes), block_size, num_blocks, key_out,
                                         value_out, ds->status, ds->sm_count, static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_failure(PA_ERR_LAUNCH, err);
  g_launches.fetch_add(1);
  return PA_OK;
}

pa_status pa_debug_status(void *stream, uint32_t *flags_out) {
  DeviceState *ds = device_state();
  if (!ds) return PA_ERR_CUDA;
  cudaError_t err = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_failure(PA_ERR_CUDA, err);
  unsigned int flags = 0;
  err = cudaMemcpy(&flags, ds->status, sizeof flags, cudaMemcpyDeviceToHost);
  if (err != cudaSuccess) return cuda_failure(PA_ERR_CUDA, err);
  const unsigned int zero = 0;
  err = cudaMemcpy(ds->status, &zero, sizeof zero, cudaMemcpyHostToDevice);
  if (err != cudaSuccess) return cuda_failure(PA_ERR_CUDA, err);
  if (flags_out) *flags_out = flags;
  return flags ? PA_ERR_DEVICE_BOUNDS : PA_OK;
}

}  // extern "C"
