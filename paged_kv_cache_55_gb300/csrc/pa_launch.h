// Host-side launch interface between the C ABI (api.cu) and the kernels'
// translation units. Internal to libpagedattn.so.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace pa {

// Record the CUDA error behind a PA_ERR_LAUNCH / PA_ERR_CUDA return, for
// pa_last_cuda_error() on the calling host thread (defined in api.cu).
void set_last_cuda_error(cudaError_t err);

cudaError_t launch_reshape_and_cache(const void *key, const void *value, int64_t key_stride,
                                     int64_t value_stride, void *key_cache, void *value_cache,
                                     const int64_t *slot_mapping, int32_t num_tokens, int32_t row_elems,
                                     int64_t num_slots, unsigned int *status, int sm_count,
                                     cudaStream_t stream);

// 8-bit caches: elements of `dtype` in, E4M3 codes of x / scale out.
cudaError_t launch_reshape_and_cache_fp8(const void *key, const void *value, int64_t key_stride,
                                         int64_t value_stride, void *key_cache, void *value_cache,
                                         const int64_t *slot_mapping, int32_t num_tokens, int32_t row_elems,
                                         int64_t num_slots, float k_scale, float v_scale, int32_t dtype,
                                         unsigned int *status, int sm_count, cudaStream_t stream);

cudaError_t launch_copy_blocks(void *key_cache, void *value_cache, const int64_t *mapping, int32_t num_pairs,
                               int64_t block_bytes, int64_t num_blocks, unsigned int *status, int sm_count,
                               cudaStream_t stream);

cudaError_t launch_rope_reshape_and_cache(void *q, int64_t q_stride, const void *key, const void *value,
                                          int64_t key_stride, int64_t value_stride, void *key_cache,
                                          void *value_cache, const int64_t *slot_mapping, const int64_t *positions,
                                          const float *cos_sin_cache, int32_t max_position, int32_t rotary_dim,
                                          bool is_neox, int32_t num_tokens, int32_t num_heads, int32_t num_kv_heads,
                                          int32_t head_dim, int64_t num_slots, int32_t dtype, bool kv8, float k_scale,
                                          float v_scale, unsigned int *status, int sm_count, cudaStream_t stream);

cudaError_t launch_gather_kv(const void *key_cache, const void *value_cache, const int32_t *table_row,
                             int32_t seq_len, int32_t row_bytes, int32_t block_size, int64_t num_blocks, void *key_out,
                             void *value_out, unsigned int *status, int sm_count, cudaStream_t stream);

// Byte offsets of the pieces of the attention workspace, and the split plan.
struct WorkspaceLayout {
  size_t item_start, nparts, item_count, items, tiles, part_lse, part_o, total;
  int32_t part_tokens;    // keys per partition
  int32_t max_parts;      // partitions of the longest request
  int32_t max_items;      // upper bound on decode work items (per KV head)
  int32_t max_tiles;      // upper bound on prefill tiles (per KV head)
  int32_t rows_per_item;  // query rows per item: 8 / group size
};

// kv8: the plan for 8-bit caches (more decode warps per SM, so partitions
// can be smaller). pa_attention_workspace_size covers both plans.
bool workspace_layout(int32_t num_seqs, int32_t total_q, int32_t max_seq_len, int32_t num_heads,
                      int32_t num_kv_heads, int32_t head_dim, bool kv8, WorkspaceLayout &w);

struct AttnLaunch {
  const void *q;
  int64_t q_stride;
  const void *key_cache, *value_cache;
  const int32_t *block_tables;
  int32_t max_blocks_per_seq;
  const int32_t *seq_lens, *query_start_loc;
  int32_t num_seqs, total_q, max_query_len, max_seq_len;
  int32_t num_heads, num_kv_heads, head_dim, block_size;
  int64_t num_blocks;
  float scale;
  int32_t dtype;  // PA_BF16 or PA_FP16 (q and out; the caches too unless kv_fp8)
  bool kv_fp8;    // caches hold E4M3 codes: K = code * k_scale, V = code * v_scale
  float k_scale, v_scale;
  void *out;
  void *workspace;
  unsigned int *status;
  int sm_count;
  cudaEvent_t ev_start, ev_stop;      // around the split-KV decode kernel, if set
  cudaEvent_t tile_start, tile_stop;  // around the prefill-tile kernel, if set and launched
};

// Enqueue planning, split-KV attention and (when a request can be split) the
// partition merge on `stream`; *launched counts kernels.
cudaError_t launch_attention(const AttnLaunch &a, cudaStream_t stream, int *launched);

}  // namespace pa
