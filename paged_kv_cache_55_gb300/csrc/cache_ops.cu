// reshape_and_cache (scatter of a step's new K/V rows into the paged cache),
// the copy-on-write block copy, and the block-table gather used to check
// addressing.
//
// vLLM inference notes ("AI Infra入门干货总结：大模型是如何高效推理的"),
// §Paged Attention: slot_mapping names where each new token's K/V goes;
// slot = block * block_size + offset. The cache is [num_blocks, block_size,
// num_kv_heads, head_dim], so cache row (block, offset) is flat row
// block * block_size + offset == slot, and a token row of num_kv_heads *
// head_dim elements is one contiguous run of 16-byte vectors.
#include "pa_common.cuh"
#include "pa_launch.h"

namespace pa {

// One thread moves one 16-byte vector of K and the matching one of V.
// Consecutive threads cover consecutive vectors of a token row, so both the
// read of key[t] and the write of the cache row are fully coalesced.
__global__ void __launch_bounds__(256) reshape_and_cache_kernel(
    const uint4 *__restrict__ key, const uint4 *__restrict__ value, int64_t key_stride16,
    int64_t value_stride16, uint4 *__restrict__ key_cache, uint4 *__restrict__ value_cache,
    const int64_t *__restrict__ slot_mapping, int32_t num_tokens, int32_t row16, int64_t num_slots,
    unsigned int *status) {
  griddep_wait();
  griddep_launch_dependents();
  const int64_t total = static_cast<int64_t>(num_tokens) * row16;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int32_t t = static_cast<int32_t>(i / row16);
    const int32_t c = static_cast<int32_t>(i - static_cast<int64_t>(t) * row16);
    const int64_t slot = ld_cg(reinterpret_cast<const long long *>(slot_mapping) + t);
    if (slot < 0) continue;  // padding token
    if (slot >= num_slots) {
      if (c == 0) flag_error(status, PA_FLAG_SLOT_RANGE);
      continue;
    }
    const uint4 k = ld_cg(key + t * key_stride16 + c);
    const uint4 v = ld_cg(value + t * value_stride16 + c);
    key_cache[slot * row16 + c] = k;
    value_cache[slot * row16 + c] = v;
  }
}

// Logical row j of one request -> contiguous output row j.
__global__ void __launch_bounds__(256) gather_kv_kernel(
    const uint4 *__restrict__ key_cache, const uint4 *__restrict__ value_cache,
    const int32_t *__restrict__ table_row, int32_t seq_len, int32_t row16, int64_t num_blocks,
    uint4 *__restrict__ key_out, uint4 *__restrict__ value_out, unsigned int *status) {
  const int64_t total = static_cast<int64_t>(seq_len) * row16;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int32_t j = static_cast<int32_t>(i / row16);
    const int32_t c = static_cast<int32_t>(i - static_cast<int64_t>(j) * row16);
    const int32_t phys = __ldg(table_row + j / kBlockSize);
    if (phys < 0 || phys >= num_blocks) {
      if (c == 0) flag_error(status, PA_FLAG_BLOCK_RANGE);
      key_out[i] = make_uint4(0, 0, 0, 0);
      value_out[i] = make_uint4(0, 0, 0, 0);
      continue;
    }
    const int64_t src = (static_cast<int64_t>(phys) * kBlockSize + (j % kBlockSize)) * row16 + c;
    key_out[i] = __ldg(key_cache + src);
    value_out[i] = __ldg(value_cache + src);
  }
}

// Copy-on-write block copy (LLM-infra reading map, §2.2: a shared block is
// copied before a request that shares it writes to it): pair i copies
// physical block mapping[2i] to block mapping[2i + 1] in both caches. A block
// of one cache is one contiguous run of block16 16-byte vectors; a CTA copies
// whole blocks, its threads striding over the vectors with four loads of each
// cache in flight. Sources are read after the dependency wait with
// ld.global.cg: a preceding kernel (the cache scatter) may have written them.
__global__ void __launch_bounds__(256) copy_blocks_kernel(uint4 *key_cache, uint4 *value_cache,
                                                          const int64_t *__restrict__ mapping, int32_t num_pairs,
                                                          int64_t block16, int64_t num_blocks, unsigned int *status) {
  griddep_wait();
  griddep_launch_dependents();
  constexpr int kUnroll = 4;
  for (int32_t pair = blockIdx.x; pair < num_pairs; pair += gridDim.x) {
    const int64_t src = ld_cg(reinterpret_cast<const long long *>(mapping) + 2 * static_cast<int64_t>(pair));
    const int64_t dst = ld_cg(reinterpret_cast<const long long *>(mapping) + 2 * static_cast<int64_t>(pair) + 1);
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
      if (threadIdx.x == 0) flag_error(status, PA_FLAG_BLOCK_RANGE);
      continue;
    }
    const uint4 *ks = key_cache + src * block16, *vs = value_cache + src * block16;
    uint4 *kd = key_cache + dst * block16, *vd = value_cache + dst * block16;
    for (int64_t i0 = threadIdx.x; i0 < block16; i0 += kUnroll * blockDim.x) {
      uint4 a[kUnroll], b[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t i = i0 + u * blockDim.x;
        if (i < block16) {
          a[u] = ld_cg(ks + i);
          b[u] = ld_cg(vs + i);
        }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t i = i0 + u * blockDim.x;
        if (i < block16) {
          kd[i] = a[u];
          vd[i] = b[u];
        }
      }
    }
  }
}

static int grid_for(int64_t work, int threads, int sm_count) {
  int64_t g = (work + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(sm_count) * 8;
  if (g > cap) g = cap;
  if (g < 1) g = 1;
  return static_cast<int>(g);
}

cudaError_t launch_reshape_and_cache(const void *key, const void *value, int64_t key_stride,
                                     int64_t value_stride, void *key_cache, void *value_cache,
                                     const int64_t *slot_mapping, int32_t num_tokens, int32_t row_elems,
                                     int64_t num_slots, unsigned int *status, int sm_count,
                                     cudaStream_t stream) {
  const int32_t row16 = row_elems / 8;
  const int grid = grid_for(static_cast<int64_t>(num_tokens) * row16, 256, sm_count);
  return launch_pdl(reshape_and_cache_kernel, dim3(grid), dim3(256), 0, stream, static_cast<const uint4 *>(key),
                    static_cast<const uint4 *>(value), key_stride / 8, value_stride / 8,
                    static_cast<uint4 *>(key_cache), static_cast<uint4 *>(value_cache), slot_mapping, num_tokens,
                    row16, num_slots, status);
}

cudaError_t launch_copy_blocks(void *key_cache, void *value_cache, const int64_t *mapping, int32_t num_pairs,
                               int64_t block_elems, int64_t num_blocks, unsigned int *status, int sm_count,
                               cudaStream_t stream) {
  int64_t grid = static_cast<int64_t>(sm_count) * 4;  // 4 CTAs of 256 threads per SM
  if (grid > num_pairs) grid = num_pairs;
  if (grid < 1) grid = 1;
  return launch_pdl(copy_blocks_kernel, dim3(static_cast<unsigned>(grid)), dim3(256), 0, stream,
                    static_cast<uint4 *>(key_cache), static_cast<uint4 *>(value_cache), mapping, num_pairs,
                    block_elems / 8, num_blocks, status);
}

cudaError_t launch_gather_kv(const void *key_cache, const void *value_cache, const int32_t *table_row,
                             int32_t seq_len, int32_t row_elems, int64_t num_blocks, void *key_out,
                             void *value_out, unsigned int *status, int sm_count, cudaStream_t stream) {
  const int32_t row16 = row_elems / 8;
  const int grid = grid_for(static_cast<int64_t>(seq_len) * row16, 256, sm_count);
  gather_kv_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint4 *>(key_cache),
                                             static_cast<const uint4 *>(value_cache), table_row, seq_len,
                                             row16, num_blocks, static_cast<uint4 *>(key_out),
                                             static_cast<uint4 *>(value_out), status);
  return cudaGetLastError();
}

}  // namespace pa
