// Types shared by the attention translation units (internal to libpagedattn.so).
#pragma once

#include <cuda.h>

#include "pa_common.cuh"

namespace pa {

using bf16 = __nv_bfloat16;

// Query rows of chunked-prefill requests are packed (position, GQA head) into
// tiles of kPrefillTileRows rows for the tensor-core path, i.e.
// kPrefillTileRows / G positions per tile. Records: {b, first query token,
// positions, absolute position of the first}, {0, key end, -1, 1}.
constexpr int kPrefillTileRows = 256;
// head_dim 256 tiles are one 128-row half (S and O of one half fill the
// tensor memory): kPrefillTileRows128 rows
constexpr int kPrefillTileRows128 = 128;
__host__ __device__ constexpr int prefill_tile_rows(int head_dim) {
  return head_dim == 256 ? kPrefillTileRows128 : kPrefillTileRows;
}

struct TileParams {
  const bf16 *q;
  int64_t q_stride;
  const int32_t *block_tables;
  int32_t max_blocks_per_seq;
  int32_t block_size;   // tokens per cache block: 8, 16 or 32
  int32_t block_shift;  // log2(block_size)
  int32_t num_heads;
  int32_t num_kv_heads;
  int64_t num_blocks;
  float scale_log2;  // softmax scale (times the K cache scale for 8-bit caches) * log2(e)
  float out_scale;   // 1, or the V cache scale for 8-bit caches
  bf16 *out;
  const int4 *tiles;
  const int32_t *tile_count;
  int32_t *tile_counter;
  int32_t num_seqs;
  int32_t total_q;
  int32_t max_tiles;
  unsigned int *status;
};

// Enqueue the tensor-core prefill-tile kernel (PDL launch) on `stream`; E is
// the element type of q and out (ElemBf16 or ElemFp16); KV8: the caches hold
// 8-bit E4M3 codes (the maps then have one-byte elements and boxes of
// min(block_size, 32) rows of head_dim codes).
// vmapb: at head_dim 128 over 16-bit caches, the value cache as whole-block
// boxes (block_size rows x both 64-element atoms; unused otherwise).
template <int D, int G, typename E, bool KV8>
cudaError_t launch_prefill_tiles(const CUtensorMap &kmap, const CUtensorMap &vmap, const CUtensorMap &vmapb,
                                 const TileParams &tp, int sm_count, cudaStream_t stream);

}  // namespace pa
