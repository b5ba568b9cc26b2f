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

// 8-bit caches (LLM-infra reading map, §4.2: the cache is quantised online
// as it is written): the same slots, each element stored as the E4M3 code of
// its binary32 quotient by the cache's scale. One thread turns 16 elements
// (two 16-byte loads) into one 16-byte vector of codes.
template <typename E>
__device__ __forceinline__ uint4 quantize16(uint4 a, uint4 b, float scale) {
  const uint32_t x[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  uint32_t c[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t p0 = e4m3x2_from_f32(__fdiv_rn(E::lo(x[2 * k]), scale), __fdiv_rn(E::hi(x[2 * k]), scale));
    const uint32_t p1 =
        e4m3x2_from_f32(__fdiv_rn(E::lo(x[2 * k + 1]), scale), __fdiv_rn(E::hi(x[2 * k + 1]), scale));
    c[k] = p0 | (p1 << 16);
  }
  return make_uint4(c[0], c[1], c[2], c[3]);
}

template <typename E>
__global__ void __launch_bounds__(256) reshape_and_cache_fp8_kernel(
    const uint4 *__restrict__ key, const uint4 *__restrict__ value, int64_t key_stride16,
    int64_t value_stride16, uint4 *__restrict__ key_cache, uint4 *__restrict__ value_cache,
    const int64_t *__restrict__ slot_mapping, int32_t num_tokens, int32_t row16, int64_t num_slots, float k_scale,
    float v_scale, unsigned int *status) {
  griddep_wait();
  griddep_launch_dependents();
  // row16: 16-element groups per token row (one 16-byte vector of codes, two of elements)
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
    const uint4 *kp = key + t * key_stride16 + 2 * c;
    const uint4 *vp = value + t * value_stride16 + 2 * c;
    key_cache[slot * row16 + c] = quantize16<E>(ld_cg(kp), ld_cg(kp + 1), k_scale);
    value_cache[slot * row16 + c] = quantize16<E>(ld_cg(vp), ld_cg(vp + 1), v_scale);
  }
}

// Logical row j of one request -> contiguous output row j.
__global__ void __launch_bounds__(256) gather_kv_kernel(
    const uint4 *__restrict__ key_cache, const uint4 *__restrict__ value_cache,
    const int32_t *__restrict__ table_row, int32_t seq_len, int32_t row16, int32_t block_size, int64_t num_blocks,
    uint4 *__restrict__ key_out, uint4 *__restrict__ value_out, unsigned int *status) {
  const int64_t total = static_cast<int64_t>(seq_len) * row16;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int32_t j = static_cast<int32_t>(i / row16);
    const int32_t c = static_cast<int32_t>(i - static_cast<int64_t>(j) * row16);
    const int32_t phys = __ldg(table_row + j / block_size);
    if (phys < 0 || phys >= num_blocks) {
      if (c == 0) flag_error(status, PA_FLAG_BLOCK_RANGE);
      key_out[i] = make_uint4(0, 0, 0, 0);
      value_out[i] = make_uint4(0, 0, 0, 0);
      continue;
    }
    const int64_t src = (static_cast<int64_t>(phys) * block_size + (j % block_size)) * row16 + c;
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

// Rotary position embedding fused with the cache scatter (vLLM notes, §LLM
// 推理全流程 2: a token's position is a rotation angle; cos_sin_cache is
// [max_position, rotary_dim], precomputed). Row p holds cos(p theta_i) in
// columns i < rotary_dim / 2 and sin(p theta_i) in the next rotary_dim / 2;
// a pair (x1, x2) becomes (x1 cos - x2 sin, x2 cos + x1 sin). Pairs are
// (i, i + rotary_dim / 2) (NEOX) or (2i, 2i + 1). One thread per 16-byte chunk
// c of one row of one token: rows [0, H) are q heads (rotated in place),
// [H, H + Hkv) K heads (rotated into the cache slot), the next Hkv V heads
// (copied to the slot). With NEOX pairing the thread of chunk c < rot / 16
// also does its partner chunk c + rot / 16. fp32 arithmetic, one rounding to
// the element type; a token whose position is outside [0, max_position) is
// skipped and flagged.
template <typename E>
__device__ __forceinline__ void rope_pair8(uint4 &a, uint4 &b, const float *c, const float *s) {
  // a holds x1 of 8 pairs, b their x2 (NEOX layout)
  uint32_t *pa = reinterpret_cast<uint32_t *>(&a), *pb = reinterpret_cast<uint32_t *>(&b);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float x10 = E::lo(pa[k]), x11 = E::hi(pa[k]), x20 = E::lo(pb[k]), x21 = E::hi(pb[k]);
    const float c0 = c[2 * k], c1 = c[2 * k + 1], s0 = s[2 * k], s1 = s[2 * k + 1];
    pa[k] = E::pack(fmaf(x10, c0, -x20 * s0), fmaf(x11, c1, -x21 * s1));
    pb[k] = E::pack(fmaf(x20, c0, x10 * s0), fmaf(x21, c1, x11 * s1));
  }
}
template <typename E>
__device__ __forceinline__ void rope_adjacent8(uint4 &a, const float *c, const float *s) {
  // a holds 4 pairs (x1, x2) side by side (GPT-J layout)
  uint32_t *pa = reinterpret_cast<uint32_t *>(&a);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float x1 = E::lo(pa[k]), x2 = E::hi(pa[k]);
    pa[k] = E::pack(fmaf(x1, c[k], -x2 * s[k]), fmaf(x2, c[k], x1 * s[k]));
  }
}

constexpr int kRopeMaxRot = 512;  // largest rotary_dim (a table row is staged in shared memory per warp)
constexpr int kRopeWarps = 8;     // tokens in flight per CTA (one per warp)

// Four floats of a table written before this kernel (the rotary table may come
// from an earlier kernel of the stream): a volatile, L1-cached load that the
// compiler cannot hoist above griddep_wait (as it may an invariant load).
__device__ __forceinline__ float4 ld_ca4(const float *p) {
  float4 v;
  asm volatile("ld.global.ca.v4.f32 {%0, %1, %2, %3}, [%4];\n"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p)
               : "memory");
  return v;
}

// Eight elements -> eight E4M3 codes of x / scale (the quantiser of reshape_and_cache_fp8).
template <typename E>
__device__ __forceinline__ uint2 quantize8(uint4 a, float scale) {
  const uint32_t x[4] = {a.x, a.y, a.z, a.w};
  uint32_t c[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const uint32_t p0 = e4m3x2_from_f32(__fdiv_rn(E::lo(x[2 * k]), scale), __fdiv_rn(E::hi(x[2 * k]), scale));
    const uint32_t p1 =
        e4m3x2_from_f32(__fdiv_rn(E::lo(x[2 * k + 1]), scale), __fdiv_rn(E::hi(x[2 * k + 1]), scale));
    c[k] = p0 | (p1 << 16);
  }
  return make_uint2(c[0], c[1]);
}

// KV8: the caches hold E4M3 codes; the rotated key row (rounded to the
// element type, as for 16-bit caches) and the value row are quantised by the
// cache scales on their way in, eight elements to one 8-byte store.
template <typename E, bool NEOX, bool KV8>
__global__ void __launch_bounds__(256) rope_reshape_and_cache_kernel(
    uint4 *q, int64_t q_stride16, const uint4 *__restrict__ key, const uint4 *__restrict__ value,
    int64_t key_stride16, int64_t value_stride16, void *__restrict__ key_cache_v, void *__restrict__ value_cache_v,
    const int64_t *__restrict__ slot_mapping, const int64_t *__restrict__ positions,
    const float *__restrict__ cos_sin, int32_t max_position, int32_t rot, int32_t num_tokens, int32_t num_heads,
    int32_t num_kv_heads, int32_t d16, int64_t num_slots, float k_scale, float v_scale, int32_t slices,
    unsigned int *status) {
  // 16-bit caches: one 16-byte vector per 8-element chunk; 8-bit: one 8-byte vector
  uint4 *key_cache = static_cast<uint4 *>(key_cache_v), *value_cache = static_cast<uint4 *>(value_cache_v);
  uint2 *key_cache8 = static_cast<uint2 *>(key_cache_v), *value_cache8 = static_cast<uint2 *>(value_cache_v);
  griddep_wait();
  griddep_launch_dependents();
  const int32_t half16 = rot / 16;  // chunks in one half of the rotated part (NEOX)
  // Work items of a token: per q head the rotated chunks (NEOX: chunk c <
  // half16 with its partner c + half16; GPT-J: chunk c < rot / 8); per K head
  // those and the chunks past the rotated part; per V head every chunk.
  const int32_t uq = NEOX ? half16 : rot / 8, uk = NEOX ? d16 - half16 : d16;
  const int32_t kq = num_heads * uq, kk = kq + num_kv_heads * uk;
  const int32_t items = kk + num_kv_heads * d16;
  const int64_t row16 = static_cast<int64_t>(num_kv_heads) * d16;

  // One warp per (token, slice of its chunks), eight per CTA at a time (a
  // step with few tokens splits each token's chunks into `slices` so that
  // every SM has work), with no CTA-wide synchronisation: the lanes read the
  // token's position and slot (one broadcast load each), stage its cos/sin
  // row in the warp's own shared memory (L1-cached loads, issued after the
  // wait above), and issue the loads of kBatch chunks each before they
  // rotate and store any. A rotating chunk's thread also does its partner
  // chunk, whichever slice that lies in.
  constexpr int kBatch = 4;
  __shared__ __align__(16) float tabs[kRopeWarps][kRopeMaxRot];
  const int wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float *tw = tabs[wid];
  const int64_t units = static_cast<int64_t>(num_tokens) * slices;
  for (int64_t u = static_cast<int64_t>(blockIdx.x) * kRopeWarps + wid; u < units;
       u += static_cast<int64_t>(gridDim.x) * kRopeWarps) {
    const int32_t t = static_cast<int32_t>(u / slices), sl = static_cast<int32_t>(u - static_cast<int64_t>(t) * slices);
    const int32_t w_begin = static_cast<int32_t>(static_cast<int64_t>(items) * sl / slices);
    const int32_t w_end = static_cast<int32_t>(static_cast<int64_t>(items) * (sl + 1) / slices);
    const int64_t pos = ld_cg(reinterpret_cast<const long long *>(positions) + t);
    const int64_t slot = ld_cg(reinterpret_cast<const long long *>(slot_mapping) + t);
    if (!(pos >= 0 && pos < max_position)) {
      if (lane == 0 && sl == 0) flag_error(status, PA_FLAG_POSITION_RANGE);
      continue;
    }
    if (slot >= num_slots && lane == 0 && sl == 0) flag_error(status, PA_FLAG_SLOT_RANGE);
    const bool cache_ok = slot >= 0 && slot < num_slots;  // slot < 0: padding token, nothing cached
    __syncwarp();  // the warp's previous token is done with tw
    for (int32_t i = lane; i < rot / 4; i += 32)
      reinterpret_cast<float4 *>(tw)[i] = ld_ca4(cos_sin + pos * rot + 4 * i);
    __syncwarp();
    for (int32_t w0 = w_begin + lane; w0 < w_end; w0 += kBatch * 32) {
      uint4 x[kBatch], y[kBatch];
      int kind[kBatch];  // 0 nothing, 1 q head, 2 K head, 3 V head
      // loads
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const int32_t w = w0 + k * 32;
        kind[k] = 0;
        if (w >= w_end) continue;
        // item -> (row kind, head, chunk); NEOX K items past the rotated pairs skip the partner chunks
        if (w < kq) {  // q head: in place
          const int32_t h = w / uq, c = w - h * uq;
          const uint4 *qrow = q + static_cast<int64_t>(t) * q_stride16 + static_cast<int64_t>(h) * d16;
          x[k] = ld_cg(qrow + c);
          if (NEOX) y[k] = ld_cg(qrow + c + half16);
          kind[k] = 1;
        } else if (!cache_ok) {
          continue;
        } else if (w < kk) {  // K head: rotated into the cache
          const int32_t h = (w - kq) / uk, j = (w - kq) - h * uk;
          const int32_t c = NEOX && j >= half16 ? j + half16 : j;
          const uint4 *src = key + static_cast<int64_t>(t) * key_stride16 + static_cast<int64_t>(h) * d16;
          x[k] = ld_cg(src + c);
          if (NEOX && c < half16) y[k] = ld_cg(src + c + half16);
          kind[k] = 2;
        } else {  // V head: copied
          const int32_t h = (w - kk) / d16, c = (w - kk) - h * d16;
          x[k] = ld_cg(value + static_cast<int64_t>(t) * value_stride16 + static_cast<int64_t>(h) * d16 + c);
          kind[k] = 3;
        }
      }
      // rotations and stores
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        if (kind[k] == 0) continue;
        const int32_t w = w0 + k * 32;
        int32_t h, c;
        if (kind[k] == 1) {
          h = w / uq;
          c = w - h * uq;
        } else if (kind[k] == 2) {
          h = (w - kq) / uk;
          const int32_t j = (w - kq) - h * uk;
          c = NEOX && j >= half16 ? j + half16 : j;
        } else {
          h = (w - kk) / d16;
          c = (w - kk) - h * d16;
        }
        const bool rotates = NEOX ? c < half16 : c < rot / 8;
        if (rotates && kind[k] != 3) {
          const int base = NEOX ? 8 * c : 4 * c;  // first frequency index of this chunk
          float cf[8], sf[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            cf[e] = (NEOX || e < 4) ? tw[base + e] : 0.f;
            sf[e] = (NEOX || e < 4) ? tw[rot / 2 + base + e] : 0.f;
          }
          if (NEOX)
            rope_pair8<E>(x[k], y[k], cf, sf);
          else
            rope_adjacent8<E>(x[k], cf, sf);
        }
        if (kind[k] == 1) {
          uint4 *qrow = q + static_cast<int64_t>(t) * q_stride16 + static_cast<int64_t>(h) * d16;
          if (NEOX) qrow[c + half16] = y[k];
          qrow[c] = x[k];
        } else if (kind[k] == 2) {
          const int64_t dofs = slot * row16 + static_cast<int64_t>(h) * d16;
          if (NEOX && rotates) {
            if constexpr (KV8)
              key_cache8[dofs + c + half16] = quantize8<E>(y[k], k_scale);
            else
              key_cache[dofs + c + half16] = y[k];
          }
          if constexpr (KV8)
            key_cache8[dofs + c] = quantize8<E>(x[k], k_scale);
          else
            key_cache[dofs + c] = x[k];
        } else {
          const int64_t dofs = slot * row16 + static_cast<int64_t>(h) * d16;
          if constexpr (KV8)
            value_cache8[dofs + c] = quantize8<E>(x[k], v_scale);
          else
            value_cache[dofs + c] = x[k];
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

cudaError_t launch_reshape_and_cache_fp8(const void *key, const void *value, int64_t key_stride,
                                         int64_t value_stride, void *key_cache, void *value_cache,
                                         const int64_t *slot_mapping, int32_t num_tokens, int32_t row_elems,
                                         int64_t num_slots, float k_scale, float v_scale, int32_t dtype,
                                         unsigned int *status, int sm_count, cudaStream_t stream) {
  const int32_t row16 = row_elems / 16;
  const int grid = grid_for(static_cast<int64_t>(num_tokens) * row16, 256, sm_count);
  auto kern = dtype == PA_FP16 ? reshape_and_cache_fp8_kernel<ElemFp16> : reshape_and_cache_fp8_kernel<ElemBf16>;
  return launch_pdl(kern, dim3(grid), dim3(256), 0, stream, static_cast<const uint4 *>(key),
                    static_cast<const uint4 *>(value), key_stride / 8, value_stride / 8,
                    static_cast<uint4 *>(key_cache), static_cast<uint4 *>(value_cache), slot_mapping, num_tokens,
                    row16, num_slots, k_scale, v_scale, status);
}

cudaError_t launch_copy_blocks(void *key_cache, void *value_cache, const int64_t *mapping, int32_t num_pairs,
                               int64_t block_bytes, int64_t num_blocks, unsigned int *status, int sm_count,
                               cudaStream_t stream) {
  int64_t grid = static_cast<int64_t>(sm_count) * 4;  // 4 CTAs of 256 threads per SM
  if (grid > num_pairs) grid = num_pairs;
  if (grid < 1) grid = 1;
  return launch_pdl(copy_blocks_kernel, dim3(static_cast<unsigned>(grid)), dim3(256), 0, stream,
                    static_cast<uint4 *>(key_cache), static_cast<uint4 *>(value_cache), mapping, num_pairs,
                    block_bytes / 16, num_blocks, status);
}

cudaError_t launch_rope_reshape_and_cache(void *q, int64_t q_stride, const void *key, const void *value,
                                          int64_t key_stride, int64_t value_stride, void *key_cache,
                                          void *value_cache, const int64_t *slot_mapping, const int64_t *positions,
                                          const float *cos_sin_cache, int32_t max_position, int32_t rotary_dim,
                                          bool is_neox, int32_t num_tokens, int32_t num_heads, int32_t num_kv_heads,
                                          int32_t head_dim, int64_t num_slots, int32_t dtype, bool kv8, float k_scale,
                                          float v_scale, unsigned int *status, int sm_count, cudaStream_t stream) {
  const int32_t d16 = head_dim / 8;
  // slices per token: enough (token, slice) units for about 24 warps per SM, at most 8 per token
  const int64_t want = static_cast<int64_t>(sm_count) * 24;
  int32_t slices = static_cast<int32_t>((want + num_tokens - 1) / (num_tokens > 0 ? num_tokens : 1));
  slices = slices < 1 ? 1 : (slices > 8 ? 8 : slices);
  int64_t g = static_cast<int64_t>(sm_count) * 4;  // CTAs of kRopeWarps units in flight: 4 per SM at most
  const int64_t need = (static_cast<int64_t>(num_tokens) * slices + kRopeWarps - 1) / kRopeWarps;
  if (g > need) g = need;
  const int grid = static_cast<int>(g < 1 ? 1 : g);
#define PA_ROPE_LAUNCH(EE, NN, K8)                                                                                \
  return launch_pdl(rope_reshape_and_cache_kernel<EE, NN, K8>, dim3(grid), dim3(256), 0, stream,                  \
                    static_cast<uint4 *>(q), q_stride / 8, static_cast<const uint4 *>(key),                        \
                    static_cast<const uint4 *>(value), key_stride / 8, value_stride / 8, key_cache, value_cache,    \
                    slot_mapping, positions, cos_sin_cache, max_position, rotary_dim, num_tokens, num_heads,        \
                    num_kv_heads, d16, num_slots, k_scale, v_scale, slices, status);
#define PA_ROPE_KV(EE, NN) \
  if (kv8) PA_ROPE_LAUNCH(EE, NN, true) else PA_ROPE_LAUNCH(EE, NN, false)
  if (dtype == PA_FP16) {
    if (is_neox) PA_ROPE_KV(ElemFp16, true) else PA_ROPE_KV(ElemFp16, false)
  } else {
    if (is_neox) PA_ROPE_KV(ElemBf16, true) else PA_ROPE_KV(ElemBf16, false)
  }
#undef PA_ROPE_KV
#undef PA_ROPE_LAUNCH
}

cudaError_t launch_gather_kv(const void *key_cache, const void *value_cache, const int32_t *table_row,
                             int32_t seq_len, int32_t row_bytes, int32_t block_size, int64_t num_blocks, void *key_out,
                             void *value_out, unsigned int *status, int sm_count, cudaStream_t stream) {
  const int32_t row16 = row_bytes / 16;
  const int grid = grid_for(static_cast<int64_t>(seq_len) * row16, 256, sm_count);
  gather_kv_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint4 *>(key_cache),
                                             static_cast<const uint4 *>(value_cache), table_row, seq_len,
                                             row16, block_size, num_blocks, static_cast<uint4 *>(key_out),
                                             static_cast<uint4 *>(value_out), status);
  return cudaGetLastError();
}

}  // namespace pa
