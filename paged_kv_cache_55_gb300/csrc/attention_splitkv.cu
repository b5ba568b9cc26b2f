// Paged attention for a continuous-batching step: planning, split-KV
// attention over the block table, and the log-sum-exp merge of partitions.
//
// Sources (vLLM inference notes, "AI Infra入门干货总结：大模型是如何高效推理的"):
//   §Paged Attention - cache [num_blocks, block_size, num_kv_heads, head_dim],
//     block_table per request, 16-token blocks keep rows contiguous inside a
//     block while blocks themselves are scattered.
//   §LLM 推理全流程 3 (Attention) - K/V read discretely through the table,
//     Q [query_lens, num_heads, head_dim], GQA by index (no KV copies);
//     FlashAttention: fused kernel, tiling, online softmax so that S and P
//     never reach HBM; decode is memory-bound (GEMV + KV read).
//   §Continuous Batching - a step mixes requests; query i of a request sits
//     at position seq_len - query_len + i and sees keys up to it.
// Splitting one request's keys into partitions and merging the partial
// results by their log-sum-exp is Flash-Decoding, which the LLM-infra reading
// map ("lpnh.cn/news/2436702", §6) names as FlashAttention's follow-up.
//
// Design:
//   * A work unit is (request, KV head, group of up to 8/G query rows,
//     partition of keys). Its 8 "columns" are (query row, head of the GQA
//     group) pairs, so one pass over a KV block serves the whole group: each
//     K/V byte is read from HBM once per step.
//   * Every warp is an independent pipeline. It takes units from a global
//     counter, and stages the (block, KV head) tiles of K and V with TMA
//     (cp.async.bulk.tensor, 128-byte swizzle) into its own ring of shared
//     memory slots, each completed through an mbarrier. The ring runs ahead
//     across unit boundaries, so the HBM stream does not drain between units.
//     No CTA-wide barrier is taken after start-up.
//   * Scores are computed transposed, S^T[16 keys x 8 columns] = K Q^T, with
//     mma.sync m16n8k16 (bf16 in, fp32 accumulate); movmatrix moves the
//     probabilities into the B-operand layout and O^T += V^T P^T is a second
//     mma, with P as a bf16 hi + lo pair so the weights keep ~16 significant
//     bits. The tensor pipe only removes instruction pressure: the kernel is
//     bound by HBM bandwidth.
//   * The last block of a request may hold stale or NaN rows past seq_len:
//     the warp zeroes those V rows in its slot before use, and masked scores
//     are selected to -inf, never multiplied by zero.
//   * Online softmax per column in the log2 domain (scale folded with log2 e),
//     max reductions by warp shuffles.
//   * Units of a split request write fp32 (o, lse) partials; a merge kernel
//     combines them: lse = log2 sum 2^lse_p, o = sum 2^(lse_p - lse) o_p,
//     summing the partitions in order (deterministic bits).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <float.h>

#include <mutex>
#include <type_traits>

#include "attention_internal.cuh"
#include "pa_launch.h"

namespace pa {

constexpr int kCols = 8;                         // (query row, head) columns per unit
constexpr int kSmemBudget = 192 * 1024;          // ring bytes per CTA
constexpr uint64_t kWaitTimeoutNs = 2000000000;  // 2 s: a TMA never takes this long

struct PlanParams {
  const int32_t *seq_lens;
  const int32_t *query_start_loc;
  int32_t num_seqs;
  int32_t total_q;
  int32_t max_query_len;
  int32_t max_seq_len;
  int32_t max_blocks_per_seq;
  int32_t block_size;     // tokens per cache block: 8, 16 or 32
  int32_t rows_per_item;  // 8 / G
  int32_t part_tokens;
  int32_t max_items;
  int32_t *class_start;   // [4][num_seqs + 1] prefix sums: 3 size classes of decode items, then tiles
  int32_t *nparts;        // [num_seqs], 0 = request produces nothing
  int4 *items;            // [2 * max_items]
  int32_t *item_count;    // [1]
  int32_t *work_counter;  // [1], zeroed here, consumed by the attention kernel
  int4 *tiles;            // [2 * max_tiles] prefill-tile records
  int32_t *tile_count;    // [1]
  int32_t *tile_counter;  // [1], zeroed here, consumed by the tile kernel
  int32_t max_tiles;
  int32_t tile_pos;       // query positions per tile: prefill_tile_rows(D) / G
  unsigned int *status;
};

struct AttnParams {
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
  const int4 *items;
  const int32_t *item_count;
  int32_t *work_counter;
  int32_t num_seqs;
  int32_t total_q;
  int32_t max_items;
  int32_t max_parts;
  float *part_o;    // [num_seqs][Hkv][max_parts][8][D]
  float *part_lse;  // [num_seqs][Hkv][max_parts][8]
  int32_t block_boxes;  // 1: 16-bit caches, head_dim 128, blocks of >= 16 tokens: one 4-D box per tile
  int32_t tiles_follow; // 1: the prefill-tile kernel is launched after this one
  unsigned int *status;
};



// ---------------------------------------------------------------------------
// Planning: per request, validate the lengths, count work items, scan, and
// write one 32-byte record per item. One CTA; no host synchronisation needed.
// Items are grouped by size so that the attention kernel's dynamic queue
// hands out the long ones first: class 0 = more keys than a partition,
// class 1 = exactly a partition, class 2 = fewer.
// Record: {b, first query token, rows, position of first row},
//         {key begin, key end, partition (-1 = whole range), partitions of the request}.
// ---------------------------------------------------------------------------
// A request whose query rows fit one column group (query_len <= 8 / G: decode
// tokens, speculative drafts) becomes split-KV decode items; a longer one
// (a chunked-prefill chunk) becomes tensor-core tiles of prefill_tile_rows / G
// positions.
// Returns the number of decode items; *ntiles receives the number of tiles.
__device__ __forceinline__ int request_shape(const PlanParams &p, int b, int &q0, int &ql, int &L, int &np,
                                             int &ntiles) {
  ntiles = 0;
  q0 = ld_cg(p.query_start_loc + b);
  const int q1 = ld_cg(p.query_start_loc + b + 1);
  L = ld_cg(p.seq_lens + b);
  ql = q1 - q0;
  np = 0;
  if (q0 < 0 || ql < 0 || q1 > p.total_q || (b == 0 && q0 != 0)) {
    flag_error(p.status, PA_FLAG_QUERY_LOC);
    return 0;
  }
  if (b == p.num_seqs - 1 && q1 != p.total_q) flag_error(p.status, PA_FLAG_QUERY_LOC);
  if (L < ql || L > p.max_seq_len || ql > p.max_query_len ||
      static_cast<int64_t>(L) > static_cast<int64_t>(p.max_blocks_per_seq) * p.block_size) {
    flag_error(p.status, PA_FLAG_LENGTHS);
    return 0;
  }
  if (ql == 0) return 0;
  if (ql > p.rows_per_item) {
    np = 1;
    ntiles = (ql + p.tile_pos - 1) / p.tile_pos;
    return 0;
  }
  np = max(1, (L + p.part_tokens - 1) / p.part_tokens);
  return np;
}

__device__ __forceinline__ void write_tile(const PlanParams &p, int idx, int b, int q0, int ql, int L, int t) {
  const int r0 = t * p.tile_pos;
  const int npos = min(p.tile_pos, ql - r0);
  const int pos0 = (L - ql) + r0;
  p.tiles[2 * idx] = make_int4(b, q0 + r0, npos, pos0);
  p.tiles[2 * idx + 1] = make_int4(0, pos0 + npos, -1, 1);
}

// Keys [kb, ke) of item k of a request, and its record fields.
struct ItemShape {
  int r0, rows, pos0, kb, ke, part;
};
__device__ __forceinline__ ItemShape item_shape(const PlanParams &p, int k, int np, int ql, int L) {
  ItemShape s;
  const int g = k / np, part = k - g * np;
  s.r0 = g * p.rows_per_item;
  s.rows = min(p.rows_per_item, ql - s.r0);
  s.pos0 = (L - ql) + s.r0;
  s.kb = 0;
  s.ke = s.pos0 + s.rows;  // the group's last row sees keys < pos0 + rows
  s.part = -1;
  if (np > 1) {
    s.kb = part * p.part_tokens;
    s.ke = min(L, s.kb + p.part_tokens);
    s.part = part;
  }
  return s;
}
__device__ __forceinline__ int size_class(int len, int part_tokens) {
  return len > part_tokens ? 0 : (len == part_tokens ? 1 : 2);
}

// Exclusive scan of one int per thread over the 1024-thread block; the block
// total goes to *total.
__device__ __forceinline__ int block_exclusive_scan(int v, int *warp_tot, int *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int t = warp_tot[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += u;
    }
    warp_tot[lane] = t;
  }
  __syncthreads();
  const int excl = (warp > 0 ? warp_tot[warp - 1] : 0) + incl - v;
  *total = warp_tot[31];
  __syncthreads();
  return excl;
}

// Exclusive block scan of a 64-bit value (four 16-bit counters packed).
__device__ __forceinline__ unsigned long long block_exclusive_scan64(unsigned long long v,
                                                                    unsigned long long *warp_tot,
                                                                    unsigned long long *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    unsigned long long t = warp_tot[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long u = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += u;
    }
    warp_tot[lane] = t;
  }
  __syncthreads();
  const unsigned long long excl = (warp > 0 ? warp_tot[warp - 1] : 0ull) + incl - v;
  *total = warp_tot[31];
  return excl;
}

constexpr int kPackBits = 16;  // four counters (3 item classes, tiles) below 2^16 in the one-pass planner
constexpr unsigned long long kPackMask = (1ull << kPackBits) - 1;

// One pass for batches of at most 1024 requests (one per thread): count the
// items of each size class, scan the three counts at once, write records.
__device__ __forceinline__ void plan_one_pass(const PlanParams &p) {
  __shared__ unsigned long long warp_tot[32];
  const int b = threadIdx.x;
  int q0 = 0, ql = 0, L = 0, np = 0, n = 0, nt = 0;
  unsigned long long packed = 0;
  if (b < p.num_seqs) {
    n = request_shape(p, b, q0, ql, L, np, nt);
    p.nparts[b] = np;
    packed += static_cast<unsigned long long>(nt) << (3 * kPackBits);
    for (int k = 0; k < n; ++k) {
      const ItemShape s = item_shape(p, k, np, ql, L);
      packed += 1ull << (kPackBits * size_class(s.ke - s.kb, p.part_tokens));
    }
  }
  unsigned long long total;
  const unsigned long long excl = block_exclusive_scan64(packed, warp_tot, &total);
  const int t0 = static_cast<int>(total & kPackMask), t1 = static_cast<int>((total >> kPackBits) & kPackMask);
  const int t2 = static_cast<int>((total >> (2 * kPackBits)) & kPackMask);
  const int t3 = static_cast<int>((total >> (3 * kPackBits)) & kPackMask);
  if (threadIdx.x == 0) {
    int all = t0 + t1 + t2;
    if (all > p.max_items) {
      flag_error(p.status, PA_FLAG_LENGTHS);
      all = p.max_items;
    }
    p.item_count[0] = all;
    p.tile_count[0] = min(t3, p.max_tiles);
  }
  const int tile0 = static_cast<int>((excl >> (3 * kPackBits)) & kPackMask);
  for (int t = 0; t < nt; ++t)  // a request's last tiles see the most keys: queue them first
    if (tile0 + t < p.max_tiles) write_tile(p, tile0 + t, b, q0, ql, L, nt - 1 - t);
  if (n == 0) return;
  int next[3] = {static_cast<int>(excl & kPackMask), t0 + static_cast<int>((excl >> kPackBits) & kPackMask),
                 t0 + t1 + static_cast<int>((excl >> (2 * kPackBits)) & kPackMask)};
  for (int k = 0; k < n; ++k) {
    const ItemShape s = item_shape(p, k, np, ql, L);
    const int idx = next[size_class(s.ke - s.kb, p.part_tokens)]++;
    if (idx < 0 || idx >= p.max_items) continue;
    p.items[2 * idx] = make_int4(b, q0 + s.r0, s.rows, s.pos0);
    p.items[2 * idx + 1] = make_int4(s.kb, s.ke, s.part, np);
  }
}

__global__ void __launch_bounds__(1024) plan_kernel(const PlanParams p) {
  __shared__ int warp_tot[32];
  __shared__ int carry[4];
  const int tid = threadIdx.x;
  const int stride = p.num_seqs + 1;
  griddep_wait();  // inputs may come from the previous kernel of the stream
  griddep_launch_dependents();
  if (tid == 0) {
    p.work_counter[0] = 0;
    p.tile_counter[0] = 0;
  }
  if (p.num_seqs <= 1024 && p.max_items < static_cast<int>(kPackMask) && p.max_tiles < static_cast<int>(kPackMask)) {
    plan_one_pass(p);
    return;
  }
  // larger batches: chunked counting and scans, then a second pass that writes
  if (tid < 4) carry[tid] = 0;
  __syncthreads();
  for (int base = 0; base < p.num_seqs; base += 1024) {
    const int b = base + tid;
    int cnt[4] = {0, 0, 0, 0};
    if (b < p.num_seqs) {
      int q0, ql, L, np, nt;
      const int n = request_shape(p, b, q0, ql, L, np, nt);
      p.nparts[b] = np;
      for (int k = 0; k < n; ++k) {
        const ItemShape s = item_shape(p, k, np, ql, L);
        ++cnt[size_class(s.ke - s.kb, p.part_tokens)];
      }
      cnt[3] = nt;
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      int tot;
      const int excl = block_exclusive_scan(cnt[c], warp_tot, &tot);
      if (b < p.num_seqs) p.class_start[c * stride + b] = carry[c] + excl;
      __syncthreads();
      if (tid == 0) carry[c] += tot;
      __syncthreads();
    }
  }
  if (tid < 4) p.class_start[tid * stride + p.num_seqs] = carry[tid];
  if (tid == 0) {
    int total = carry[0] + carry[1] + carry[2];
    if (total > p.max_items) {
      flag_error(p.status, PA_FLAG_LENGTHS);
      total = p.max_items;
    }
    p.item_count[0] = total;
    p.tile_count[0] = min(carry[3], p.max_tiles);
  }
  __syncthreads();
  const int base1 = carry[0], base2 = carry[0] + carry[1];
  for (int b = tid; b < p.num_seqs; b += 1024) {
    const int np = p.nparts[b];
    if (np == 0) continue;
    const int q0 = ld_cg(p.query_start_loc + b);
    const int ql = ld_cg(p.query_start_loc + b + 1) - q0;
    const int L = ld_cg(p.seq_lens + b);
    if (ql > p.rows_per_item) {
      const int nt = (ql + p.tile_pos - 1) / p.tile_pos;
      const int tile0 = p.class_start[3 * stride + b];
      for (int t = 0; t < nt; ++t)
        if (tile0 + t >= 0 && tile0 + t < p.max_tiles) write_tile(p, tile0 + t, b, q0, ql, L, nt - 1 - t);
      continue;
    }
    int next[3] = {p.class_start[b], base1 + p.class_start[stride + b], base2 + p.class_start[2 * stride + b]};
    const int n = np;
    for (int k = 0; k < n; ++k) {
      const ItemShape s = item_shape(p, k, np, ql, L);
      const int idx = next[size_class(s.ke - s.kb, p.part_tokens)]++;
      if (idx < 0 || idx >= p.max_items) continue;
      p.items[2 * idx] = make_int4(b, q0 + s.r0, s.rows, s.pos0);
      p.items[2 * idx + 1] = make_int4(s.kb, s.ke, s.part, np);
    }
  }
}

struct Unit {
  int valid, skip, b, row0, nrows, pos0, kv_begin, kv_end, part, nparts, kvh, kb0, kb1;
};

// ---------------------------------------------------------------------------
// Log-sum-exp merge of the partitions of split requests, after the attention
// kernel (PDL: launched early, waits for it). One CTA per (request, KV
// head): four warps, warp w merging columns w and w + 4 (a decode request's
// G columns are the first G, one warp each), or eight warps, one per
// column, when the pairs fit one wave of such CTAs. The request's partition
// count and query rows are loaded together, then each lane reads its D/32
// outputs of the partitions eight at a time with independent loads, keeping
// a running maximum so one pass suffices. Partitions are summed in order.
// (Eight warps for every pair hold 60 registers x 256 threads: four CTAs
// per SM, 3.4 waves at batch 256 x 8 KV heads.)
// ---------------------------------------------------------------------------
struct MergeParams {
  const int32_t *query_start_loc;
  const int32_t *nparts;
  int32_t num_seqs;
  int32_t num_kv_heads;
  int32_t num_heads;
  int32_t max_parts;
  const float *part_o;
  const float *part_lse;
  bf16 *out;
};

// NW warps per CTA (columns w, w + NW, ...): four when the (request, KV
// head) pairs are many (more CTAs per SM), eight when they fit one wave of
// eight-warp CTAs (the columns in parallel).
template <int D, int G, typename E, int NW>
__global__ void __launch_bounds__(NW * 32, (D > 128 ? 4 : 8) * 4 / NW) lse_merge_kernel(const MergeParams p) {
  // outputs per lane: 8 (D=256), 4 (D=128), 2 (D=64), else ceil(D / 32) consecutive
  // elements with the lane's last ones past D unused (D = 80, 96)
  constexpr int EPL = (D + 31) / 32;
  constexpr bool VEC = D % 64 == 0;
  griddep_wait();
  const int b = blockIdx.x / p.num_kv_heads, kvh = blockIdx.x - b * p.num_kv_heads;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // independent loads, one round trip
  const int np = ld_cg(p.nparts + b);
  const int q0 = ld_cg(p.query_start_loc + b);
  const int ql = ld_cg(p.query_start_loc + b + 1) - q0;
  if (np <= 1 || np > p.max_parts) return;
#pragma unroll 1
  for (int col = warp; col < kCols; col += NW) {
    const int qi = col / G, g = col % G;
    if (qi >= ql) break;  // columns run over query rows in order
    const int64_t base = (static_cast<int64_t>(b) * p.num_kv_heads + kvh) * p.max_parts * kCols + col;
    // one pass with a running maximum (every lane holds the same values)
    float M = -INFINITY;
    float acc[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
    float wsum = 0.f;
    for (int k0 = 0; k0 < np; k0 += 8) {
      float lv[8], ov[8][EPL];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int k = min(k0 + j, np - 1);
        lv[j] = ld_cg(p.part_lse + base + k * kCols);
        const float *src = p.part_o + (base + k * kCols) * D + lane * EPL;
        if constexpr (!VEC) {
#pragma unroll
          for (int e = 0; e < EPL; ++e) ov[j][e] = lane * EPL + e < D ? ld_cg(src + e) : 0.f;
        } else if constexpr (EPL >= 4) {
#pragma unroll
          for (int e = 0; e < EPL; e += 4) {
            const float4 v = ld_cg(reinterpret_cast<const float4 *>(src + e));
            ov[j][e] = v.x;
            ov[j][e + 1] = v.y;
            ov[j][e + 2] = v.z;
            ov[j][e + 3] = v.w;
          }
        } else {
          const float2 v = ld_cg(reinterpret_cast<const float2 *>(src));
          ov[j][0] = v.x;
          ov[j][1] = v.y;
        }
      }
      float Mn = M;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (k0 + j < np) Mn = fmaxf(Mn, lv[j]);
      const float Ms = Mn == -INFINITY ? 0.f : Mn;
      const float r = ex2_approx(M - Ms);  // rescale what was summed so far (0 on the first pack)
      wsum *= r;
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[e] *= r;
      M = Mn;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (k0 + j < np) {
          const float w = ex2_approx(lv[j] - Ms);
          wsum += w;
#pragma unroll
          for (int e = 0; e < EPL; ++e) acc[e] += w * ov[j][e];
        }
      }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    bf16 *dst = p.out + static_cast<int64_t>(q0 + qi) * p.num_heads * D + static_cast<int64_t>(kvh * G + g) * D +
                lane * EPL;
    if constexpr (!VEC) {
#pragma unroll
      for (int e = 0; e < EPL; ++e)
        if (lane * EPL + e < D) {
          const uint32_t v = E::pack(acc[e] * inv, 0.f);
          *reinterpret_cast<unsigned short *>(dst + e) = static_cast<unsigned short>(v & 0xffffu);
        }
    } else if constexpr (EPL >= 4) {
#pragma unroll
      for (int e = 0; e < EPL; e += 4)
        *reinterpret_cast<uint2 *>(dst + e) =
            make_uint2(E::pack(acc[e] * inv, acc[e + 1] * inv), E::pack(acc[e + 2] * inv, acc[e + 3] * inv));
    } else {
      *reinterpret_cast<uint32_t *>(dst) = E::pack(acc[0] * inv, acc[1] * inv);
    }
  }
}

// ---------------------------------------------------------------------------
// Split-KV attention: one independent TMA pipeline per warp.
// ---------------------------------------------------------------------------
// KT: keys per ring tile (units start at multiples of it).
template <int KT>
__device__ __forceinline__ Unit fetch_unit(const AttnParams &p, int total_units, int lane) {
  int u = 0;
  if (lane == 0) u = atomicAdd(p.work_counter, 1);
  u = __shfl_sync(0xffffffffu, u, 0);
  Unit U;
  U.valid = u < total_units;
  if (!U.valid) return U;
  const int item = u / p.num_kv_heads;
  U.kvh = u - item * p.num_kv_heads;
  const int4 r0 = ld_cg(p.items + 2 * item);
  const int4 r1 = ld_cg(p.items + 2 * item + 1);
  U.b = r0.x;
  U.row0 = r0.y;
  U.nrows = r0.z;
  U.pos0 = r0.w;
  U.kv_begin = r1.x;
  U.kv_end = r1.y;
  U.part = r1.z;
  U.nparts = r1.w;
  // A record is trusted only inside the bounds the host passed; anything else
  // is recorded and the unit becomes empty (no loads, no stores).
  const bool sane = U.b >= 0 && U.b < p.num_seqs && U.nrows >= 1 && U.nrows <= kCols && U.row0 >= 0 &&
                    U.row0 + U.nrows <= p.total_q && U.kv_begin >= 0 && U.kv_begin % KT == 0 &&
                    U.kv_begin < U.kv_end &&
                    U.kv_end <= static_cast<int64_t>(p.max_blocks_per_seq) * p.block_size &&
                    U.part < p.max_parts && U.nparts >= 1 && U.nparts <= p.max_parts;
  if (!sane) {
    if (lane == 0) flag_error(p.status, PA_FLAG_LENGTHS);
    U.skip = 1;
    U.kv_begin = U.kv_end = 0;
  } else {
    U.skip = 0;
  }
  U.kb0 = U.kv_begin / KT;
  U.kb1 = (U.kv_end + KT - 1) / KT;
  return U;
}

template <int D, bool KV8>
struct TileGeom;
// 16-bit caches: a 16-key tile is D / 64 boxes of 16 rows x 128 bytes (128-byte swizzle).
// head_dim 80 or 96: rows padded to whole atoms; the box columns past
// head_dim lie outside the tensor, so TMA fills them with zeros (no HBM read).
template <int D>
struct TileGeom<D, false> {
  static constexpr int HALVES = (D + 63) / 64;         // 64-element (128-byte) swizzle atoms per row
  static constexpr int HALF_BYTES = kTileKeys * 128;  // 16 rows x 128 B
  static constexpr int TILE_BYTES = HALVES * HALF_BYTES;
  static constexpr int SLOT_BYTES = 2 * TILE_BYTES;  // K tile then V tile
  // Byte offset of 16-byte chunk c (of D/8) of row r in a TMA SW128 tile.
  static __device__ __forceinline__ uint32_t off(int r, int c) {
    return (c >> 3) * HALF_BYTES + r * 128 + (((c & 7) ^ (r & 7)) << 4);
  }
};
// 8-bit caches: a ring tile is 32 keys (half the bytes of a 16-bit key, so
// the per-tile bookkeeping is paid per 32 keys), rows of D codes with 128-byte
// swizzle at D = 128 (16-byte chunk c of row r at c ^ (r % 8)) and 64-byte
// swizzle at D = 64 (chunk c of row r at c ^ (r / 2 % 4)); either way eight
// consecutive rows read at one chunk hit eight different bank groups, and
// rows 16..31 have the layout of rows 0..15 shifted by 16 * ROW bytes.
constexpr int kTileKeys8 = 32;
// head_dim 256: rows of two 128-code atoms, stored atom after atom (32 rows x
// 128 bytes each), so chunk c of row r sits in atom c / 8.
template <int D>
struct TileGeom<D, true> {
  static_assert(D <= 256, "head dims up to 256");
  static constexpr int ROW = D <= 64 ? 64 : 128;  // row bytes per atom (head_dim 80, 96: padded, zero-filled by TMA)
  static constexpr int ATOMS = D > 128 ? D / 128 : 1;
  static constexpr int ATOM_BYTES = kTileKeys8 * ROW;
  static constexpr int TILE_BYTES = ATOMS * ATOM_BYTES;
  static constexpr int SLOT_BYTES = 2 * TILE_BYTES;
  static __device__ __forceinline__ uint32_t off(int r, int c) {
    const uint32_t in_atom = ROW == 128 ? r * 128 + (((c ^ r) & 7) << 4) : r * 64 + (((c ^ (r >> 1)) & 3) << 4);
    return ATOMS == 1 ? in_atom : (c >> 3) * ATOM_BYTES + in_atom;  // one atom: no atom term at all
  }
};

template <int D, int G, int NWARPS, typename E, bool KV8>
__global__ void __launch_bounds__(NWARPS * 32, 1)
    splitkv_attention_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                             const __grid_constant__ CUtensorMap kmap4, const __grid_constant__ CUtensorMap vmap4,
                             const AttnParams p) {
  using T = TileGeom<D, KV8>;
  // Tensor-core operand type: E, except over 8-bit caches, where K, V and P
  // are fp16 whatever q is (E4M3 widens to fp16 in one hardware conversion)
  // and a bf16 q is converted to fp16 exactly (see the unit set-up).
  using M = typename std::conditional<KV8, ElemFp16, E>::type;
  constexpr int KT = KV8 ? kTileKeys8 : kTileKeys;            // keys per ring tile
  constexpr int S = kSmemBudget / (NWARPS * T::SLOT_BYTES);  // ring slots per warp
  static_assert(S >= 2, "ring needs at least two slots");
  constexpr int MT = D / 16;  // k steps of S, m tiles of O
  // 8-bit caches: an ldmatrix.x4 covers 32 d, so fragments come in pairs; a
  // head_dim of 80 computes one more (all-zero) k step and m tile
  constexpr int MQ = KV8 ? 2 * ((D + 31) / 32) : MT;

  extern __shared__ unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t bars[NWARPS][S];
  const uint32_t ring = (smem_u32(smem_raw) + 1023u) & ~1023u;

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x < NWARPS * S) mbar_init(smem_u32(&bars[0][0] + threadIdx.x), 1);
  if (threadIdx.x == 0) {
    prefetch_tmap(&kmap);
    prefetch_tmap(&vmap);
    if (p.block_boxes) {
      prefetch_tmap(&kmap4);
      prefetch_tmap(&vmap4);
    }
  }
  fence_mbar_init();
  __syncthreads();
  griddep_wait();  // the plan (and the cache scatter before it) must be complete
  // When prefill tiles follow, they may be scheduled from now on: tile CTAs
  // take over SMs as this kernel's CTAs exit, and read only what the kernels
  // before this one wrote. (A merge kernel that follows directly is left to
  // start after this kernel: resident early, its CTAs slowed the step.)
  if (p.tiles_follow) griddep_launch_dependents();

  const int Hkv = p.num_kv_heads;
  const int total_units = min(max(ld_cg(p.item_count), 0), p.max_items) * Hkv;
  const uint32_t my_ring = ring + warp * S * T::SLOT_BYTES;

  // Producer side (lane 0 issues): stage KT-key tile kb of unit U into ring
  // slot seq % S. Keys k live in cache row table[k / bs] * bs + k % bs: a
  // tile is KT / box_rows boxes of box_rows = min(bs, KT) consecutive rows of
  // one block each (16-bit caches: 16-key tiles; 8-bit: 32-key tiles). A
  // block-table entry is read only for a block that holds a key below the
  // unit's end; boxes past it are read at a negative row (zero fill).
  auto issue = [&](const Unit &U, int kb, uint32_t seq) {
    if (lane == 0) {
      const uint32_t slot = seq % S;
      const uint32_t bar = smem_u32(&bars[warp][slot]);
      const uint32_t dst = my_ring + slot * T::SLOT_BYTES;
      const int32_t *trow = p.block_tables + static_cast<int64_t>(U.b) * p.max_blocks_per_seq;
      const int bs = p.block_size;
      const int box_rows = bs < KT ? bs : KT;
      const int nbox = KT / box_rows;
      mbar_arrive_expect_tx(bar, T::SLOT_BYTES);
      for (int j = 0; j < nbox; ++j) {
        const int key = kb * KT + j * box_rows;  // first key of this box
        int z = -box_rows;                              // entirely outside the tensor: TMA fills zeros
        if (key < U.kv_end) {  // block sizes are powers of two: shift and mask
          const int phys = __ldg(trow + (key >> p.block_shift));
          if (phys < 0 || phys >= p.num_blocks)
            flag_error(p.status, PA_FLAG_BLOCK_RANGE);
          else
            z = (phys << p.block_shift) + (key & (bs - 1));
        }
        if constexpr (KV8) {
#pragma unroll
          for (int a = 0; a < T::ATOMS; ++a) {
            tma_load_3d(dst + a * T::ATOM_BYTES + j * box_rows * T::ROW, &kmap, bar, a * 128, U.kvh, z);
            tma_load_3d(dst + T::TILE_BYTES + a * T::ATOM_BYTES + j * box_rows * T::ROW, &vmap, bar, a * 128,
                        U.kvh, z);
          }
        } else if (D == 128 && p.block_boxes) {
          // one box per cache holds both 64-element atoms of the tile's 16 rows,
          // atom after atom: the layout T::off addresses (one TMA instruction
          // instead of two; the engine moves larger boxes at a higher rate)
          tma_load_4d(dst, &kmap4, bar, 0, z, 0, U.kvh);
          tma_load_4d(dst + T::TILE_BYTES, &vmap4, bar, 0, z, 0, U.kvh);
        } else {
#pragma unroll
          for (int h = 0; h < T::HALVES; ++h) {
            tma_load_3d(dst + h * T::HALF_BYTES + j * box_rows * 128, &kmap, bar, h * 64, U.kvh, z);
            tma_load_3d(dst + T::TILE_BYTES + h * T::HALF_BYTES + j * box_rows * 128, &vmap, bar, h * 64, U.kvh,
                        z);
          }
        }
      }
    }
  };

  Unit cur = fetch_unit<KT>(p, total_units, lane);
  Unit nxt;
  nxt.valid = 0;
  bool have_nxt = false;
  int p_unit = 0;  // which unit the producer is issuing: 0 = cur, 1 = nxt
  int p_kb = cur.kb0;
  uint32_t issued = 0, consumed = 0;

  // Issue blocks in stream order (cur's, then nxt's) while fewer than `limit` are issued.
  auto produce = [&](uint32_t limit) {
    while (issued < limit) {
      if (p_unit == 0) {
        if (!cur.valid) break;
        if (p_kb < cur.kb1) {
          issue(cur, p_kb++, issued++);
          continue;
        }
        if (!have_nxt) {
          nxt = fetch_unit<KT>(p, total_units, lane);
          have_nxt = true;
        }
        p_unit = 1;
        p_kb = nxt.kb0;
        continue;
      }
      if (nxt.valid && p_kb < nxt.kb1) {
        issue(nxt, p_kb++, issued++);
        continue;
      }
      break;  // the producer runs at most one unit ahead
    }
  };

  const int arow = (lane & 7) + ((lane >> 3) & 1) * 8;  // ldmatrix row for K (A operand)
  const int vrow = (lane & 7) + (lane >> 4) * 8;        // ldmatrix row for V (transposed A)

  while (cur.valid) {
    // ---- per-unit set-up: q fragments (B operand of S^T = K Q^T), causal limits ----
    uint32_t qf[MQ][2];
    float col_scale[2] = {p.scale_log2, p.scale_log2};  // log2-domain score factor of accumulator columns
    {
      const int n = lane >> 2, qi = n / G, g = n % G;
      const bool ok = qi < cur.nrows;
      const bf16 *qp = p.q + static_cast<int64_t>(cur.row0 + (ok ? qi : 0)) * p.q_stride +
                       static_cast<int64_t>(cur.kvh * G + g) * D;
      if constexpr (KV8) {
        // k step kk pairs d = 16kk + 4(lane % 4) + (0, 2) and (1, 3): the order
        // in which the 8-bit K fragments below hold d
        qp += 4 * (lane & 3);
#pragma unroll
        for (int kk = 0; kk < MQ; ++kk) {
          const bool in = ok && kk < MT;  // k steps past head_dim multiply zero-filled codes: q is 0 there
          const uint32_t x = in ? __ldg(reinterpret_cast<const uint32_t *>(qp + 16 * kk)) : 0u;
          const uint32_t y = in ? __ldg(reinterpret_cast<const uint32_t *>(qp + 16 * kk + 2)) : 0u;
          qf[kk][0] = __byte_perm(x, y, 0x5410);
          qf[kk][1] = __byte_perm(x, y, 0x7632);
        }
        if constexpr (std::is_same<E, ElemBf16>::value) {
          // bf16 -> fp16, exactly: a column (lanes 4n..4n+3 hold column n)
          // whose largest |q| reaches 2^15 is first scaled by 2^-e so that it
          // lies in [2^14, 2^15); its scores are scaled back by 2^e below.
          // Every bf16 value of at least 2^-17 times the column's scale then
          // converts exactly (fp16 keeps 11 significant bits, bf16 has 8).
          float amax = 0.f;
#pragma unroll
          for (int kk = 0; kk < MQ; ++kk)
#pragma unroll
            for (int h = 0; h < 2; ++h)
              amax = fmaxf(amax, fmaxf(fabsf(ElemBf16::lo(qf[kk][h])), fabsf(ElemBf16::hi(qf[kk][h]))));
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
          const int ex = static_cast<int>((__float_as_uint(amax) >> 23) & 0xffu) - 127;  // floor(log2(amax))
          const int e = ex >= 15 ? min(ex - 14, 120) : 0;
          const float f = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);  // 2^-e
#pragma unroll
          for (int kk = 0; kk < MQ; ++kk)
#pragma unroll
            for (int h = 0; h < 2; ++h)
              qf[kk][h] = ElemFp16::pack(ElemBf16::lo(qf[kk][h]) * f, ElemBf16::hi(qf[kk][h]) * f);
          // accumulator column c = 2(lane % 4) + j is B-fragment column c, held by lane 4c
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int ec = __shfl_sync(0xffffffffu, e, 4 * (2 * (lane & 3) + j));
            col_scale[j] = p.scale_log2 * __uint_as_float(static_cast<uint32_t>(127 + ec) << 23);
          }
        }
      } else {
        qp += 2 * (lane & 3);
#pragma unroll
        for (int kk = 0; kk < MT; ++kk) {
          qf[kk][0] = ok ? __ldg(reinterpret_cast<const uint32_t *>(qp + 16 * kk)) : 0u;
          qf[kk][1] = ok ? __ldg(reinterpret_cast<const uint32_t *>(qp + 16 * kk + 8)) : 0u;
        }
      }
    }
    int lim[2];  // keys j < lim[e] are visible to accumulator column 2*(lane%4)+e
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int qi = (2 * (lane & 3) + e) / G;
      lim[e] = qi < cur.nrows ? min(cur.pos0 + qi + 1, cur.kv_end) : cur.kv_begin;
    }
    float o[MQ][4];
#pragma unroll
    for (int mt = 0; mt < MQ; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    float m[2] = {-INFINITY, -INFINITY};
    float l[2] = {0.f, 0.f};

    // Rows past the request's last key may hold anything (even NaN): zero them in V.
    auto zero_tail = [&](uint32_t vt, int valid_rows) {
      constexpr int CPR = KV8 ? D / 16 : D / 8;  // 16-byte chunks per row
      const int n = (KT - valid_rows) * CPR;
      for (int i = lane; i < n; i += 32) {
        const int r = valid_rows + i / CPR, c = i % CPR;
        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};\n" ::"r"(vt + T::off(r, c)), "r"(0u) : "memory");
      }
      fence_proxy_async_smem();  // order these generic writes before the slot's next TMA fill
      __syncwarp();
    };
    // S^T = K Q^T of one 16-key tile over D (two independent accumulator chains), summed into s.
    auto scores = [&](uint32_t kt, float (&s)[4]) {
      float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
      if constexpr (KV8) {
        // one x4 load = 16 keys x 32 codes: per lane 4 consecutive d of keys
        // lane/4 and lane/4 + 8 in each of two 16-d chunks, widened exactly
        // into the A fragments of two k steps (d paired as q is above)
#pragma unroll
        for (int j = 0; j < MQ / 2; ++j) {
          uint32_t r0, r1, r2, r3, l0, h0, l1, h1;
          ldsm_x4(kt + T::off(arow, 2 * j + (lane >> 4)), r0, r1, r2, r3);
          M::from_e4m3x4(r0, l0, h0);
          M::from_e4m3x4(r1, l1, h1);
          M::mma(sa, l0, l1, h0, h1, qf[2 * j][0], qf[2 * j][1]);
          M::from_e4m3x4(r2, l0, h0);
          M::from_e4m3x4(r3, l1, h1);
          M::mma(sb, l0, l1, h0, h1, qf[2 * j + 1][0], qf[2 * j + 1][1]);
        }
      } else {
#pragma unroll
        for (int kk = 0; kk < MT; ++kk) {
          uint32_t a0, a1, a2, a3;
          ldsm_x4(kt + T::off(arow, 2 * kk + (lane >> 4)), a0, a1, a2, a3);
          if (kk & 1)
            M::mma(sb, a0, a1, a2, a3, qf[kk][0], qf[kk][1]);
          else
            M::mma(sa, a0, a1, a2, a3, qf[kk][0], qf[kk][1]);
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) s[i] = sa[i] + sb[i];
    };
    // O^T += V^T P^T of one tile; P^T (keys x columns) comes as hi (b0, b1) + lo (c0, c1).
    auto pv = [&](uint32_t vt, uint32_t b0, uint32_t b1, uint32_t c0, uint32_t c1) {
      if constexpr (KV8) {
        // transposed x4 load of 16 keys x 32 codes: per lane keys (2(lane%4),
        // +1) (+8) at d = 2(lane/4) and 2(lane/4) + 1 of each 16-d chunk. Row
        // lane/4 of m tile mt holds d = 16mt + 2(lane/4), row lane/4 + 8 holds
        // d = 16mt + 2(lane/4) + 1; the epilogue puts d back in order.
#pragma unroll
        for (int j = 0; j < MQ / 2; ++j) {
          uint32_t r0, r1, r2, r3, l0, h0, l1, h1;
          ldsm_x4_t(vt + T::off(arow, 2 * j + (lane >> 4)), r0, r1, r2, r3);
          M::from_e4m3x4(r0, l0, h0);
          M::from_e4m3x4(r1, l1, h1);
          M::mma(o[2 * j], l0, h0, l1, h1, b0, b1);
          M::mma(o[2 * j], l0, h0, l1, h1, c0, c1);
          M::from_e4m3x4(r2, l0, h0);
          M::from_e4m3x4(r3, l1, h1);
          M::mma(o[2 * j + 1], l0, h0, l1, h1, b0, b1);
          M::mma(o[2 * j + 1], l0, h0, l1, h1, c0, c1);
        }
      } else {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          uint32_t a0, a1, a2, a3;
          ldsm_x4_t(vt + T::off(vrow, 2 * mt + ((lane >> 3) & 1)), a0, a1, a2, a3);
          M::mma(o[mt], a0, a1, a2, a3, b0, b1);
          M::mma(o[mt], a0, a1, a2, a3, c0, c1);
        }
      }
    };

    // 32 keys per step: two 16-key tiles (one, at the end of an odd run) of a
    // 16-bit cache, or the two halves of one 32-key tile of an 8-bit cache.
    // One softmax update per step; O rescaled only when a column's maximum grew.
    for (int kb = cur.kb0; kb < cur.kb1; kb += KV8 ? 1 : 2) {
      const bool two = KV8 || kb + 1 < cur.kb1;  // warp-uniform
      produce(consumed + S);
      uint32_t kt0, vt0, kt1, vt1;
      bool landed;
      if constexpr (KV8) {
        const uint32_t slot = consumed % S;
        landed = mbar_wait_bounded(smem_u32(&bars[warp][slot]), (consumed / S) & 1u, kWaitTimeoutNs);
        kt0 = my_ring + slot * T::SLOT_BYTES;
        vt0 = kt0 + T::TILE_BYTES;
        kt1 = kt0 + kTileKeys * T::ROW;  // rows 16..31
        vt1 = vt0 + kTileKeys * T::ROW;
      } else {
        const uint32_t slot0 = consumed % S, slot1 = (consumed + 1) % S;
        landed = mbar_wait_bounded(smem_u32(&bars[warp][slot0]), (consumed / S) & 1u, kWaitTimeoutNs);
        if (two && landed)
          landed = mbar_wait_bounded(smem_u32(&bars[warp][slot1]), ((consumed + 1) / S) & 1u, kWaitTimeoutNs);
        kt0 = my_ring + slot0 * T::SLOT_BYTES;
        vt0 = kt0 + T::TILE_BYTES;
        kt1 = my_ring + slot1 * T::SLOT_BYTES;
        vt1 = kt1 + T::TILE_BYTES;
      }
      if (!__all_sync(0xffffffffu, landed)) {  // leave together, never with a diverged warp
        if (lane == 0) {
          flag_error(p.status, PA_FLAG_TIMEOUT);
          // Loads this warp issued into its ring may still be in flight: wait
          // for each of them (bounded) before the warp stops using its slots.
          for (uint32_t g = consumed; g < issued; ++g)
            (void)mbar_wait_bounded(smem_u32(&bars[warp][g % S]), (g / S) & 1u, kWaitTimeoutNs);
        }
        __syncwarp();
        return;
      }
      // only the unit's last tile can be partial
      const int last_valid = cur.kv_end - (cur.kb1 - 1) * KT;
      if constexpr (KV8) {
        if (last_valid < KT && kb == cur.kb1 - 1) zero_tail(vt0, last_valid);
      } else {
        if (last_valid < KT && kb + (two ? 1 : 0) == cur.kb1 - 1) zero_tail(two ? vt1 : vt0, last_valid);
      }

      float s0[4], s1[4];
      scores(kt0, s0);
      if (two) scores(kt1, s1);
      const int t0 = kb * KT + (lane >> 2), t1 = t0 + 8, t2 = t0 + kTileKeys, t3 = t1 + kTileKeys;
      const float x0 = t0 < lim[0] ? __fmul_rn(s0[0], col_scale[0]) : -INFINITY;
      const float x1 = t0 < lim[1] ? __fmul_rn(s0[1], col_scale[1]) : -INFINITY;
      const float x2 = t1 < lim[0] ? __fmul_rn(s0[2], col_scale[0]) : -INFINITY;
      const float x3 = t1 < lim[1] ? __fmul_rn(s0[3], col_scale[1]) : -INFINITY;
      const float y0 = two && t2 < lim[0] ? __fmul_rn(s1[0], col_scale[0]) : -INFINITY;
      const float y1 = two && t2 < lim[1] ? __fmul_rn(s1[1], col_scale[1]) : -INFINITY;
      const float y2 = two && t3 < lim[0] ? __fmul_rn(s1[2], col_scale[0]) : -INFINITY;
      const float y3 = two && t3 < lim[1] ? __fmul_rn(s1[3], col_scale[1]) : -INFINITY;
      // rounded products (never contracted into the subtractions below), so the
      // maximum's exponent is exactly zero whatever the magnitude of the scores
      float mx0 = fmaxf(fmaxf(x0, x2), fmaxf(y0, y2)), mx1 = fmaxf(fmaxf(x1, x3), fmaxf(y1, y3));
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
      }
      const float mn0 = fmaxf(m[0], mx0), mn1 = fmaxf(m[1], mx1);
      const float ms0 = mn0 == -INFINITY ? 0.f : mn0;
      const float ms1 = mn1 == -INFINITY ? 0.f : mn1;
      const float al0 = ex2_approx(m[0] - ms0), al1 = ex2_approx(m[1] - ms1);
      const float p0 = ex2_approx(x0 - ms0), p1 = ex2_approx(x1 - ms1);
      const float p2 = ex2_approx(x2 - ms0), p3 = ex2_approx(x3 - ms1);
      const float q0 = ex2_approx(y0 - ms0), q1 = ex2_approx(y1 - ms1);
      const float q2 = ex2_approx(y2 - ms0), q3 = ex2_approx(y3 - ms1);
      l[0] = l[0] * al0 + ((p0 + p2) + (q0 + q2));
      l[1] = l[1] * al1 + ((p1 + p3) + (q1 + q3));
      m[0] = mn0;
      m[1] = mn1;
      if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
        for (int mt = 0; mt < MQ; ++mt) {
          o[mt][0] *= al0;
          o[mt][1] *= al1;
          o[mt][2] *= al0;
          o[mt][3] *= al1;
        }
      }
      // P^T (keys x columns) -> B operand by transposition; P as hi + lo pairs.
      {
        const uint32_t h01 = M::pack(p0, p1), h23 = M::pack(p2, p3);
        const uint32_t l01 = M::pack(p0 - M::lo(h01), p1 - M::hi(h01));
        const uint32_t l23 = M::pack(p2 - M::lo(h23), p3 - M::hi(h23));
        pv(vt0, movmatrix_t(h01), movmatrix_t(h23), movmatrix_t(l01), movmatrix_t(l23));
      }
      if (two) {
        const uint32_t h01 = M::pack(q0, q1), h23 = M::pack(q2, q3);
        const uint32_t l01 = M::pack(q0 - M::lo(h01), q1 - M::hi(h01));
        const uint32_t l23 = M::pack(q2 - M::lo(h23), q3 - M::hi(h23));
        pv(vt1, movmatrix_t(h01), movmatrix_t(h23), movmatrix_t(l01), movmatrix_t(l23));
      }
      __syncwarp();  // every lane is done with these slots before they are refilled
      consumed += (KV8 || !two) ? 1 : 2;
    }

    // ---- unit epilogue: normalise and write the output or the partial ----
    if (!cur.skip) {
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        l[0] += __shfl_xor_sync(0xffffffffu, l[0], off);
        l[1] += __shfl_xor_sync(0xffffffffu, l[1], off);
      }
      const float inv0 = l[0] > 0.f ? p.out_scale / l[0] : 0.f;
      const float inv1 = l[1] > 0.f ? p.out_scale / l[1] : 0.f;
      if (cur.part < 0) {
        // transpose the bf16 result so each lane owns two consecutive d of one column
        const int col = lane >> 2, qi = col / G, g = col % G;
        bf16 *dst = p.out + static_cast<int64_t>(cur.row0 + (qi < cur.nrows ? qi : 0)) * p.num_heads * D +
                    static_cast<int64_t>(cur.kvh * G + g) * D;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const uint32_t lo8 = movmatrix_t(E::pack(o[mt][0] * inv0, o[mt][1] * inv1));
          const uint32_t hi8 = movmatrix_t(E::pack(o[mt][2] * inv0, o[mt][3] * inv1));
          if (qi < cur.nrows) {
            if constexpr (KV8) {
              // lo8 holds d = 16mt + 4(lane%4) + (0, 2), hi8 d + (1, 3)
              *reinterpret_cast<uint2 *>(dst + 16 * mt + 4 * (lane & 3)) =
                  make_uint2(__byte_perm(lo8, hi8, 0x5410), __byte_perm(lo8, hi8, 0x7632));
            } else {
              *reinterpret_cast<uint32_t *>(dst + 16 * mt + 2 * (lane & 3)) = lo8;
              *reinterpret_cast<uint32_t *>(dst + 16 * mt + 2 * (lane & 3) + 8) = hi8;
            }
          }
        }
      } else {
        const int64_t base = ((static_cast<int64_t>(cur.b) * Hkv + cur.kvh) * p.max_parts + cur.part) * kCols;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int col = 2 * (lane & 3) + e;
          if (col / G < cur.nrows) {
            const float inv = e ? inv1 : inv0;
            if constexpr (KV8) {
              float *dst = p.part_o + (base + col) * D + 2 * (lane >> 2);
#pragma unroll
              for (int mt = 0; mt < MT; ++mt)
                *reinterpret_cast<float2 *>(dst + 16 * mt) = make_float2(o[mt][e] * inv, o[mt][2 + e] * inv);
            } else {
              float *dst = p.part_o + (base + col) * D + (lane >> 2);
#pragma unroll
              for (int mt = 0; mt < MT; ++mt) {
                dst[16 * mt] = o[mt][e] * inv;
                dst[16 * mt + 8] = o[mt][2 + e] * inv;
              }
            }
            if (lane < 4) {
              const float lc = e ? l[1] : l[0], mc = e ? m[1] : m[0];
              p.part_lse[base + col] = lc > 0.f ? mc + __log2f(lc) : -INFINITY;
            }
          }
        }
      }
    }

    // ---- advance to the next unit (the producer may already be streaming it) ----
    if (p_unit == 0) {
      if (!have_nxt) {
        nxt = fetch_unit<KT>(p, total_units, lane);
        have_nxt = true;
      }
      p_kb = nxt.kb0;
    }
    cur = nxt;
    have_nxt = false;
    p_unit = 0;
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

// Keys per partition. Partitions bound the work of one unit, so that a few
// long requests cannot leave most SMs idle at the end of the step; each one
// costs a partial (D + 1 floats per column) written here and read back by
// the merge. With many (request, KV head) pairs against the decode kernel's
// warps (152 SMs x 8 warps for 16-bit caches, x 12 for 8-bit ones on GB300;
// fixed figures so that the host-only sizing calls need no device query)
// 512 keys balance best; with few pairs, about one partition of the longest
// request per warp, in multiples of 512 keys up to 2048, keeps every warp
// busy with fewer partials. Measured on GB300 (step time): batch 256 GQA and
// 64 MHA are fastest at 512; 8 requests of 32768 keys at 2048 (8 % faster
// than at 512) with 16-bit caches.
int partition_tokens(int32_t num_seqs, int32_t max_seq_len, int32_t num_kv_heads, bool kv8) {
  const int64_t kWarps = 152 * (kv8 ? 12 : 8);
  const int64_t pairs = static_cast<int64_t>(num_seqs) * num_kv_heads;
  if (pairs <= 0 || max_seq_len <= 0 || pairs * 2 >= kWarps) return 512;
  const int64_t per_warp = static_cast<int64_t>(max_seq_len) * pairs / kWarps;
  const int64_t p = (per_warp + 511) / 512 * 512;
  return static_cast<int>(p < 512 ? 512 : (p > 2048 ? 2048 : p));
}

static size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

bool workspace_layout(int32_t num_seqs, int32_t total_q, int32_t max_seq_len, int32_t num_heads,
                      int32_t num_kv_heads, int32_t head_dim, bool kv8, WorkspaceLayout &w) {
  if (num_seqs < 0 || total_q < 0 || max_seq_len < 0 || num_heads <= 0 || num_kv_heads <= 0 ||
      head_dim <= 0 || num_heads % num_kv_heads != 0)
    return false;
  const int G = num_heads / num_kv_heads;
  if (G > 8) return false;
  w.rows_per_item = 8 / G;
  w.part_tokens = partition_tokens(num_seqs, max_seq_len, num_kv_heads, kv8);
  w.max_parts = max_seq_len > 0 ? (max_seq_len + w.part_tokens - 1) / w.part_tokens : 1;
  const int64_t items = static_cast<int64_t>(num_seqs) * w.max_parts;  // decode items: one group per request
  const int tile_rows = prefill_tile_rows(head_dim);
  const int64_t tiles = (static_cast<int64_t>(total_q) * G + tile_rows - 1) / tile_rows + num_seqs;
  if (items * num_kv_heads > (1LL << 30) || tiles * num_kv_heads > (1LL << 30)) return false;
  w.max_items = static_cast<int32_t>(items > 0 ? items : 1);
  w.max_tiles = static_cast<int32_t>(tiles > 0 ? tiles : 1);
  const size_t nsplit = static_cast<size_t>(num_seqs) * num_kv_heads * w.max_parts * kCols;
  size_t off = 0;
  w.item_start = off; off += align256(sizeof(int32_t) * 4 * (static_cast<size_t>(num_seqs) + 1));
  w.nparts = off;     off += align256(sizeof(int32_t) * (static_cast<size_t>(num_seqs) + 1));
  w.item_count = off; off += align256(4 * sizeof(int32_t));  // items, work counter, tiles, tile counter
  w.items = off;      off += align256(sizeof(int4) * 2 * static_cast<size_t>(w.max_items));
  w.tiles = off;      off += align256(sizeof(int4) * 2 * static_cast<size_t>(w.max_tiles));
  w.part_lse = off;   off += align256(sizeof(float) * nsplit);
  w.part_o = off;     off += align256(sizeof(float) * nsplit * head_dim);
  w.total = off;
  return true;
}

// cuTensorMapEncodeTiled from the driver, found once through the runtime.
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, []() {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// 3-D view of one cache, [num_blocks * 16 rows][Hkv][D], with a box of
// 16 rows x 1 head x 64 elements (128 bytes, 128-byte swizzle).
// 8-bit caches: elements of one byte and a box of up to 32 rows x 1 head x D
// codes (128-byte swizzle at D = 128, 64-byte at D = 64).
static bool encode_cache_map(CUtensorMap *map, const void *cache, int64_t num_blocks, int32_t num_kv_heads,
                             int32_t head_dim, int32_t block_size, int32_t dtype, bool kv8) {
  auto encode = tensor_map_encoder();
  if (!encode) return false;
  const cuuint64_t esize = kv8 ? 1 : 2;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(num_kv_heads),
                              static_cast<cuuint64_t>(num_blocks) * block_size};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(head_dim) * esize,
                                 static_cast<cuuint64_t>(num_kv_heads) * head_dim * esize};
  // box rows: min(block_size, keys per tile), the tile being 16 keys (32 for 8-bit caches)
  const int kt = kv8 ? kTileKeys8 : kTileKeys;
  const cuuint32_t rows = static_cast<cuuint32_t>(block_size < kt ? block_size : kt);
  // 8-bit rows: one box of 64 or 128 codes (head_dim 80, 96: the columns past it are zero-filled)
  const cuuint32_t box[3] = {kv8 ? (head_dim <= 64 ? 64u : 128u) : 64u, 1, rows};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType type = kv8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                       : (dtype == PA_FP16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                           : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
  const CUtensorMapSwizzle swz =
      kv8 && head_dim <= 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
  return encode(map, type, 3, const_cast<void *>(cache), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 4-D view of one 16-bit cache at head_dim 128, [Hkv][2 atoms][num_blocks *
// block_size rows][64 elements] from the outermost dimension in (strides:
// head D * 2 bytes, atom 128 bytes, row Hkv * D * 2 bytes), with a box of
// `rows` rows x both atoms x 1 head: a whole (block, KV head) tile of up to
// 32 rows in one TMA instruction, landing atom after atom (128-byte swizzle).
// Every coordinate the kernels use lies inside the cache; a negative row
// coordinate reads zeros.
static bool encode_block_map(CUtensorMap *map, const void *cache, int64_t num_blocks, int32_t num_kv_heads,
                             int32_t block_size, int32_t rows, int32_t dtype) {
  auto encode = tensor_map_encoder();
  if (!encode) return false;
  constexpr int D = 128;
  const cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(num_blocks) * block_size, 2,
                              static_cast<cuuint64_t>(num_kv_heads)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(num_kv_heads) * D * 2, 128, D * 2};
  const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(rows), 2, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapDataType type =
      dtype == PA_FP16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  return encode(map, type, 4, const_cast<void *>(cache), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr int kAttnWarps = 8;   // 16-bit caches: two warps per scheduler
constexpr int kAttnWarps8 = 12; // 8-bit caches: three, to hide the latency of the per-tile widening
// head_dim 256: a ring slot (K and V of one tile) is 16 KB, so four warps of
// three slots fill the ring budget (192 KB in flight per SM, as at 128)
template <int D, bool KV8>
constexpr int decode_warps() {
  return D == 256 ? 4 : (KV8 ? kAttnWarps8 : kAttnWarps);
}

template <int D, int G, typename E, bool KV8>
static cudaError_t launch_typed(const AttnLaunch &a, const WorkspaceLayout &w, cudaStream_t stream,
                                int *launched) {
  char *ws = static_cast<char *>(a.workspace);
  PlanParams pp;
  pp.seq_lens = a.seq_lens;
  pp.query_start_loc = a.query_start_loc;
  pp.num_seqs = a.num_seqs;
  pp.total_q = a.total_q;
  pp.max_query_len = a.max_query_len;
  pp.max_seq_len = a.max_seq_len;
  pp.max_blocks_per_seq = a.max_blocks_per_seq;
  pp.block_size = a.block_size;
  pp.rows_per_item = w.rows_per_item;
  pp.part_tokens = w.part_tokens;
  pp.max_items = w.max_items;
  pp.class_start = reinterpret_cast<int32_t *>(ws + w.item_start);
  pp.nparts = reinterpret_cast<int32_t *>(ws + w.nparts);
  pp.items = reinterpret_cast<int4 *>(ws + w.items);
  pp.item_count = reinterpret_cast<int32_t *>(ws + w.item_count);
  pp.work_counter = pp.item_count + 1;
  pp.tile_count = pp.item_count + 2;
  pp.tile_counter = pp.item_count + 3;
  pp.tiles = reinterpret_cast<int4 *>(ws + w.tiles);
  pp.max_tiles = w.max_tiles;
  pp.tile_pos = prefill_tile_rows(D) / G;
  pp.status = a.status;

  CUtensorMap kmap, vmap;
  if (!encode_cache_map(&kmap, a.key_cache, a.num_blocks, a.num_kv_heads, D, a.block_size, a.dtype, KV8) ||
      !encode_cache_map(&vmap, a.value_cache, a.num_blocks, a.num_kv_heads, D, a.block_size, a.dtype, KV8))
    return cudaErrorInvalidValue;
  // whole-block boxes (16-bit caches at head_dim 128): 16-row tiles for the
  // decode kernel when blocks hold at least 16 tokens
  const bool block_boxes = !KV8 && D == 128 && a.block_size >= kTileKeys;
  CUtensorMap kmap4 = kmap, vmap4 = vmap;
  if (block_boxes &&
      (!encode_block_map(&kmap4, a.key_cache, a.num_blocks, a.num_kv_heads, a.block_size, kTileKeys, a.dtype) ||
       !encode_block_map(&vmap4, a.value_cache, a.num_blocks, a.num_kv_heads, a.block_size, kTileKeys, a.dtype)))
    return cudaErrorInvalidValue;

  cudaError_t err = launch_pdl(plan_kernel, dim3(1), dim3(1024), 0, stream, pp);
  if (err != cudaSuccess) return err;
  ++*launched;

  AttnParams ap;
  ap.q = static_cast<const bf16 *>(a.q);
  ap.q_stride = a.q_stride;
  ap.block_tables = a.block_tables;
  ap.max_blocks_per_seq = a.max_blocks_per_seq;
  ap.block_size = a.block_size;
  ap.block_shift = a.block_size == 8 ? 3 : (a.block_size == 16 ? 4 : 5);
  ap.num_heads = a.num_heads;
  ap.num_kv_heads = a.num_kv_heads;
  ap.num_blocks = a.num_blocks;
  ap.scale_log2 = (KV8 ? a.scale * a.k_scale : a.scale) * 1.4426950408889634f;
  ap.out_scale = KV8 ? a.v_scale : 1.0f;
  ap.out = static_cast<bf16 *>(a.out);
  ap.items = pp.items;
  ap.item_count = pp.item_count;
  ap.work_counter = pp.work_counter;
  ap.num_seqs = a.num_seqs;
  ap.total_q = a.total_q;
  ap.max_items = w.max_items;
  ap.max_parts = w.max_parts;
  ap.part_o = reinterpret_cast<float *>(ws + w.part_o);
  ap.part_lse = reinterpret_cast<float *>(ws + w.part_lse);
  ap.block_boxes = block_boxes ? 1 : 0;
  ap.tiles_follow = a.max_query_len > w.rows_per_item ? 1 : 0;
  ap.status = a.status;

  constexpr int smem = kSmemBudget + 1024;  // ring + alignment slack
  constexpr int NW = decode_warps<D, KV8>();
  auto kern = splitkv_attention_kernel<D, G, NW, E, KV8>;
  err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  err = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (err != cudaSuccess) return err;
  // one CTA per SM; fewer when there are fewer units than warps
  int64_t grid = a.sm_count;
  const int64_t units_upper = static_cast<int64_t>(w.max_items) * a.num_kv_heads;
  if (grid * NW > units_upper) grid = (units_upper + NW - 1) / NW;
  if (grid < 1) grid = 1;
  if (a.ev_start) cudaEventRecord(a.ev_start, stream);
  err = launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(NW * 32), smem, stream, kmap, vmap, kmap4, vmap4,
                   ap);
  if (err != cudaSuccess) return err;
  ++*launched;
  if (a.ev_stop) cudaEventRecord(a.ev_stop, stream);

  if (a.max_query_len > w.rows_per_item) {  // some request may be a prefill chunk
    TileParams tp;
    tp.q = ap.q;
    tp.q_stride = a.q_stride;
    tp.block_tables = a.block_tables;
    tp.max_blocks_per_seq = a.max_blocks_per_seq;
    tp.block_size = a.block_size;
    tp.block_shift = ap.block_shift;
    tp.num_heads = a.num_heads;
    tp.num_kv_heads = a.num_kv_heads;
    tp.num_blocks = a.num_blocks;
    tp.scale_log2 = ap.scale_log2;
    tp.out_scale = ap.out_scale;
    tp.out = ap.out;
    tp.tiles = pp.tiles;
    tp.tile_count = pp.tile_count;
    tp.tile_counter = pp.tile_counter;
    tp.num_seqs = a.num_seqs;
    tp.total_q = a.total_q;
    tp.max_tiles = w.max_tiles;
    tp.status = a.status;
    // value cache in whole-block boxes for the tile kernel (block_size rows)
    CUtensorMap vmapb = vmap;
    if (!KV8 && D == 128 &&
        !encode_block_map(&vmapb, a.value_cache, a.num_blocks, a.num_kv_heads, a.block_size, a.block_size, a.dtype))
      return cudaErrorInvalidValue;
    if (a.tile_start) cudaEventRecord(a.tile_start, stream);
    err = launch_prefill_tiles<D, G, E, KV8>(kmap, vmap, vmapb, tp, a.sm_count, stream);
    if (err == cudaSuccess && a.tile_stop) cudaEventRecord(a.tile_stop, stream);
    if (err != cudaSuccess) return err;
    ++*launched;
  }

  if (w.max_parts > 1) {
    MergeParams mp;
    mp.query_start_loc = a.query_start_loc;
    mp.nparts = pp.nparts;
    mp.num_seqs = a.num_seqs;
    mp.num_kv_heads = a.num_kv_heads;
    mp.num_heads = a.num_heads;
    mp.max_parts = w.max_parts;
    mp.part_o = ap.part_o;
    mp.part_lse = ap.part_lse;
    mp.out = ap.out;
    const unsigned pairs = static_cast<unsigned>(a.num_seqs * a.num_kv_heads);
    if (pairs <= 4u * static_cast<unsigned>(a.sm_count))
      err = launch_pdl(lse_merge_kernel<D, G, E, 8>, dim3(pairs), dim3(8 * 32), 0, stream, mp);
    else
      err = launch_pdl(lse_merge_kernel<D, G, E, 4>, dim3(pairs), dim3(4 * 32), 0, stream, mp);
    if (err != cudaSuccess) return err;
    ++*launched;
  }

  return cudaSuccess;
}

cudaError_t launch_attention(const AttnLaunch &a, cudaStream_t stream, int *launched) {
  WorkspaceLayout w;
  if (!workspace_layout(a.num_seqs, a.total_q, a.max_seq_len, a.num_heads, a.num_kv_heads, a.head_dim, a.kv_fp8, w))
    return cudaErrorInvalidValue;
  const int G = a.num_heads / a.num_kv_heads;
#define PA_DISPATCH(DD, GG)                                                                     \
  if (a.head_dim == DD && G == GG) {                                                            \
    if (a.kv_fp8)                                                                               \
      return a.dtype == PA_FP16 ? launch_typed<DD, GG, ElemFp16, true>(a, w, stream, launched)  \
                                : launch_typed<DD, GG, ElemBf16, true>(a, w, stream, launched); \
    return a.dtype == PA_FP16 ? launch_typed<DD, GG, ElemFp16, false>(a, w, stream, launched)   \
                              : launch_typed<DD, GG, ElemBf16, false>(a, w, stream, launched);  \
  }
  PA_DISPATCH(128, 1) PA_DISPATCH(128, 2) PA_DISPATCH(128, 4) PA_DISPATCH(128, 8)
  PA_DISPATCH(64, 1) PA_DISPATCH(64, 2) PA_DISPATCH(64, 4) PA_DISPATCH(64, 8)
  PA_DISPATCH(96, 1) PA_DISPATCH(96, 2) PA_DISPATCH(96, 4) PA_DISPATCH(96, 8)
  PA_DISPATCH(80, 1) PA_DISPATCH(80, 2) PA_DISPATCH(80, 4) PA_DISPATCH(80, 8)
  PA_DISPATCH(256, 1) PA_DISPATCH(256, 2) PA_DISPATCH(256, 4) PA_DISPATCH(256, 8)
#undef PA_DISPATCH
  return cudaErrorInvalidValue;
}

}  // namespace pa
