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
// Design (one CTA of 4 warps per work item):
//   * A work item is (request, KV head, group of up to 8/G query rows,
//     partition of keys). The item's 8 "columns" are (query row, head of the
//     GQA group) pairs, so one pass over a KV block serves the whole group:
//     each K/V byte is read from HBM once per step.
//   * Scores are computed transposed, S^T[16 keys x 8 columns] = K Q^T, with
//     mma.sync m16n8k16 (bf16 in, fp32 accumulate); the probabilities are
//     moved into the B-operand layout with movmatrix and O^T += V^T P^T uses a
//     second mma (P enters as a bf16 hi + lo pair, two mmas, so the weights keep
//     ~16 significant bits). The tensor pipe only removes instruction pressure: the
//     kernel is bound by HBM bandwidth.
//   * K/V blocks are staged into shared memory with 16-byte cp.async through
//     the block table (a 3-stage ring of 4 blocks, one block per warp), with
//     an XOR swizzle so ldmatrix reads are free of bank conflicts. Tokens
//     past the partition end are zero-filled, so stale or NaN cache contents
//     never reach the arithmetic; masked scores are selected to -inf, never
//     multiplied by zero.
//   * Online softmax per column in the log2 domain (scale folded with log2 e),
//     max reductions by warp shuffles; the 4 warps' states are merged in
//     shared memory at the end of the item.
//   * Items of a split request write fp32 (o, lse) partials; the merge kernel
//     combines them: lse = log2 sum 2^lse_p, o = sum 2^(lse_p - lse) o_p.
#include <float.h>

#include "pa_common.cuh"
#include "pa_launch.h"

namespace pa {

using bf16 = __nv_bfloat16;

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 3;
constexpr int kBlocksPerStage = kWarps;  // one 16-token block per warp per stage

struct PlanParams {
  const int32_t *seq_lens;
  const int32_t *query_start_loc;
  int32_t num_seqs;
  int32_t total_q;
  int32_t max_query_len;
  int32_t max_seq_len;
  int32_t max_blocks_per_seq;
  int32_t rows_per_item;  // 8 / G
  int32_t part_tokens;
  int32_t max_items;
  int32_t *item_start;  // [num_seqs + 1]
  int32_t *nparts;      // [num_seqs], 0 = request produces nothing
  int4 *items;          // [2 * max_items]
  int32_t *item_count;  // [1]
  unsigned int *status;
};

struct AttnParams {
  const bf16 *q;
  int64_t q_stride;
  const bf16 *key_cache;
  const bf16 *value_cache;
  const int32_t *block_tables;
  int32_t max_blocks_per_seq;
  int32_t num_heads;
  int32_t num_kv_heads;
  int64_t num_blocks;
  float scale_log2;
  bf16 *out;
  const int4 *items;
  const int32_t *item_count;
  int32_t max_parts;
  float *part_o;    // [num_seqs][Hkv][max_parts][8][D]
  float *part_lse;  // [num_seqs][Hkv][max_parts][8]
  unsigned int *status;
};

struct MergeParams {
  const int32_t *query_start_loc;
  const int32_t *nparts;
  int32_t num_kv_heads;
  int32_t num_heads;
  int32_t max_parts;
  const float *part_o;
  const float *part_lse;
  bf16 *out;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------------------
// Planning: per request, validate the lengths, count work items, scan, and
// write one 32-byte record per item. One CTA; no host synchronisation needed.
// Record: {b, first query token, rows, position of first row},
//         {key begin, key end, partition (-1 = whole range), 0}.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int request_shape(const PlanParams &p, int b, int &q0, int &ql, int &L, int &np) {
  q0 = __ldg(p.query_start_loc + b);
  const int q1 = __ldg(p.query_start_loc + b + 1);
  L = __ldg(p.seq_lens + b);
  ql = q1 - q0;
  np = 0;
  if (q0 < 0 || ql < 0 || q1 > p.total_q || (b == 0 && q0 != 0)) {
    flag_error(p.status, PA_FLAG_QUERY_LOC);
    return 0;
  }
  if (b == p.num_seqs - 1 && q1 != p.total_q) flag_error(p.status, PA_FLAG_QUERY_LOC);
  if (L < ql || L > p.max_seq_len || ql > p.max_query_len ||
      static_cast<int64_t>(L) > static_cast<int64_t>(p.max_blocks_per_seq) * kBlockSize) {
    flag_error(p.status, PA_FLAG_LENGTHS);
    return 0;
  }
  if (ql == 0) return 0;
  const int groups = (ql + p.rows_per_item - 1) / p.rows_per_item;
  np = (groups == 1) ? max(1, (L + p.part_tokens - 1) / p.part_tokens) : 1;
  return groups * np;
}

__global__ void __launch_bounds__(1024) plan_kernel(const PlanParams p) {
  __shared__ int warp_tot[32];
  __shared__ int carry;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < p.num_seqs; base += 1024) {
    const int b = base + tid;
    int cnt = 0;
    if (b < p.num_seqs) {
      int q0, ql, L, np;
      cnt = request_shape(p, b, q0, ql, L, np);
      p.nparts[b] = np;
    }
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int t = warp_tot[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, t, o);
        if (lane >= o) t += v;
      }
      warp_tot[lane] = t;  // inclusive over warps
    }
    __syncthreads();
    const int before = carry + (warp > 0 ? warp_tot[warp - 1] : 0);
    if (b < p.num_seqs) p.item_start[b] = before + incl - cnt;
    __syncthreads();
    if (tid == 0) carry += warp_tot[31];
    __syncthreads();
  }
  if (tid == 0) {
    int total = carry;
    if (total > p.max_items) {
      flag_error(p.status, PA_FLAG_LENGTHS);
      total = p.max_items;
    }
    p.item_start[p.num_seqs] = carry;
    p.item_count[0] = total;
  }
  __syncthreads();
  for (int b = tid; b < p.num_seqs; b += 1024) {
    const int np = p.nparts[b];
    if (np == 0) continue;
    const int q0 = __ldg(p.query_start_loc + b);
    const int ql = __ldg(p.query_start_loc + b + 1) - q0;
    const int L = __ldg(p.seq_lens + b);
    const int ctx = L - ql;
    const int first = p.item_start[b];
    const int cnt = p.item_start[b + 1] - first;
    for (int k = 0; k < cnt; ++k) {
      const int idx = first + k;
      if (idx >= p.max_items) break;
      const int g = k / np, part = k - g * np;
      const int r0 = g * p.rows_per_item;
      const int rows = min(p.rows_per_item, ql - r0);
      const int pos0 = ctx + r0;
      int kb = 0, ke = pos0 + rows;  // the item's last row sees keys < pos0 + rows
      if (np > 1) {
        kb = part * p.part_tokens;
        ke = min(L, kb + p.part_tokens);
      }
      p.items[2 * idx] = make_int4(b, q0 + r0, rows, pos0);
      p.items[2 * idx + 1] = make_int4(kb, ke, np > 1 ? part : -1, 0);
    }
  }
}

// ---------------------------------------------------------------------------
// Split-KV attention. One CTA (4 warps) per work item, persistent over items.
// ---------------------------------------------------------------------------
template <int D, int G>
__global__ void __launch_bounds__(kThreads, 2) splitkv_attention_kernel(const AttnParams p) {
  constexpr int kCols = 8;
  constexpr int CH = D / 8;                                // 16-byte chunks per row
  constexpr int TILE = kBlockSize * D;                     // elements of one block tile
  constexpr int STAGE = 2 * kBlocksPerStage * TILE;        // K tiles then V tiles
  constexpr int MT = D / 16;                               // k-steps of QK^T, m-tiles of O^T
  constexpr int RED_LD = D + 4;                            // padded row of the merge buffer
  static_assert(kWarps * kCols * RED_LD * 4 <= kStages * STAGE * 2, "merge buffer must fit the ring");

  extern __shared__ __align__(1024) unsigned char smem_raw[];
  bf16 *ring = reinterpret_cast<bf16 *>(smem_raw);
  float *red_o = reinterpret_cast<float *>(smem_raw);  // used only while the ring is empty
  __shared__ float red_m[kWarps][kCols];
  __shared__ float red_l[kWarps][kCols];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Hkv = p.num_kv_heads;
  const int64_t total_work = static_cast<int64_t>(__ldg(p.item_count)) * Hkv;

  for (int64_t wk = blockIdx.x; wk < total_work; wk += gridDim.x) {
    const int item = static_cast<int>(wk / Hkv);
    const int kvh = static_cast<int>(wk - static_cast<int64_t>(item) * Hkv);
    const int4 r0 = __ldg(p.items + 2 * item);
    const int4 r1 = __ldg(p.items + 2 * item + 1);
    const int b = r0.x, row0 = r0.y, nrows = r0.z, pos0 = r0.w;
    const int kv_begin = r1.x, kv_end = r1.y, part = r1.z;
    const int32_t *table = p.block_tables + static_cast<int64_t>(b) * p.max_blocks_per_seq;

    // B operand of S^T = K Q^T: column n = lane / 4 is (query row n / G, head n % G).
    uint32_t qf[MT][2];
    {
      const int n = lane >> 2, qi = n / G, g = n % G;
      const bool ok = qi < nrows;
      const bf16 *qp = p.q + static_cast<int64_t>(row0 + (ok ? qi : 0)) * p.q_stride +
                       static_cast<int64_t>(kvh * G + g) * D + 2 * (lane & 3);
#pragma unroll
      for (int kk = 0; kk < MT; ++kk) {
        qf[kk][0] = ok ? __ldg(reinterpret_cast<const uint32_t *>(qp + 16 * kk)) : 0u;
        qf[kk][1] = ok ? __ldg(reinterpret_cast<const uint32_t *>(qp + 16 * kk + 8)) : 0u;
      }
    }
    // Keys j < lim[e] are visible to this thread's accumulator column 2*(lane%4)+e.
    int lim[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int qi = (2 * (lane & 3) + e) / G;
      lim[e] = qi < nrows ? min(pos0 + qi + 1, kv_end) : kv_begin;
    }

    float o[MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    float m[2] = {-INFINITY, -INFINITY};
    float l[2] = {0.f, 0.f};

    const int kb0 = kv_begin / kBlockSize;
    const int kb1 = (kv_end + kBlockSize - 1) / kBlockSize;
    const int nst = (kb1 - kb0 + kBlocksPerStage - 1) / kBlocksPerStage;

    auto issue = [&](int s) {
      bf16 *st = ring + (s % kStages) * STAGE;
      constexpr int PER = 2 * kBlocksPerStage * kBlockSize * CH;
#pragma unroll 4
      for (int i = tid; i < PER; i += kThreads) {
        const int c = i % CH;
        const int row = (i / CH) % kBlockSize;
        const int t2 = i / (CH * kBlockSize);
        const int blk = t2 >> 1, isv = t2 & 1;
        const int kb = kb0 + s * kBlocksPerStage + blk;
        if (kb < kb1) {
          int phys = __ldg(table + kb);
          int bytes = (kb * kBlockSize + row < kv_end) ? 16 : 0;
          if (phys < 0 || phys >= p.num_blocks) {
            if (c == 0 && row == 0 && isv == 0) flag_error(p.status, PA_FLAG_BLOCK_RANGE);
            phys = 0;
            bytes = 0;
          }
          const bf16 *src = (isv ? p.value_cache : p.key_cache) +
                            ((static_cast<int64_t>(phys) * kBlockSize + row) * Hkv + kvh) * D + c * 8;
          bf16 *dst = st + isv * kBlocksPerStage * TILE + blk * TILE + swz(row, c, D);
          cp_async_16(smem_u32(dst), src, bytes);
        }
      }
    };

#pragma unroll
    for (int s = 0; s < kStages - 1; ++s) {
      if (s < nst) issue(s);
      cp_async_commit();
    }

    const int arow = (lane & 7) + ((lane >> 3) & 1) * 8;  // ldmatrix row for K (A operand)
    const int vrow = (lane & 7) + (lane >> 4) * 8;        // ldmatrix row for V (transposed A)
    for (int s = 0; s < nst; ++s) {
      cp_async_wait<kStages - 2>();
      __syncthreads();
      if (s + kStages - 1 < nst) issue(s + kStages - 1);
      cp_async_commit();

      const int kb = kb0 + s * kBlocksPerStage + warp;
      if (kb < kb1) {
        const bf16 *kt = ring + (s % kStages) * STAGE + warp * TILE;
        const bf16 *vt = kt + kBlocksPerStage * TILE;
        const uint32_t kbase = smem_u32(kt), vbase = smem_u32(vt);

        float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < MT; ++kk) {
          uint32_t a0, a1, a2, a3;
          ldsm_x4(kbase + 2 * swz(arow, 2 * kk + (lane >> 4), D), a0, a1, a2, a3);
          mma_16816(sc, a0, a1, a2, a3, qf[kk][0], qf[kk][1]);
        }
        const int t0 = kb * kBlockSize + (lane >> 2), t1 = t0 + 8;
        const float x0 = t0 < lim[0] ? sc[0] * p.scale_log2 : -INFINITY;
        const float x1 = t0 < lim[1] ? sc[1] * p.scale_log2 : -INFINITY;
        const float x2 = t1 < lim[0] ? sc[2] * p.scale_log2 : -INFINITY;
        const float x3 = t1 < lim[1] ? sc[3] * p.scale_log2 : -INFINITY;
        float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const float mn0 = fmaxf(m[0], mx0), mn1 = fmaxf(m[1], mx1);
        const float ms0 = mn0 == -INFINITY ? 0.f : mn0;
        const float ms1 = mn1 == -INFINITY ? 0.f : mn1;
        const float al0 = ex2(m[0] - ms0), al1 = ex2(m[1] - ms1);
        const float p0 = ex2(x0 - ms0), p1 = ex2(x1 - ms1);
        const float p2 = ex2(x2 - ms0), p3 = ex2(x3 - ms1);
        l[0] = l[0] * al0 + p0 + p2;
        l[1] = l[1] * al1 + p1 + p3;
        m[0] = mn0;
        m[1] = mn1;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          o[mt][0] *= al0;
          o[mt][1] *= al1;
          o[mt][2] *= al0;
          o[mt][3] *= al1;
        }
        // P^T rows (keys) x columns -> B operand (k = key, n = column) by transposition.
        // P is carried as a bf16 pair hi + lo (hi = bf16(p), lo = bf16(p - hi)), so the
        // probabilities enter the fp32 accumulation with ~16 significant bits instead of 8.
        const uint32_t h01 = pack_bf16x2(p0, p1), h23 = pack_bf16x2(p2, p3);
        const uint32_t l01 = pack_bf16x2(p0 - bf16_lo(h01), p1 - bf16_hi(h01));
        const uint32_t l23 = pack_bf16x2(p2 - bf16_lo(h23), p3 - bf16_hi(h23));
        const uint32_t b0 = movmatrix_t(h01), b1 = movmatrix_t(h23);
        const uint32_t c0 = movmatrix_t(l01), c1 = movmatrix_t(l23);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          uint32_t a0, a1, a2, a3;
          ldsm_x4_t(vbase + 2 * swz(vrow, 2 * mt + ((lane >> 3) & 1), D), a0, a1, a2, a3);
          mma_16816(o[mt], a0, a1, a2, a3, b0, b1);
          mma_16816(o[mt], a0, a1, a2, a3, c0, c1);
        }
      }
    }
    cp_async_wait<0>();
    __syncthreads();

    // ---- merge the 4 warps' (m, l, O) per column ----
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l[0] += __shfl_xor_sync(0xffffffffu, l[0], off);
      l[1] += __shfl_xor_sync(0xffffffffu, l[1], off);
    }
    if (lane < 4) {
      red_m[warp][2 * lane] = m[0];
      red_m[warp][2 * lane + 1] = m[1];
      red_l[warp][2 * lane] = l[0];
      red_l[warp][2 * lane + 1] = l[1];
    }
    __syncthreads();
    {
      float f[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int c = 2 * (lane & 3) + e;
        float M = red_m[0][c];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) M = fmaxf(M, red_m[w][c]);
        const float Ms = M == -INFINITY ? 0.f : M;
        f[e] = ex2(m[e] - Ms);
      }
      float *ro = red_o + warp * kCols * RED_LD;
      const int c0 = 2 * (lane & 3);
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const int d = 16 * mt + (lane >> 2);
        ro[c0 * RED_LD + d] = o[mt][0] * f[0];
        ro[(c0 + 1) * RED_LD + d] = o[mt][1] * f[1];
        ro[c0 * RED_LD + d + 8] = o[mt][2] * f[0];
        ro[(c0 + 1) * RED_LD + d + 8] = o[mt][3] * f[1];
      }
    }
    __syncthreads();
    {
      constexpr int TPC = kThreads / kCols;  // threads per column
      constexpr int EPT = D / TPC;           // elements per thread
      const int col = tid / TPC, d0 = (tid % TPC) * EPT;
      const int qi = col / G, g = col % G;
      if (qi < nrows) {
        float M = red_m[0][col];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) M = fmaxf(M, red_m[w][col]);
        const float Ms = M == -INFINITY ? 0.f : M;
        float Lc = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) Lc += red_l[w][col] * ex2(red_m[w][col] - Ms);
        const float inv = Lc > 0.f ? 1.f / Lc : 0.f;
        float acc[EPT];
#pragma unroll
        for (int e = 0; e < EPT; ++e) {
          float s = 0.f;
#pragma unroll
          for (int w = 0; w < kWarps; ++w) s += red_o[(w * kCols + col) * RED_LD + d0 + e];
          acc[e] = s * inv;
        }
        if (part < 0) {
          bf16 *dst = p.out + static_cast<int64_t>(row0 + qi) * p.num_heads * D +
                      static_cast<int64_t>(kvh * G + g) * D + d0;
          uint32_t pk[EPT / 2];
#pragma unroll
          for (int e = 0; e < EPT / 2; ++e) pk[e] = pack_bf16x2(acc[2 * e], acc[2 * e + 1]);
          if constexpr (EPT == 8) {
            *reinterpret_cast<uint4 *>(dst) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          } else {
            *reinterpret_cast<uint2 *>(dst) = make_uint2(pk[0], pk[1]);
          }
        } else {
          const int64_t idx = ((static_cast<int64_t>(b) * Hkv + kvh) * p.max_parts + part) * kCols + col;
          float *dst = p.part_o + idx * D + d0;
#pragma unroll
          for (int e = 0; e < EPT; e += 4)
            *reinterpret_cast<float4 *>(dst + e) = make_float4(acc[e], acc[e + 1], acc[e + 2], acc[e + 3]);
          if (tid % TPC == 0) p.part_lse[idx] = Lc > 0.f ? Ms + __log2f(Lc) : -INFINITY;
        }
      }
    }
    __syncthreads();  // the merge buffers alias the ring used by the next item
  }
}

// ---------------------------------------------------------------------------
// Log-sum-exp merge of the partitions of split requests (decode rows).
// One CTA per (request, KV head); 16 threads per column.
// ---------------------------------------------------------------------------
template <int D, int G>
__global__ void __launch_bounds__(128) lse_merge_kernel(const MergeParams p) {
  constexpr int kCols = 8;
  constexpr int TPC = 128 / kCols;
  constexpr int EPT = D / TPC;
  const int b = blockIdx.x / p.num_kv_heads;
  const int kvh = blockIdx.x - b * p.num_kv_heads;
  const int np = __ldg(p.nparts + b);
  if (np <= 1) return;
  const int q0 = __ldg(p.query_start_loc + b);
  const int ql = __ldg(p.query_start_loc + b + 1) - q0;
  const int col = threadIdx.x / TPC, d0 = (threadIdx.x % TPC) * EPT;
  const int qi = col / G, g = col % G;
  if (qi >= ql) return;
  const int64_t base = (static_cast<int64_t>(b) * p.num_kv_heads + kvh) * p.max_parts;
  float M = -INFINITY;
  for (int k = 0; k < np; ++k) M = fmaxf(M, __ldg(p.part_lse + (base + k) * kCols + col));
  const float Ms = M == -INFINITY ? 0.f : M;
  float acc[EPT];
#pragma unroll
  for (int e = 0; e < EPT; ++e) acc[e] = 0.f;
  float wsum = 0.f;
  for (int k = 0; k < np; ++k) {
    const int64_t idx = (base + k) * kCols + col;
    const float w = ex2(__ldg(p.part_lse + idx) - Ms);
    wsum += w;
    const float *src = p.part_o + idx * D + d0;
#pragma unroll
    for (int e = 0; e < EPT; e += 4) {
      const float4 v = __ldg(reinterpret_cast<const float4 *>(src + e));
      acc[e] += w * v.x;
      acc[e + 1] += w * v.y;
      acc[e + 2] += w * v.z;
      acc[e + 3] += w * v.w;
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  bf16 *dst = p.out + static_cast<int64_t>(q0 + qi) * p.num_heads * D + static_cast<int64_t>(kvh * G + g) * D + d0;
  uint32_t pk[EPT / 2];
#pragma unroll
  for (int e = 0; e < EPT / 2; ++e) pk[e] = pack_bf16x2(acc[2 * e] * inv, acc[2 * e + 1] * inv);
  if constexpr (EPT == 8) {
    *reinterpret_cast<uint4 *>(dst) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  } else {
    *reinterpret_cast<uint2 *>(dst) = make_uint2(pk[0], pk[1]);
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

// Keys per partition. Partitions bound the work of one item, so that a few
// long requests cannot leave most SMs idle at the end of the step.
int partition_tokens(int32_t num_seqs, int32_t max_seq_len, int32_t num_kv_heads) {
  (void)num_seqs;
  (void)max_seq_len;
  (void)num_kv_heads;
  return 512;
}


static size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

bool workspace_layout(int32_t num_seqs, int32_t total_q, int32_t max_seq_len, int32_t num_heads,
                      int32_t num_kv_heads, int32_t head_dim, WorkspaceLayout &w) {
  if (num_seqs < 0 || total_q < 0 || max_seq_len < 0 || num_heads <= 0 || num_kv_heads <= 0 ||
      head_dim <= 0 || num_heads % num_kv_heads != 0)
    return false;
  const int G = num_heads / num_kv_heads;
  if (G > 8) return false;
  w.rows_per_item = 8 / G;
  w.part_tokens = partition_tokens(num_seqs, max_seq_len, num_kv_heads);
  w.max_parts = max_seq_len > 0 ? (max_seq_len + w.part_tokens - 1) / w.part_tokens : 1;
  const int64_t items = static_cast<int64_t>(num_seqs) * w.max_parts +
                        (static_cast<int64_t>(total_q) + w.rows_per_item - 1) / w.rows_per_item + num_seqs;
  if (items > (1LL << 30)) return false;
  w.max_items = static_cast<int32_t>(items);
  const size_t nsplit = static_cast<size_t>(num_seqs) * num_kv_heads * w.max_parts * 8;
  size_t off = 0;
  w.item_start = off; off += align256(sizeof(int32_t) * (static_cast<size_t>(num_seqs) + 1));
  w.nparts = off;     off += align256(sizeof(int32_t) * (static_cast<size_t>(num_seqs) + 1));
  w.item_count = off; off += align256(sizeof(int32_t));
  w.items = off;      off += align256(sizeof(int4) * 2 * static_cast<size_t>(w.max_items));
  w.part_lse = off;   off += align256(sizeof(float) * nsplit);
  w.part_o = off;     off += align256(sizeof(float) * nsplit * head_dim);
  w.total = off;
  return true;
}


template <int D, int G>
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
  pp.rows_per_item = w.rows_per_item;
  pp.part_tokens = w.part_tokens;
  pp.max_items = w.max_items;
  pp.item_start = reinterpret_cast<int32_t *>(ws + w.item_start);
  pp.nparts = reinterpret_cast<int32_t *>(ws + w.nparts);
  pp.items = reinterpret_cast<int4 *>(ws + w.items);
  pp.item_count = reinterpret_cast<int32_t *>(ws + w.item_count);
  pp.status = a.status;
  plan_kernel<<<1, 1024, 0, stream>>>(pp);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  ++*launched;

  AttnParams ap;
  ap.q = static_cast<const bf16 *>(a.q);
  ap.q_stride = a.q_stride;
  ap.key_cache = static_cast<const bf16 *>(a.key_cache);
  ap.value_cache = static_cast<const bf16 *>(a.value_cache);
  ap.block_tables = a.block_tables;
  ap.max_blocks_per_seq = a.max_blocks_per_seq;
  ap.num_heads = a.num_heads;
  ap.num_kv_heads = a.num_kv_heads;
  ap.num_blocks = a.num_blocks;
  ap.scale_log2 = a.scale * 1.4426950408889634f;
  ap.out = static_cast<bf16 *>(a.out);
  ap.items = pp.items;
  ap.item_count = pp.item_count;
  ap.max_parts = w.max_parts;
  ap.part_o = reinterpret_cast<float *>(ws + w.part_o);
  ap.part_lse = reinterpret_cast<float *>(ws + w.part_lse);
  ap.status = a.status;

  constexpr int smem = kStages * 2 * kBlocksPerStage * kBlockSize * D * 2;
  auto kern = splitkv_attention_kernel<D, G>;
  err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  int occ = 0;
  err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kThreads, smem);
  if (err != cudaSuccess) return err;
  if (occ < 1) occ = 1;
  int64_t grid = static_cast<int64_t>(a.sm_count) * occ;
  const int64_t upper = static_cast<int64_t>(w.max_items) * a.num_kv_heads;
  if (grid > upper) grid = upper;
  if (grid < 1) grid = 1;
  if (a.ev_start) cudaEventRecord(a.ev_start, stream);
  kern<<<static_cast<int>(grid), kThreads, smem, stream>>>(ap);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  ++*launched;
  if (a.ev_stop) cudaEventRecord(a.ev_stop, stream);

  if (w.max_parts > 1 && a.num_seqs > 0) {
    MergeParams mp;
    mp.query_start_loc = a.query_start_loc;
    mp.nparts = pp.nparts;
    mp.num_kv_heads = a.num_kv_heads;
    mp.num_heads = a.num_heads;
    mp.max_parts = w.max_parts;
    mp.part_o = ap.part_o;
    mp.part_lse = ap.part_lse;
    mp.out = ap.out;
    lse_merge_kernel<D, G><<<a.num_seqs * a.num_kv_heads, 128, 0, stream>>>(mp);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    ++*launched;
  }
  return cudaSuccess;
}

cudaError_t launch_attention(const AttnLaunch &a, cudaStream_t stream, int *launched) {
  WorkspaceLayout w;
  if (!workspace_layout(a.num_seqs, a.total_q, a.max_seq_len, a.num_heads, a.num_kv_heads, a.head_dim, w))
    return cudaErrorInvalidValue;
  const int G = a.num_heads / a.num_kv_heads;
#define PA_DISPATCH(DD, GG) \
  if (a.head_dim == DD && G == GG) return launch_typed<DD, GG>(a, w, stream, launched);
  PA_DISPATCH(128, 1) PA_DISPATCH(128, 2) PA_DISPATCH(128, 4) PA_DISPATCH(128, 8)
  PA_DISPATCH(64, 1) PA_DISPATCH(64, 2) PA_DISPATCH(64, 4) PA_DISPATCH(64, 8)
#undef PA_DISPATCH
  return cudaErrorInvalidValue;
}

}  // namespace pa
