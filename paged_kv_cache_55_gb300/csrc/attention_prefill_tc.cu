// Chunked-prefill attention on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// Sources (vLLM inference notes, "AI Infra入门干货总结：大模型是如何高效推理的"):
//   §LLM 推理全流程 3 - prefill is a dense, compute-bound GEMM; FlashAttention
//     fuses QK^T, softmax and PV with tiling and online softmax; GQA maps a
//     group of query heads to one KV head by index.
//   §Continuous Batching - a request's query chunk sits at positions
//     ctx .. ctx + query_len - 1 and each query sees keys up to its own
//     position (chunked prefill, named in the LLM-infra reading map,
//     "lpnh.cn/news/2436702", §2.3).
//
// One CTA handles one tile of 128 "packed rows" = (query position, head of
// the GQA group) pairs of one request and one KV head, so each K/V byte
// staged for the tile serves all G heads. The keys are walked in ranges of
// 64 by three kinds of warps that hand work over through mbarriers only:
//   * a producer warp issues TMA loads of the (block, KV head) tiles of K and
//     V through the block table into 128-byte-swizzled shared memory (the
//     decode path's boxes), two buffers each with full/empty barriers,
//     K(r+1) ahead of V(r);
//   * an MMA warp issues tcgen05.mma: S = Q K^T into tensor memory as soon
//     as K(r) has landed and the softmax has released S, then O += P_hi V +
//     P_lo V for the previous range (P read from tensor memory, V an MN-major
//     shared-memory operand), so the softmax of range r runs while the tensor
//     cores multiply range r-1; it zeroes V rows past the last key first;
//   * four softmax warps own one row each per thread (its TMEM lane): they
//     read the 64 scores, apply the causal limit, keep the running max and
//     sum (log2 domain) and store P into tensor memory as a bf16 hi + lo pair;
//     O accumulates in tensor memory and a row is rescaled there only when
//     its running maximum grows by more than 2^8.
// Two CTAs share an SM (96 KB of shared memory, 256 TMEM columns each). All
// shared state is in the dynamic segment, whose start must be 1024-byte
// aligned for the swizzled tiles (checked). Waits on mbarriers are bounded
// (a thread waits out at most one timeout, then runs to the unit barrier);
// tensor memory is released on every exit path.
#include "attention_internal.cuh"

namespace pa {

constexpr int kTileRows = 128;  // UMMA M
constexpr int kKeyTile = 64;    // keys per range (UMMA N of S, K of P V)
constexpr int kSoftmaxWarps = 4, kMmaWarp = 4, kTmaWarp = 5;
constexpr int kTileThreads = 32 * (kTmaWarp + 1);
constexpr uint64_t kTcWaitTimeoutNs = 2000000000;

// Tensor memory columns: S [0, 64), O [64, 64 + D), P_hi and P_lo 32 each.
template <int D>
struct TcTmem {
  static constexpr uint32_t S = 0, O = kKeyTile, PHI = kKeyTile + D, PLO = PHI + kKeyTile / 2;
  static constexpr uint32_t USED = PLO + kKeyTile / 2;
  static constexpr uint32_t COLS = USED <= 128 ? 128u : (USED <= 256 ? 256u : 512u);  // power of two
};

template <int D>
struct TcLayout {
  static constexpr int HALVES = D / 64;           // 64-element swizzle atoms along D
  static constexpr int Q_HALF = kTileRows * 128;  // 128 rows x 128 B
  static constexpr int KV_HALF = kKeyTile * 128;  // 64 rows x 128 B
  static constexpr int Q_BYTES = HALVES * Q_HALF;
  static constexpr int KV_BYTES = HALVES * KV_HALF;
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + Q_BYTES;          // two K buffers
  static constexpr int V_OFF = K_OFF + 2 * KV_BYTES;     // two V buffers
  static constexpr int TABLE_OFF = V_OFF + 2 * KV_BYTES;  // the tile's block-table entries
  static constexpr int TABLE_ENTRIES = 1024;             // keys < 16384 read from here
  static constexpr int BAR_OFF = TABLE_OFF + TABLE_ENTRIES * 4;
  // barriers: k_full[2], k_empty[2], v_full[2], v_empty[2], s_full, p_full, o_done, q_full
  static constexpr int NBARS = 12;
  static constexpr int BYTES = BAR_OFF + 8 * NBARS + 16;
  // Shared memory requested per CTA: at least 77 KB so that no more than two
  // CTAs (2 x 256 TMEM columns) can ever share an SM.
  static constexpr int REQUEST = BYTES > 77 * 1024 ? BYTES : 77 * 1024;
  // byte offset of 16-byte chunk c of row r in a swizzled tile with `half` bytes per atom column
  static __device__ __forceinline__ uint32_t off(int r, int c, int half) {
    return (c >> 3) * half + r * 128 + (((c & 7) ^ (r & 7)) << 4);
  }
};

// Bounded wait that is skipped once this thread has given up: a thread waits
// out at most one timeout, then runs to the next unit barrier.
__device__ __forceinline__ void wait_or_fail(uint32_t bar, uint32_t parity, bool &failed) {
  if (!failed) failed = !mbar_wait_bounded(bar, parity, kTcWaitTimeoutNs);
}

template <int D, int G>
__global__ void __launch_bounds__(kTileThreads, 2)
    prefill_tile_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                        const TileParams p) {
  using Lay = TcLayout<D>;
  using Tm = TcTmem<D>;
  constexpr int KSTEPS_S = D / 16;         // UMMA K steps of S = Q K^T
  constexpr int KSTEPS_O = kKeyTile / 16;  // UMMA K steps of O = P V
  constexpr int BLOCKS = kKeyTile / kBlockSize;
  constexpr uint32_t IDESC_S = f16_idesc(kTileRows, kKeyTile, 0);
  constexpr uint32_t IDESC_O = f16_idesc(kTileRows, D, 1);
  // O stays in TMEM and is rescaled only when a row's running maximum grows
  // by more than 2^8 (log2 domain); in between, probabilities are taken
  // against the older maximum and stay below 256.
  constexpr float kRescaleLog2 = 8.f;

  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t base = smem_u32(smem_raw);
  if (base & 1023u) {  // the swizzled tiles need 1024-byte alignment; never touch misaligned tiles
    if (tid == 0) flag_error(p.status, PA_FLAG_LENGTHS);
    return;
  }
  const uint32_t sQ = base + Lay::Q_OFF, sK0 = base + Lay::K_OFF, sV0 = base + Lay::V_OFF;
  const uint32_t bars = base + Lay::BAR_OFF;
  const uint32_t bar_kfull = bars, bar_kempty = bars + 16, bar_vfull = bars + 32, bar_vempty = bars + 48;
  const uint32_t bar_s = bars + 64, bar_p = bars + 72, bar_o = bars + 80, bar_q = bars + 88;
  uint32_t *tmem_base_s = reinterpret_cast<uint32_t *>(smem_raw + Lay::BAR_OFF + 8 * Lay::NBARS);
  int *unit_s = reinterpret_cast<int *>(smem_raw + Lay::BAR_OFF + 8 * Lay::NBARS + 4);
  int *stable = reinterpret_cast<int *>(smem_raw + Lay::TABLE_OFF);

  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_base_s), Tm::COLS);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < 8; ++i) mbar_init(bars + 8 * i, 1);  // full: producer, empty: MMA commits
    mbar_init(bar_s, 1);
    mbar_init(bar_p, kSoftmaxWarps);
    mbar_init(bar_o, 1);
    mbar_init(bar_q, kSoftmaxWarps);
    prefetch_tmap(&kmap);
    prefetch_tmap(&vmap);
  }
  fence_mbar_init();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_base_s;
  griddep_wait();

  const int Hkv = p.num_kv_heads;
  const int total_units = min(max(ld_cg(p.tile_count), 0), p.max_tiles) * Hkv;
  // Per-role counters from which every mbarrier parity follows (they run on
  // across units, like the barriers themselves).
  uint32_t kload[2] = {0, 0}, vload[2] = {0, 0};  // producer: loads issued per buffer
  uint32_t kseen[2] = {0, 0}, vseen[2] = {0, 0};  // MMA: loads consumed per buffer
  uint32_t n_p = 0, n_q = 0;                      // MMA: softmax hand-offs consumed
  uint32_t n_s = 0, n_o = 0;                      // softmax: S and P V products consumed
  bool failed = false;

  for (;;) {
    if (tid == 0) *unit_s = atomicAdd(p.tile_counter, 1);
    if (__syncthreads_or(failed)) break;  // unit barrier: every role is done with the last unit
    const int u = *unit_s;
    if (u >= total_units) break;
    const int item = u / Hkv, kvh = u - item * Hkv;
    const int4 r0 = ld_cg(p.tiles + 2 * item);
    const int4 r1 = ld_cg(p.tiles + 2 * item + 1);
    const int b = r0.x, row0 = r0.y, npos = r0.z, pos0 = r0.w, kv_end = r1.y;
    const bool sane = b >= 0 && b < p.num_seqs && npos >= 1 && npos <= kTileRows / G && row0 >= 0 &&
                      row0 + npos <= p.total_q && pos0 >= 0 && kv_end == pos0 + npos &&
                      kv_end <= static_cast<int64_t>(p.max_blocks_per_seq) * kBlockSize;
    if (!sane) {
      if (tid == 0) flag_error(p.status, PA_FLAG_LENGTHS);
      __syncthreads();  // unit_s is rewritten next iteration
      continue;
    }
    const int32_t *table = p.block_tables + static_cast<int64_t>(b) * p.max_blocks_per_seq;
    const int nblk = (kv_end + kBlockSize - 1) / kBlockSize;
    const int nkt = (kv_end + kKeyTile - 1) / kKeyTile;
    for (int i = tid; i < min(nblk, Lay::TABLE_ENTRIES); i += kTileThreads) stable[i] = __ldg(table + i);
    __syncthreads();

    if (warp == kTmaWarp) {
      // ---------------- producer: K(j+1) ahead of V(j) ----------------
      if (lane == 0) {
        auto load = [&](int kt, bool is_v) {
          const int buf = kt & 1;
          uint32_t &n = is_v ? vload[buf] : kload[buf];
          if (n > 0) wait_or_fail((is_v ? bar_vempty : bar_kempty) + 8 * buf, (n - 1) & 1u, failed);
          ++n;
          if (failed) return;
          const uint32_t bar = (is_v ? bar_vfull : bar_kfull) + 8 * buf;
          const uint32_t dst = (is_v ? sV0 : sK0) + buf * Lay::KV_BYTES;
          const void *map = is_v ? static_cast<const void *>(&vmap) : static_cast<const void *>(&kmap);
          mbar_arrive_expect_tx(bar, Lay::KV_BYTES);
#pragma unroll
          for (int blk = 0; blk < BLOCKS; ++blk) {
            const int kb = kt * BLOCKS + blk;
            int z = -kBlockSize;  // past the keys this tile needs: TMA fills zeros
            if (kb < nblk) {
              const int phys = kb < Lay::TABLE_ENTRIES ? stable[kb] : __ldg(table + kb);
              if (phys >= 0 && phys < p.num_blocks)
                z = phys * kBlockSize;
              else if (!is_v)
                flag_error(p.status, PA_FLAG_BLOCK_RANGE);
            }
#pragma unroll
            for (int h = 0; h < Lay::HALVES; ++h)
              tma_load_3d(dst + h * Lay::KV_HALF + blk * 2048, map, bar, h * 64, kvh, z);
          }
        };
        load(0, false);
        for (int j = 0; j < nkt; ++j) {
          if (j + 1 < nkt) load(j + 1, false);
          load(j, true);
        }
      }
    } else if (warp == kMmaWarp) {
      // ---------------- MMA issue: S(kt), then P V of the previous range ----------------
      // The whole warp follows the loop (it zeroes the tail of the last V
      // range); lane 0 alone issues tensor-core work and commits.
      auto issue_pv = [&](int kt) {
        const int buf = kt & 1;
        wait_or_fail(bar_vfull + 8 * buf, vseen[buf] & 1u, failed);
        ++vseen[buf];
        const uint32_t sV = sV0 + buf * Lay::KV_BYTES;
        const int key0 = kt * kKeyTile;
        if (!failed && key0 + kKeyTile > kv_end) {
          // rows of keys past kv_end may hold anything (even NaN): zero them in V
          const int vr0 = kv_end - key0;
          const int n = (kKeyTile - vr0) * (D / 8);
          for (int i = lane; i < n; i += 32) {
            const int rr = vr0 + i / (D / 8), c = i % (D / 8);
            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};\n" ::"r"(sV + Lay::off(rr, c, Lay::KV_HALF)),
                         "r"(0u)
                         : "memory");
          }
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0 && !failed) {
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < KSTEPS_O; ++ks) {
            const uint64_t vd = sw128_desc(sV + ks * 2048, Lay::KV_HALF, 1024);
            tc_mma_f16_ta(tmem + Tm::O, tmem + Tm::PHI + ks * 8, vd, IDESC_O, (kt > 0 || ks > 0) ? 1u : 0u);
            tc_mma_f16_ta(tmem + Tm::O, tmem + Tm::PLO + ks * 8, vd, IDESC_O, 1u);
          }
          tc_commit(bar_o);
          tc_commit(bar_vempty + 8 * buf);
        }
        __syncwarp();
      };
      wait_or_fail(bar_q, n_q & 1u, failed);
      ++n_q;
      for (int kt = 0; kt < nkt; ++kt) {
        const int buf = kt & 1;
        wait_or_fail(bar_kfull + 8 * buf, kseen[buf] & 1u, failed);
        ++kseen[buf];
        if (kt > 0) {  // softmax of the previous range is done: S is free, its P is ready
          wait_or_fail(bar_p, n_p & 1u, failed);
          ++n_p;
        }
        if (lane == 0 && !failed) {
          tc_fence_after();
          const uint32_t sK = sK0 + buf * Lay::KV_BYTES;
#pragma unroll
          for (int ks = 0; ks < KSTEPS_S; ++ks) {
            const uint64_t a = sw128_desc(sQ + (ks >> 2) * Lay::Q_HALF + (ks & 3) * 32, 16, 1024);
            const uint64_t bd = sw128_desc(sK + (ks >> 2) * Lay::KV_HALF + (ks & 3) * 32, 16, 1024);
            tc_mma_f16(tmem + Tm::S, a, bd, IDESC_S, ks > 0);
          }
          tc_commit(bar_s);
          tc_commit(bar_kempty + 8 * buf);
        }
        __syncwarp();
        if (kt > 0) issue_pv(kt - 1);
      }
      wait_or_fail(bar_p, n_p & 1u, failed);
      ++n_p;
      issue_pv(nkt - 1);
    } else {
      // ---------------- softmax: one row per thread (its TMEM lane) ----------------
      const uint32_t t_lane = tmem + (static_cast<uint32_t>(warp * 32) << 16);
      const int r = tid, qi = r / G, g = r % G;
      const bool row_valid = qi < npos;
      {  // Q tile: row r = (position r / G, head r % G), K-major, swizzled
        const uint32_t *src = reinterpret_cast<const uint32_t *>(
            p.q + static_cast<int64_t>(row0 + (row_valid ? qi : 0)) * p.q_stride + static_cast<int64_t>(kvh * G + g) * D);
#pragma unroll 4
        for (int c = 0; c < D / 8; ++c) {
          uint32_t w0 = 0, w1 = 0, w2 = 0, w3 = 0;
          if (row_valid) {
            w0 = __ldg(src + 4 * c);
            w1 = __ldg(src + 4 * c + 1);
            w2 = __ldg(src + 4 * c + 2);
            w3 = __ldg(src + 4 * c + 3);
          }
          asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};\n" ::"r"(sQ + Lay::off(r, c, Lay::Q_HALF)),
                       "r"(w0), "r"(w1), "r"(w2), "r"(w3)
                       : "memory");
        }
        fence_proxy_async_smem();  // the MMA reads Q through the async proxy
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_q);
      }
      float m_used = -INFINITY, l = 0.f;
      const int lim = row_valid ? pos0 + qi + 1 : 0;  // keys j < lim are visible to this row
      for (int kt = 0; kt < nkt; ++kt) {
        const int key0 = kt * kKeyTile;
        wait_or_fail(bar_s, n_s & 1u, failed);
        ++n_s;
        tc_fence_after();
        float x[kKeyTile];
        {
          float s0[32], s1[32];
          tmem_ld32(t_lane + Tm::S, s0);
          tmem_ld32(t_lane + Tm::S + 32, s1);
          if (key0 + kKeyTile <= lim) {  // every key of the range is visible to this row
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              x[i] = s0[i] * p.scale_log2;
              x[32 + i] = s1[i] * p.scale_log2;
            }
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              x[i] = key0 + i < lim ? s0[i] * p.scale_log2 : -INFINITY;
              x[32 + i] = key0 + 32 + i < lim ? s1[i] * p.scale_log2 : -INFINITY;
            }
          }
        }
        float t8[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          float a = fmaxf(fmaxf(x[j], x[j + 8]), fmaxf(x[j + 16], x[j + 24]));
          float c = fmaxf(fmaxf(x[j + 32], x[j + 40]), fmaxf(x[j + 48], x[j + 56]));
          t8[j] = fmaxf(a, c);
        }
        const float mx = fmaxf(fmaxf(fmaxf(t8[0], t8[1]), fmaxf(t8[2], t8[3])),
                               fmaxf(fmaxf(t8[4], t8[5]), fmaxf(t8[6], t8[7])));
        // the previous product must be complete before O is rescaled or P rewritten
        if (kt > 0) {
          wait_or_fail(bar_o, n_o & 1u, failed);
          ++n_o;
          tc_fence_after();
        }
        if (mx > -INFINITY && (m_used == -INFINITY || mx > m_used + kRescaleLog2)) {
          if (kt > 0 && m_used > -INFINITY) {
            const float alpha = ex2_approx(m_used - mx);
            l *= alpha;
#pragma unroll
            for (int ch = 0; ch < D / 32; ++ch) {
              float t[32];
              tmem_ld32(t_lane + Tm::O + ch * 32, t);
#pragma unroll
              for (int i = 0; i < 32; ++i) t[i] *= alpha;
              tmem_st32(t_lane + Tm::O + ch * 32, t);
            }
          }
          m_used = mx;
        }
        const float ms = m_used == -INFINITY ? 0.f : m_used;
        float rs4[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t hi[kKeyTile / 2], lo[kKeyTile / 2];
#pragma unroll
        for (int i = 0; i < kKeyTile / 2; ++i) {
          const float p0 = ex2_approx(x[2 * i] - ms);
          const float p1 = ex2_approx(x[2 * i + 1] - ms);
          rs4[i & 3] += p0 + p1;
          hi[i] = pack_bf16x2(p0, p1);
          lo[i] = pack_bf16x2(p0 - bf16_lo(hi[i]), p1 - bf16_hi(hi[i]));
        }
        tmem_st32u(t_lane + Tm::PHI, hi);
        tmem_st32u(t_lane + Tm::PLO, lo);
        tmem_wait_st();
        l += (rs4[0] + rs4[1]) + (rs4[2] + rs4[3]);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_p);
      }
      // epilogue: the last P V product, normalised
      wait_or_fail(bar_o, n_o & 1u, failed);
      ++n_o;
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      bf16 *dst = p.out + static_cast<int64_t>(row0 + (row_valid ? qi : 0)) * p.num_heads * D +
                  static_cast<int64_t>(kvh * G + g) * D;
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        float t[32];
        tmem_ld32(t_lane + Tm::O + ch * 32, t);
        if (row_valid && !failed) {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint4 v = make_uint4(pack_bf16x2(t[8 * c] * inv, t[8 * c + 1] * inv),
                                       pack_bf16x2(t[8 * c + 2] * inv, t[8 * c + 3] * inv),
                                       pack_bf16x2(t[8 * c + 4] * inv, t[8 * c + 5] * inv),
                                       pack_bf16x2(t[8 * c + 6] * inv, t[8 * c + 7] * inv));
            *reinterpret_cast<uint4 *>(dst + ch * 32 + 8 * c) = v;
          }
        }
      }
      tc_fence_before();  // O is overwritten by the next unit's first product after the unit barrier
    }
  }

  if (failed) flag_error(p.status, PA_FLAG_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, Tm::COLS);
}

template <int D, int G>
cudaError_t launch_prefill_tiles(const CUtensorMap &kmap, const CUtensorMap &vmap, const TileParams &tp, int sm_count,
                                 cudaStream_t stream) {
  constexpr int smem = TcLayout<D>::REQUEST;
  auto kern = prefill_tile_kernel<D, G>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  err = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);  // two CTAs per SM
  if (err != cudaSuccess) return err;
  int64_t grid = static_cast<int64_t>(sm_count) * 2;
  const int64_t units = static_cast<int64_t>(tp.max_tiles) * tp.num_kv_heads;
  if (grid > units) grid = units;
  if (grid < 1) grid = 1;
  return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(kTileThreads), smem, stream, kmap, vmap, tp);
}

#define PA_TILE_INST(DD, GG)                                                                                    \
  template cudaError_t launch_prefill_tiles<DD, GG>(const CUtensorMap &, const CUtensorMap &, const TileParams &, \
                                                    int, cudaStream_t);
PA_TILE_INST(128, 1)
PA_TILE_INST(128, 2)
PA_TILE_INST(128, 4)
PA_TILE_INST(128, 8)
PA_TILE_INST(64, 1)
PA_TILE_INST(64, 2)
PA_TILE_INST(64, 4)
PA_TILE_INST(64, 8)
#undef PA_TILE_INST

}  // namespace pa
