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
// One CTA (4 warps) handles one tile of 128 "packed rows" = (query position,
// head of the GQA group) pairs of one request and one KV head, so each K/V
// byte staged for the tile serves all G heads. Per tile of 64 keys:
//   1. one thread issues TMA loads of the 4 (block, KV head) tiles of K and
//      of V, read through the block table, into 128-byte-swizzled shared
//      memory (the same boxes as the decode path); K and V are double
//      buffered, and the next range is requested before this one is used;
//   2. one thread issues tcgen05.mma: S[128 x 64] = Q K^T into tensor memory;
//   3. every thread owns one row (its TMEM lane): it loads its 64 scores,
//      applies the causal limit, updates the running max and sum (log2
//      domain), and writes P as a bf16 hi + lo pair into shared memory in the
//      canonical K-major layout (hi over the consumed K tile);
//   4. one thread issues O += P_hi V + P_lo V (V is an MN-major operand); O
//      accumulates in tensor memory and a row is rescaled there only when its
//      running maximum grows by more than 2^8.
// One CTA barrier per key range; every other ordering goes through mbarriers.
// Two CTAs share an SM (112 KB of shared memory and 256 TMEM columns each at
// D = 128), so one CTA's softmax runs while the other's MMAs do. All shared
// state lives in the dynamic segment, whose start must be 1024-byte aligned
// for the swizzled tiles; the kernel checks that and reports otherwise. Waits on mbarriers are
// bounded; tensor memory is released on every exit path.
#include "attention_internal.cuh"

namespace pa {

constexpr int kTileRows = 128;                   // UMMA M
constexpr int kKeyTile = 64;                     // keys per KV tile (UMMA N of S, K of PV)
constexpr int kKeyTileCols = kKeyTile;           // TMEM columns of S
// Tensor memory per CTA: S in columns [0, 64), O_t in [64, 64 + D); a power of
// two >= 32. At most 512 columns exist per SM: D = 128 uses 256 (2 CTAs per
// SM by shared memory), D = 64 uses 128 (up to 4), so no CTA waits in alloc.
template <int D>
__host__ __device__ constexpr uint32_t tmem_cols() { return D + kKeyTileCols <= 128 ? 128u : 256u; }
constexpr uint64_t kTcWaitTimeoutNs = 2000000000;

template <int D>
struct TcLayout {
  static constexpr int HALVES = D / 64;                 // 64-element swizzle atoms along D
  static constexpr int Q_HALF = kTileRows * 128;        // 128 rows x 128 B
  static constexpr int KV_HALF = kKeyTile * 128;        // 64 rows x 128 B
  static constexpr int Q_BYTES = HALVES * Q_HALF;
  static constexpr int K_BYTES = HALVES * KV_HALF;
  static constexpr int P_BYTES = kTileRows * kKeyTile * 2;  // one 128-byte atom column
  static constexpr int KP_BYTES = K_BYTES > P_BYTES ? K_BYTES : P_BYTES;
  static constexpr int V_BYTES = HALVES * KV_HALF;
  static constexpr int Q_OFF = 0;
  static constexpr int KP_OFF = Q_OFF + Q_BYTES;     // two K buffers (P_hi overwrites the one in use)
  static constexpr int V_OFF = KP_OFF + 2 * KP_BYTES;  // two V buffers
  static constexpr int PLO_OFF = V_OFF + 2 * V_BYTES;
  static constexpr int BAR_OFF = PLO_OFF + P_BYTES;  // 2 TMA + 2 MMA barriers, TMEM base, unit
  static constexpr int BYTES = BAR_OFF + 64;
  // byte offset of 16-byte chunk c of row r in a swizzled tile with `half` bytes per atom column
  static __device__ __forceinline__ uint32_t off(int r, int c, int half) {
    return (c >> 3) * half + r * 128 + (((c & 7) ^ (r & 7)) << 4);
  }
};

template <int D, int G>
__global__ void __launch_bounds__(128, 2)
    prefill_tile_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                        const TileParams p) {
  using Lay = TcLayout<D>;
  constexpr int KSTEPS_S = D / 16;          // UMMA K steps of S = Q K^T
  constexpr int KSTEPS_O = kKeyTile / 16;   // UMMA K steps of O = P V
  constexpr int BLOCKS = kKeyTile / kBlockSize;
  constexpr uint32_t IDESC_S = f16_idesc(kTileRows, kKeyTile, 0);
  constexpr uint32_t IDESC_O = f16_idesc(kTileRows, D, 1);
  // O stays in TMEM and is rescaled only when a row's running maximum grows
  // by more than 2^8 (log2 domain); in between, probabilities are taken
  // against the older maximum and stay below 256.
  constexpr float kRescaleLog2 = 8.f;

  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const int tid = threadIdx.x, warp = tid >> 5;
  const uint32_t base = smem_u32(smem_raw);
  if (base & 1023u) {  // the swizzled tiles need 1024-byte alignment; never touch misaligned tiles
    if (tid == 0) flag_error(p.status, PA_FLAG_LENGTHS);
    return;
  }
  const uint32_t sQ = base + Lay::Q_OFF, sK0 = base + Lay::KP_OFF, sPlo = base + Lay::PLO_OFF;
  const uint32_t sV0 = base + Lay::V_OFF;
  const uint32_t bar_tma0 = base + Lay::BAR_OFF, bar_s = bar_tma0 + 16, bar_o = bar_tma0 + 24;
  uint32_t *tmem_base_s = reinterpret_cast<uint32_t *>(smem_raw + Lay::BAR_OFF + 32);
  int *unit_s = reinterpret_cast<int *>(smem_raw + Lay::BAR_OFF + 36);

  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_base_s), tmem_cols<D>());
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(bar_tma0, 1);
    mbar_init(bar_tma0 + 8, 1);
    mbar_init(bar_s, 1);
    mbar_init(bar_o, 1);
    prefetch_tmap(&kmap);
    prefetch_tmap(&vmap);
  }
  fence_mbar_init();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_base_s;
  const uint32_t t_lane = tmem + (static_cast<uint32_t>(warp * 32) << 16);  // this warp's TMEM lanes
  const uint32_t tS = t_lane, tO = t_lane + kKeyTile;
  griddep_wait();

  const int Hkv = p.num_kv_heads;
  const int total_units = min(max(ld_cg(p.tile_count), 0), p.max_tiles) * Hkv;
  uint32_t ph_tma[2] = {0, 0}, ph_s = 0, ph_o = 0;
  bool failed = false;  // this thread gave up on a wait; the CTA stops at its next barrier

  for (;;) {
    if (tid == 0) *unit_s = atomicAdd(p.tile_counter, 1);
    if (__syncthreads_or(failed)) break;
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

    // ---- Q tile: row r = (position r / G, head r % G), K-major, swizzled ----
    const int r = tid, qi = r / G, g = r % G;
    const bool row_valid = qi < npos;
    {
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
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};\n" ::"r"(sQ + Lay::off(r, c, Lay::Q_HALF)), "r"(w0),
                     "r"(w1), "r"(w2), "r"(w3)
                     : "memory");
      }
      fence_proxy_async_smem();  // the MMA reads Q through the async proxy
    }

    float m_used = -INFINITY, l = 0.f;
    const int lim = row_valid ? pos0 + qi + 1 : 0;  // keys j < lim are visible to this row
    const int nkt = (kv_end + kKeyTile - 1) / kKeyTile;

    // K and V of the 64-key range kt into buffer kt % 2 (thread 0 issues)
    auto load_range = [&](int kt) {
      const int buf = kt & 1;
      const uint32_t bar = bar_tma0 + 8 * buf;
      const uint32_t sK = sK0 + buf * Lay::KP_BYTES, sV = sV0 + buf * Lay::V_BYTES;
      mbar_arrive_expect_tx(bar, Lay::K_BYTES + Lay::V_BYTES);
#pragma unroll
      for (int blk = 0; blk < BLOCKS; ++blk) {
        const int kb = kt * BLOCKS + blk;
        int z = -kBlockSize;  // past the keys this tile needs: TMA fills zeros
        if (kb < nblk) {
          const int phys = __ldg(table + kb);
          if (phys >= 0 && phys < p.num_blocks)
            z = phys * kBlockSize;
          else
            flag_error(p.status, PA_FLAG_BLOCK_RANGE);
        }
#pragma unroll
        for (int h = 0; h < Lay::HALVES; ++h) {
          tma_load_3d(sK + h * Lay::KV_HALF + blk * 2048, &kmap, bar, h * 64, kvh, z);
          tma_load_3d(sV + h * Lay::KV_HALF + blk * 2048, &vmap, bar, h * 64, kvh, z);
        }
      }
    };
    if (tid == 0) load_range(0);

    for (int kt = 0; kt < nkt; ++kt) {
      const int key0 = kt * kKeyTile;
      const int buf = kt & 1;
      const uint32_t sKP = sK0 + buf * Lay::KP_BYTES, sV = sV0 + buf * Lay::V_BYTES;
      // 1. the other buffer is free once the previous P V product is done:
      //    request the next key range into it
      if (tid == 0) {
        if (kt > 0) failed |= !mbar_wait_bounded(bar_o, ph_o, kTcWaitTimeoutNs);
        if (kt + 1 < nkt) load_range(kt + 1);
      }
      failed |= !mbar_wait_bounded(bar_tma0 + 8 * buf, ph_tma[buf], kTcWaitTimeoutNs);
      ph_tma[buf] ^= 1;
      if (key0 + kKeyTile > kv_end) {
        // rows of keys past kv_end may hold anything (even NaN): zero them in V
        const int vr0 = kv_end - key0;
        const int n = (kKeyTile - vr0) * (D / 8);
        for (int i = tid; i < n; i += 128) {
          const int rr = vr0 + i / (D / 8), c = i % (D / 8);
          asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};\n" ::"r"(sV + Lay::off(rr, c, Lay::KV_HALF)),
                       "r"(0u)
                       : "memory");
        }
        fence_proxy_async_smem();  // ordered before the P V MMA by the barrier below
      }

      // 2. S = Q K^T into TMEM columns [0, 64)
      if (tid == 0) {
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < KSTEPS_S; ++ks) {
          const uint64_t a = sw128_desc(sQ + (ks >> 2) * Lay::Q_HALF + (ks & 3) * 32, 16, 1024);
          const uint64_t bd = sw128_desc(sKP + (ks >> 2) * Lay::KV_HALF + (ks & 3) * 32, 16, 1024);
          tc_mma_f16(tmem, a, bd, IDESC_S, ks > 0);
        }
        tc_commit(bar_s);
      }
      failed |= !mbar_wait_bounded(bar_s, ph_s, kTcWaitTimeoutNs);
      ph_s ^= 1;
      tc_fence_after();

      // 3. online softmax on this thread's row (one pass over the 64 scores)
      float x[kKeyTile];
      {
        float s0[32], s1[32];
        tmem_ld32(tS, s0);
        tmem_ld32(tS + 32, s1);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          x[i] = key0 + i < lim ? s0[i] * p.scale_log2 : -INFINITY;
          x[32 + i] = key0 + 32 + i < lim ? s1[i] * p.scale_log2 : -INFINITY;
        }
      }
      float mx = -INFINITY;
#pragma unroll
      for (int i = 0; i < kKeyTile; ++i) mx = fmaxf(mx, x[i]);
      // the previous P V product must be complete before O or P_lo change
      if (kt > 0) {
        failed |= !mbar_wait_bounded(bar_o, ph_o, kTcWaitTimeoutNs);
        ph_o ^= 1;
        tc_fence_after();
      }
      if (mx > -INFINITY && (m_used == -INFINITY || mx > m_used + kRescaleLog2)) {
        if (kt > 0 && m_used > -INFINITY) {
          const float alpha = ex2_approx(m_used - mx);
          l *= alpha;
#pragma unroll
          for (int ch = 0; ch < D / 32; ++ch) {
            float t[32];
            tmem_ld32(tO + ch * 32, t);
#pragma unroll
            for (int i = 0; i < 32; ++i) t[i] *= alpha;
            tmem_st32(tO + ch * 32, t);
          }
        }
        m_used = mx;
      }
      const float ms = m_used == -INFINITY ? 0.f : m_used;
      float rs = 0.f;
#pragma unroll
      for (int c = 0; c < kKeyTile / 8; ++c) {  // 8 keys = one 16-byte chunk of P
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float p0 = ex2_approx(x[8 * c + 2 * e] - ms);
          const float p1 = ex2_approx(x[8 * c + 2 * e + 1] - ms);
          rs += p0 + p1;
          hi[e] = pack_bf16x2(p0, p1);
          lo[e] = pack_bf16x2(p0 - bf16_lo(hi[e]), p1 - bf16_hi(hi[e]));
        }
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};\n" ::"r"(sKP + Lay::off(r, c, Lay::P_BYTES)),
                     "r"(hi[0]), "r"(hi[1]), "r"(hi[2]), "r"(hi[3])
                     : "memory");
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};\n" ::"r"(sPlo + Lay::off(r, c, Lay::P_BYTES)),
                     "r"(lo[0]), "r"(lo[1]), "r"(lo[2]), "r"(lo[3])
                     : "memory");
      }
      l += rs;
      fence_proxy_async_smem();
      tc_fence_before();
      if (__syncthreads_or(failed)) {
        failed = true;
        break;
      }

      // 4. O += P_hi V + P_lo V in TMEM columns [64, 64 + D)
      if (tid == 0) {
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < KSTEPS_O; ++ks) {
          const uint64_t vd = sw128_desc(sV + ks * 2048, Lay::KV_HALF, 1024);
          tc_mma_f16(tmem + kKeyTile, sw128_desc(sKP + ks * 32, 16, 1024), vd, IDESC_O, (kt > 0 || ks > 0) ? 1u : 0u);
          tc_mma_f16(tmem + kKeyTile, sw128_desc(sPlo + ks * 32, 16, 1024), vd, IDESC_O, 1);
        }
        tc_commit(bar_o);
      }
    }
    if (failed) break;

    // ---- epilogue: wait for the last P V product, normalise, store this row ----
    failed |= !mbar_wait_bounded(bar_o, ph_o, kTcWaitTimeoutNs);
    ph_o ^= 1;
    tc_fence_after();
    const float inv = l > 0.f ? 1.f / l : 0.f;
    bf16 *dst = p.out + static_cast<int64_t>(row0 + (row_valid ? qi : 0)) * p.num_heads * D +
                static_cast<int64_t>(kvh * G + g) * D;
#pragma unroll
    for (int ch = 0; ch < D / 32; ++ch) {
      float t[32];
      tmem_ld32(tO + ch * 32, t);
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
    tc_fence_before();  // O is overwritten by the next unit's first product after the next barrier
  }

  if (failed && tid == 0) flag_error(p.status, PA_FLAG_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, tmem_cols<D>());
}

template <int D, int G>
cudaError_t launch_prefill_tiles(const CUtensorMap &kmap, const CUtensorMap &vmap, const TileParams &tp, int sm_count,
                                 cudaStream_t stream) {
  constexpr int smem = TcLayout<D>::BYTES;
  auto kern = prefill_tile_kernel<D, G>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  err = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);  // two CTAs per SM
  if (err != cudaSuccess) return err;
  int64_t grid = static_cast<int64_t>(sm_count) * 2;
  const int64_t units = static_cast<int64_t>(tp.max_tiles) * tp.num_kv_heads;
  if (grid > units) grid = units;
  if (grid < 1) grid = 1;
  return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(128), smem, stream, kmap, vmap, tp);
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
