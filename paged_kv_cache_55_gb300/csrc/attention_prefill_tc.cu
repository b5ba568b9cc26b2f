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
// One CTA handles one tile of 256 "packed rows" = (query position, head of
// the GQA group) pairs of one request and one KV head, as two halves A and B
// of 128 rows (the UMMA M) that share every K/V range staged for the tile, so
// each K/V byte serves 2 x 128 rows. The keys are walked in ranges of 128 (an
// M128 x N128 product runs at close to the tensor cores' peak; N64 at half)
// by three kinds of warps that hand work over through mbarriers only:
//   * a producer warp issues TMA loads of the (block, KV head) tiles of K and
//     V through the block table into 128-byte-swizzled shared memory (the
//     decode path's boxes), into one ring of K(0), V(0), K(1), V(1), ...
//     (as many 128-key slots as shared memory holds: five at D = 128), each
//     slot with full/empty barriers, so loads run two ranges ahead;
//   * an MMA warp issues tcgen05.mma. Each half owns one score buffer in
//     tensor memory: S(r) = Q K(r)^T lands there, the softmax overwrites it
//     in place with P(r), and O += P_hi(r) V(r) + P_lo(r) V(r) reads P from
//     there (V an MN-major shared-memory operand). The order is P V_A(r),
//     S_A(r+1) once that product has completed, P V_B(r), S_B(r+1): while one
//     half's softmax runs, the tensor cores work on the other half. The warp
//     zeroes V rows past the last key before the first product reads them;
//   * eight softmax warps, four per half, own one row each per thread (its
//     TMEM lane). Per range they read the 128 scores once, 32 at a time,
//     apply the causal limit, keep the running max and sum (log2 domain) and
//     write P as bf16 hi + lo pairs over the scores they came from. O
//     accumulates in tensor memory; O, the row sum and the probabilities
//     already written are rescaled (by the whole warp, each row by its own
//     factor) only when a row's running maximum grows by more than 2^8; no
//     product is in flight then. The softmax warps of TMEM lanes 0-31 share
//     a scheduler with the MMA warp, whose issue rate the tensor cores depend
//     on, so their arithmetic is kept lean (paired fp32 instructions).
// Half A holds the earlier positions, so it may stop some ranges before half
// B (its keys end sooner); a half without valid rows does no work at all.
// One CTA per SM (all 512 TMEM columns, 256 per half). All shared state is in
// the dynamic segment, whose start must be 1024-byte aligned for the swizzled
// tiles (checked). Waits on mbarriers are bounded (a thread waits out at most
// one timeout, then runs to the unit barrier); in-flight loads and products
// are waited for (bounded) and tensor memory is released on every exit path.
#include <type_traits>

#include "attention_internal.cuh"

namespace pa {

constexpr int kHalfRows = 128;  // UMMA M: rows per half
constexpr int kHalves = kPrefillTileRows / kHalfRows;
static_assert(kHalves == 2, "the pipeline interleaves exactly two halves");
constexpr int kKeyTile = 128;  // keys per range (UMMA N of S, K of P V)
constexpr int kMaxSlots = 8;   // K/V ring slots (as many as shared memory holds)
constexpr int kSoftmaxWarps = 4 * kHalves, kMmaWarp = kSoftmaxWarps, kTmaWarp = kSoftmaxWarps + 1;
constexpr int kTileThreads = 32 * (kTmaWarp + 1);
// 8-bit caches: two more warps widen each staged range to fp16 in place.
constexpr int kConvWarp = kTmaWarp + 1, kConvWarps = 2;
constexpr int kTileThreads8 = kTileThreads + 32 * kConvWarps;
constexpr int kRawBoxRows = 32;  // 8-bit boxes: min(block_size, 32) rows
constexpr uint64_t kTcWaitTimeoutNs = 2000000000;
constexpr uint32_t kTmemCols = 512;

// Tensor memory columns of half A: the score buffer SP [0, 128) and O
// [128, 128 + D); half B's are the same plus HALF. SP holds S (fp32, column
// = key) and then P: the 16 keys of UMMA K step k occupy columns [16k, 16k+16)
// of either, as 8 columns of P_hi pairs followed by 8 of P_lo pairs.
template <int D>
struct TcTmem {
  static constexpr uint32_t SP = 0, O = kKeyTile;
  static constexpr uint32_t HALF = kTmemCols / kHalves;
  static_assert(O + D <= HALF, "a half's columns must fit its share of TMEM");
};

template <int D>
struct TcLayout {
  // 64-element swizzle atoms along D; head_dim 80 or 96 is padded to two, the
  // columns past it zero-filled by TMA (K, V) and never read (Q)
  static constexpr int ATOMS = (D + 63) / 64;
  static constexpr int Q_ATOM = kHalfRows * 128;   // 128 rows x 128 B
  static constexpr int KV_ATOM = kKeyTile * 128;   // 128 keys x 128 B
  static constexpr int Q_BYTES = ATOMS * Q_ATOM;   // Q of one half
  static constexpr int KV_BYTES = ATOMS * KV_ATOM;             // one K or V range: a ring slot
  static constexpr int TABLE_ENTRIES = 512;  // staged TMA row coordinates: boxes of keys < 8192 (4096 at bs 8)
  // barriers: full[kMaxSlots], empty[kMaxSlots], per half s_full, p_full, o_done,
  // then q_full and drain (the MMA thread's last commit), then raw[kMaxSlots]
  // (8-bit caches: the staged codes of a slot have landed)
  static constexpr int NBARS = 3 * kMaxSlots + 3 * kHalves + 2;
  static constexpr int FIXED = kHalves * Q_BYTES + TABLE_ENTRIES * 4 + 8 * NBARS + 16;
  static constexpr int FIT = (227 * 1024 - FIXED) / KV_BYTES;
  static constexpr int SLOTS = FIT < kMaxSlots ? FIT : kMaxSlots;
  static_assert(SLOTS >= 4, "the ring holds at least K and V of two ranges");
  static constexpr int Q_OFF = 0;                                // Q of halves A and B
  static constexpr int RING_OFF = Q_OFF + kHalves * Q_BYTES;     // K(0), V(0), K(1), V(1), ... in SLOTS slots
  static constexpr int TABLE_OFF = RING_OFF + SLOTS * KV_BYTES;  // the unit's box coordinates
  static constexpr int BAR_OFF = TABLE_OFF + TABLE_ENTRIES * 4;
  static constexpr int BYTES = BAR_OFF + 8 * NBARS + 16;
  // Shared memory requested per CTA: more than half an SM's, so that a second
  // CTA (which would wait for TMEM) never lands on the same SM.
  static constexpr int REQUEST = BYTES > 116 * 1024 ? BYTES : 116 * 1024;
  // byte offset of 16-byte chunk c of row r in a swizzled tile with `atom` bytes per atom column
  static __device__ __forceinline__ uint32_t off(int r, int c, int atom) {
    return (c >> 3) * atom + r * 128 + (((c & 7) ^ (r & 7)) << 4);
  }
};
static_assert(TcLayout<128>::BYTES <= 227 * 1024, "shared memory of one CTA");

// Bounded wait that is skipped once this thread has given up: a thread waits
// out at most one timeout, then runs to the next unit barrier.
__device__ __forceinline__ void wait_or_fail(uint32_t bar, uint32_t parity, bool &failed) {
  if (!failed) failed = !mbar_wait_bounded(bar, parity, kTcWaitTimeoutNs);
}

// The two 32-bit words of a 128-byte-swizzle shared-memory descriptor (the
// layout sw128_desc builds). The low word holds the start address >> 4 in
// bits 0-13, so a tile's descriptors differ from its first one by adding the
// byte offset >> 4 to the low word (shared addresses stay below 256 KB: no
// carry out of the field). Building them once per unit keeps the issuing
// thread at two additions per MMA: it shares its scheduler with two softmax
// warps, and the tensor core queues only a couple of instructions.
__device__ __forceinline__ uint32_t desc_lo(uint32_t smem_addr, uint32_t lbo) {
  return ((smem_addr & 0x3FFFFu) >> 4) | (((lbo >> 4) & 0x3FFFu) << 16);
}
__host__ __device__ constexpr uint32_t desc_hi(uint32_t sbo) {
  return ((sbo >> 4) & 0x3FFFu) | (1u << 14) | (2u << 29);  // SBO, version (bit 46), 128-byte swizzle (61-63)
}
// D[tmem] (+)= A[smem] * B[smem] with descriptors given as words; ACC = 0 overwrites D.
template <int ACC>
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint32_t a_lo, uint32_t a_hi, uint32_t b_lo, uint32_t b_hi,
                                       uint32_t idesc) {
  asm volatile(
      "{\n .reg .pred p;\n .reg .b64 a, b;\n setp.ne.b32 p, %6, 0;\n mov.b64 a, {%1, %2};\n"
      " mov.b64 b, {%3, %4};\n tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %5, p;\n}\n" ::"r"(d_tmem),
      "r"(a_lo), "r"(a_hi), "r"(b_lo), "r"(b_hi), "r"(idesc), "n"(ACC)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem].
template <int ACC>
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t b_hi, uint32_t idesc) {
  asm volatile(
      "{\n .reg .pred p;\n .reg .b64 b;\n setp.ne.b32 p, %5, 0;\n mov.b64 b, {%2, %3};\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], b, %4, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "r"(b_lo), "r"(b_hi), "r"(idesc), "n"(ACC)
      : "memory");
}

// 64 consecutive 32-bit columns of this thread's TMEM lane; the wait is in
// the same statement, so no use of the registers can be scheduled before it.
__device__ __forceinline__ void tmem_ld64_wait(uint32_t taddr, uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
}

// The same for 32 columns.
__device__ __forceinline__ void tmem_ld32_wait(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

// The same for 16 columns.
__device__ __forceinline__ void tmem_ld16_wait(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// Packed pairs of fp32 operations (one instruction for two lanes of data).
__device__ __forceinline__ void fma2(float &d0, float &d1, float a0, float a1, float b0, float b1, float c0, float c1) {
  asm("{\n .reg .b64 a, b, c, d;\n mov.b64 a, {%2, %3};\n mov.b64 b, {%4, %5};\n mov.b64 c, {%6, %7};\n"
      " fma.rn.f32x2 d, a, b, c;\n mov.b64 {%0, %1}, d;\n}\n"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}
__device__ __forceinline__ void add2(float &d0, float &d1, float a0, float a1, float b0, float b1) {
  asm("{\n .reg .b64 a, b, d;\n mov.b64 a, {%2, %3};\n mov.b64 b, {%4, %5};\n add.rn.f32x2 d, a, b;\n"
      " mov.b64 {%0, %1}, d;\n}\n"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
__device__ __forceinline__ void sub2(float &d0, float &d1, float a0, float a1, float b0, float b1) {
  asm("{\n .reg .b64 a, b, d;\n mov.b64 a, {%2, %3};\n mov.b64 b, {%4, %5};\n sub.rn.f32x2 d, a, b;\n"
      " mov.b64 {%0, %1}, d;\n}\n"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Row maximum of 32 raw scores, key ck0 + i visible while ck0 + i < lim.
__device__ __forceinline__ float masked_max32(const uint32_t (&s)[32], int ck0, int lim) {
  float m = -INFINITY;
  if (ck0 + 32 <= lim) {
    // a tree of depth 4 (a chain of 16 three-input maxima would be 16 deep)
    float t[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      t[i] = max3(__uint_as_float(s[4 * i]), __uint_as_float(s[4 * i + 1]),
                  fmaxf(__uint_as_float(s[4 * i + 2]), __uint_as_float(s[4 * i + 3])));
    m = max3(max3(t[0], t[1], t[2]), max3(t[3], t[4], t[5]), fmaxf(t[6], t[7]));
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) m = ck0 + i < lim ? fmaxf(m, __uint_as_float(s[i])) : m;
  }
  return m;
}

// P for 32 keys (scores s[0..32), visible while ck0 + i < lim): p =
// 2^(s * sl2 - ms), summed into *sum and packed as the TMEM columns of two
// UMMA K steps. SPLIT (bf16 operands, 8 significant bits): P as a hi + lo
// pair, 32 columns [hi pairs of keys 0-15, lo pairs of 0-15, hi 16-31, lo
// 16-31]; otherwise (fp16, 11 bits: a weight's relative rounding error of
// at most 2^-11 moves the output by at most 2^-11 max|V|, and far less when
// the roundings are independent) one pair per two keys, 16 columns.
// The exponent is one fused multiply-add, whose unrounded product differs
// from the rounded one ms was taken from by at most half an ulp of ms: below
// 2^-12 while |ms| <= 2^12. EXACT rows (larger |ms|) round the product first,
// so the row maximum's exponent is exactly zero and none exceeds the growth
// the caller allowed.
template <typename E, bool EXACT, bool SPLIT>
__device__ __forceinline__ void probs32(const uint32_t (&s)[32], int ck0, int lim, float sl2, float ms, float &sum,
                                        uint32_t (&u)[32]) {
  const bool full = ck0 + 32 <= lim;
  float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    float x0 = __uint_as_float(s[2 * i]), x1 = __uint_as_float(s[2 * i + 1]);
    if (!full) {
      x0 = ck0 + 2 * i < lim ? x0 : -INFINITY;
      x1 = ck0 + 2 * i + 1 < lim ? x1 : -INFINITY;
    }
    float e0, e1;
    if (EXACT) {
      // scalar round-to-nearest intrinsics, which are never merged into a fused multiply-add
      e0 = __fsub_rn(__fmul_rn(x0, sl2), ms);
      e1 = __fsub_rn(__fmul_rn(x1, sl2), ms);
    } else {
      fma2(e0, e1, x0, x1, sl2, sl2, -ms, -ms);
    }
    const float p0 = ex2_approx(e0), p1 = ex2_approx(e1);
    add2(acc0, acc1, acc0, acc1, p0, p1);
    const uint32_t hi = E::pack(p0, p1);
    if (SPLIT) {
      float l0, l1;
      sub2(l0, l1, p0, p1, E::lo(hi), E::hi(hi));
      const int step = i >> 3, k = i & 7;
      u[16 * step + k] = hi;
      u[16 * step + 8 + k] = E::pack(l0, l1);
    } else {
      u[i] = hi;
    }
  }
  sum += acc0 + acc1;
}

// Multiply the probabilities already stored in a 32-column chunk of P (the
// layout probs32 writes) by alpha, re-splitting each into hi + lo.
// The same for a chunk of single pairs (16 columns).
template <typename E>
__device__ __forceinline__ void rescale_p16(uint32_t taddr, float alpha) {
  uint32_t w[16];
  tmem_ld16_wait(taddr, w);
#pragma unroll
  for (int i = 0; i < 16; ++i) w[i] = E::pack(E::lo(w[i]) * alpha, E::hi(w[i]) * alpha);
  tmem_st16u(taddr, w);
}

template <typename E>
__device__ __forceinline__ void rescale_p32(uint32_t taddr, float alpha) {
  uint32_t w[32];
  tmem_ld32_wait(taddr, w);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int hk = 16 * (i >> 3) + (i & 7);
    const float p0 = (E::lo(w[hk]) + E::lo(w[hk + 8])) * alpha;
    const float p1 = (E::hi(w[hk]) + E::hi(w[hk + 8])) * alpha;
    const uint32_t hi = E::pack(p0, p1);
    w[hk] = hi;
    w[hk + 8] = E::pack(p0 - E::lo(hi), p1 - E::hi(hi));
  }
  tmem_st32u(taddr, w);
}

// 8-bit caches (KV8): the producer stages a range's codes in the back half of
// its ring slot (kKeyTile x D bytes, the TMA boxes' own 128- or 64-byte
// swizzle); two converter warps load them, meet at a named barrier (the
// fp16 rows they then write overlap the codes), widen them exactly to fp16
// in the layout the 16-bit path's TMA writes, and arrive on the slot's full
// barrier. The tensor cores then take fp16 operands whatever q is: a bf16 Q
// row is stored as fp16, scaled first by a power of two when its largest |q|
// reaches 2^15, and its thread's softmax factor is scaled back.
template <int D, int G, typename E, bool KV8>
// Ten warps (twelve with 8-bit caches): three share each of two (all four) of
// the SM's register-file partitions, so a thread gets at most 168 registers.
__global__ void __launch_bounds__(KV8 ? kTileThreads8 : kTileThreads, 1)
    prefill_tile_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                        const TileParams p) {
  using Lay = TcLayout<D>;
  using Tm = TcTmem<D>;
  using M = typename std::conditional<KV8, ElemFp16, E>::type;  // tensor-core operand type
  constexpr bool SPLIT = std::is_same<M, ElemBf16>::value;      // P as a hi + lo pair (bf16 operands only)
  constexpr int PCOLS = SPLIT ? 32 : 16;                        // TMEM columns of P per 32 keys
  constexpr int NTHREADS = KV8 ? kTileThreads8 : kTileThreads;
  constexpr int RAW_ROW = D <= 64 ? 64 : 128;      // bytes per staged row of codes (padded past head_dim)
  constexpr int RAW_BYTES = kKeyTile * RAW_ROW;    // 8-bit codes of one range
  constexpr uint32_t RAW_OFF = Lay::KV_BYTES / 2;  // staged in the back half of the slot
  static_assert(RAW_BYTES == Lay::KV_BYTES / 2, "a range's codes fill half of its 16-bit slot");
  constexpr int KSTEPS_S = D / 16;         // UMMA K steps of S = Q K^T
  constexpr int KSTEPS_O = kKeyTile / 16;  // UMMA K steps of O = P V
  constexpr int TILES = kKeyTile / kTileKeys;  // 16-key tiles per range
  constexpr int POS_PER_HALF = kHalfRows / G;
  constexpr uint32_t IDESC_S = f16_idesc(kHalfRows, kKeyTile, 0, M::kUmmaFormat);
  constexpr uint32_t IDESC_O = f16_idesc(kHalfRows, D, 1, M::kUmmaFormat);
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
  constexpr int SLOTS = Lay::SLOTS;
  const uint32_t sQ0 = base + Lay::Q_OFF, sRing = base + Lay::RING_OFF;
  const uint32_t bars = base + Lay::BAR_OFF;
  const uint32_t bar_full = bars, bar_empty = bars + 8 * kMaxSlots;  // per ring slot: barrier + 8 * slot
  // per half h: barrier + 8 * h
  const uint32_t bar_s = bars + 16 * kMaxSlots, bar_p = bar_s + 8 * kHalves, bar_o = bar_p + 8 * kHalves;
  const uint32_t bar_q = bar_o + 8 * kHalves, bar_drain = bar_q + 8;
  const uint32_t bar_raw = bar_drain + 8;  // per ring slot: barrier + 8 * slot
  uint32_t *tmem_base_s = reinterpret_cast<uint32_t *>(smem_raw + Lay::BAR_OFF + 8 * Lay::NBARS);
  int *unit_s = reinterpret_cast<int *>(smem_raw + Lay::BAR_OFF + 8 * Lay::NBARS + 4);
  int *zbox = reinterpret_cast<int *>(smem_raw + Lay::TABLE_OFF);

  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_base_s), kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    // full: the producer's TMA (16-bit caches) or one arrival per converter warp (8-bit); empty: MMA commits
    for (int i = 0; i < kMaxSlots; ++i) mbar_init(bar_full + 8 * i, KV8 ? kConvWarps : 1);
    for (int i = 0; i < kMaxSlots; ++i) mbar_init(bar_empty + 8 * i, 1);
    for (int i = 0; i < kMaxSlots; ++i) mbar_init(bar_raw + 8 * i, 1);
    for (int h = 0; h < kHalves; ++h) {
      mbar_init(bar_s + 8 * h, 1);
      mbar_init(bar_p + 8 * h, 4);  // the half's four softmax warps
      mbar_init(bar_o + 8 * h, 1);
    }
    mbar_init(bar_q, kSoftmaxWarps);
    mbar_init(bar_drain, 1);
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
  // Phase bookkeeping (it runs on across units, like the barriers). Each
  // half's s_full, p_full and o_done complete once per range of that half,
  // so range r of a unit is phase ph[h] + r. The ring carries K(0), V(0),
  // K(1), V(1), ... of every unit in turn: load number g = ring0 + 2 r (+1
  // for V) sits in slot g % SLOTS as that slot's use g / SLOTS.
  uint32_t ph[kHalves] = {0, 0};
  uint32_t ring0 = 0;
  uint32_t issued = 0;  // producer: loads actually issued
  uint32_t n_q = 0;
  bool failed = false;

  for (;;) {
    if (tid == 0) *unit_s = atomicAdd(p.tile_counter, 1);
    if (__syncthreads_or(failed)) break;  // unit barrier: every role is done with the last unit
    const int u = *unit_s;
    if (u >= total_units) break;
    const int item = u / Hkv, kvh = u - item * Hkv;
    (void)RAW_OFF;
    const int4 r0 = ld_cg(p.tiles + 2 * item);
    const int4 r1 = ld_cg(p.tiles + 2 * item + 1);
    const int b = r0.x, row0 = r0.y, npos = r0.z, pos0 = r0.w, kv_end = r1.y;
    const bool sane = b >= 0 && b < p.num_seqs && npos >= 1 && npos <= kPrefillTileRows / G && row0 >= 0 &&
                      row0 + npos <= p.total_q && pos0 >= 0 && kv_end == pos0 + npos &&
                      kv_end <= static_cast<int64_t>(p.max_blocks_per_seq) * p.block_size;
    if (!sane) {
      if (tid == 0) flag_error(p.status, PA_FLAG_LENGTHS);
      __syncthreads();  // unit_s is rewritten next iteration
      continue;
    }
    const int32_t *table = p.block_tables + static_cast<int64_t>(b) * p.max_blocks_per_seq;
    const int bs = p.block_size;
    // A TMA box is box_rows consecutive keys of one block (16, or 8 with
    // 8-token blocks). The cache row of box i's first key, k = i * box_rows,
    // is table[k / bs] * bs + k % bs (powers of two: shift and mask); boxes
    // past the keys, or of a block id out of range, are read at -box_rows
    // (zero fill). All threads compute the unit's coordinates once here, so
    // the producer only reads one from shared memory per box.
    constexpr int MAXROWS = KV8 ? kRawBoxRows : kTileKeys;
    const int box_rows = bs < MAXROWS ? bs : MAXROWS;
    const int nboxes = (kv_end + box_rows - 1) / box_rows;
    auto box_z = [&](int i) {
      const int key = i * box_rows;
      if (key >= kv_end) return -box_rows;
      const int phys = __ldg(table + (key >> p.block_shift));
      if (phys < 0 || phys >= p.num_blocks) {
        flag_error(p.status, PA_FLAG_BLOCK_RANGE);
        return -box_rows;
      }
      return (phys << p.block_shift) + (key & (bs - 1));
    };
    const int nkt = (kv_end + kKeyTile - 1) / kKeyTile;
    // key ranges each half needs: up to its last valid position (0 = no valid rows)
    int nkt_h[kHalves];
#pragma unroll
    for (int h = 0; h < kHalves; ++h) {
      const int last = min(npos, (h + 1) * POS_PER_HALF);  // positions [h * POS_PER_HALF, last)
      nkt_h[h] = last > h * POS_PER_HALF ? (pos0 + last + kKeyTile - 1) / kKeyTile : 0;
    }
    for (int i = tid; i < min(nboxes, Lay::TABLE_ENTRIES); i += NTHREADS) zbox[i] = box_z(i);
    __syncthreads();

    if (warp == kTmaWarp) {
      // ---------------- producer: K(j+1) ahead of V(j) ----------------
      if (lane == 0) {
        auto load = [&](int kt, bool is_v) {
          const uint32_t g = ring0 + 2 * kt + (is_v ? 1 : 0);
          const uint32_t slot = g % SLOTS, use = g / SLOTS;
          if (use > 0) wait_or_fail(bar_empty + 8 * slot, (use - 1) & 1u, failed);
          if (failed) return;
          issued = g + 1;
          const void *map = is_v ? static_cast<const void *>(&vmap) : static_cast<const void *>(&kmap);
          if constexpr (KV8) {
            // the range's codes: kKeyTile / box_rows boxes of box_rows x D bytes
            const uint32_t bar = bar_raw + 8 * slot;
            const uint32_t dst = sRing + slot * Lay::KV_BYTES + RAW_OFF;
            mbar_arrive_expect_tx(bar, RAW_BYTES);
            const int nb = kKeyTile / box_rows;
            for (int j = 0; j < nb; ++j) {
              const int i = kt * nb + j;
              const int z = i < nboxes ? (i < Lay::TABLE_ENTRIES ? zbox[i] : box_z(i)) : -box_rows;
              tma_load_3d(dst + j * box_rows * RAW_ROW, map, bar, 0, kvh, z);
            }
            return;
          }
          const uint32_t bar = bar_full + 8 * slot;
          const uint32_t dst = sRing + slot * Lay::KV_BYTES;
          mbar_arrive_expect_tx(bar, Lay::KV_BYTES);
          // a 16-key tile is one 16-row box (16- or 32-token blocks) or two
          // 8-row boxes of consecutive 8-token blocks
          auto boxes = [&](auto nbox_c) {
            constexpr int NBOX = decltype(nbox_c)::value, ROWS = kTileKeys / NBOX;
#pragma unroll
            for (int tile = 0; tile < TILES; ++tile) {
#pragma unroll
              for (int j = 0; j < NBOX; ++j) {
                const int i = (kt * TILES + tile) * NBOX + j;
                const int z = i < nboxes ? (i < Lay::TABLE_ENTRIES ? zbox[i] : box_z(i)) : -ROWS;
#pragma unroll
                for (int a = 0; a < Lay::ATOMS; ++a)
                  tma_load_3d(dst + a * Lay::KV_ATOM + tile * 2048 + j * ROWS * 128, map, bar, a * 64, kvh, z);
              }
            }
          };
          if constexpr (!KV8) {
            if (bs < kTileKeys)
              boxes(std::integral_constant<int, 2>());
            else
              boxes(std::integral_constant<int, 1>());
          }
        };
        // the order the products consume them: S(j) needs K(j) before P V(j) needs V(j)
        for (int j = 0; j < nkt; ++j) {
          load(j, false);
          load(j, true);
        }
      }
    } else if (warp >= kConvWarp) {
      // ---------------- 8-bit caches: widen staged codes to fp16 in place ----------------
      if constexpr (KV8) {
        // Lane l of converter warp w takes 16-byte code chunk c of rows
        // r0 + l % 8, so the eight lanes of one shared-memory phase touch eight
        // rows at one chunk: distinct bank groups in both swizzled layouts.
        constexpr int CPR = RAW_ROW / 16;      // code chunks per staged row (zeros past head_dim)
        constexpr int ROWS_PASS = 8 * (8 / CPR);  // rows per pass of the 64 threads
        constexpr int PASSES = kKeyTile / ROWS_PASS;
        const int ct = (warp - kConvWarp) * 32 + lane;
        const int q8 = ct >> 3, c = q8 % CPR, rsub = (q8 / CPR) * 8 + (ct & 7);
        for (int j = 0; j < 2 * nkt; ++j) {
          const uint32_t g = ring0 + j;
          const uint32_t slot = g % SLOTS, use = g / SLOTS;
          wait_or_fail(bar_raw + 8 * slot, use & 1u, failed);
          const uint32_t sbase = sRing + slot * Lay::KV_BYTES;
          uint4 codes[PASSES];
          if (!failed) {
#pragma unroll
            for (int i = 0; i < PASSES; ++i) {
              const int r = i * ROWS_PASS + rsub;
              const uint32_t a = sbase + RAW_OFF + (RAW_ROW == 128 ? r * 128 + (((c ^ r) & 7) << 4)
                                                                     : r * 64 + (((c ^ (r >> 1)) & 3) << 4));
              asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];\n"
                           : "=r"(codes[i].x), "=r"(codes[i].y), "=r"(codes[i].z), "=r"(codes[i].w)
                           : "r"(a));
            }
          }
          // every code of the slot is in registers before any fp16 row overwrites them
          asm volatile("bar.sync 1, %0;\n" ::"n"(32 * kConvWarps) : "memory");
          if (!failed) {
#pragma unroll
            for (int i = 0; i < PASSES; ++i) {
              const int r = i * ROWS_PASS + rsub;
              const uint32_t w[4] = {codes[i].x, codes[i].y, codes[i].z, codes[i].w};
              uint32_t h[8];
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                asm("{\n .reg .b16 l, u;\n mov.b32 {l, u}, %2;\n cvt.rn.f16x2.e4m3x2 %0, l;\n"
                    " cvt.rn.f16x2.e4m3x2 %1, u;\n}\n"
                    : "=r"(h[2 * k]), "=r"(h[2 * k + 1])
                    : "r"(w[k]));
              }
              // codes d = 16c .. 16c + 15 -> fp16 chunks 2c (d .. d + 7) and 2c + 1
              asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};\n" ::"r"(sbase + Lay::off(r, 2 * c, Lay::KV_ATOM)),
                           "r"(h[0]), "r"(h[1]), "r"(h[2]), "r"(h[3])
                           : "memory");
              asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};\n" ::"r"(
                               sbase + Lay::off(r, 2 * c + 1, Lay::KV_ATOM)),
                           "r"(h[4]), "r"(h[5]), "r"(h[6]), "r"(h[7])
                           : "memory");
            }
            fence_proxy_async_smem();  // the MMA reads the slot through the async proxy
          }
          __syncwarp();
          if (lane == 0 && !failed) mbar_arrive(bar_full + 8 * slot);
        }
      }
    } else if (warp == kMmaWarp) {
      // ---------------- MMA issue ----------------
      // The whole warp follows the loop (it zeroes the tail of the last V
      // range); lane 0 alone issues tensor-core work and commits. Range r is
      // read by the halves with r < nkt_h: the first of them waits for the
      // K/V loads, the last one's commit releases the buffers.
      auto first_reader = [&](int kt) { return kt < nkt_h[0] ? 0 : 1; };
      auto last_reader = [&](int kt) { return kt < nkt_h[1] ? 1 : 0; };
      // ring slot of K(kt) (v = 0) or V(kt) (v = 1), and the parity of its full barrier
      auto slot_of = [&](int kt, int v) { return (ring0 + 2 * kt + v) % SLOTS; };
      auto full_parity = [&](int kt, int v) { return ((ring0 + 2 * kt + v) / SLOTS) & 1u; };
      constexpr uint32_t DHI = desc_hi(1024);
      const uint32_t q_lo0 = desc_lo(sQ0, 16), q_lo1 = desc_lo(sQ0 + Lay::Q_BYTES, 16);
      const uint32_t k_lo = desc_lo(sRing, 16), v_lo = desc_lo(sRing, Lay::KV_ATOM);  // slot 0
      constexpr uint32_t SLOT_STEP = Lay::KV_BYTES >> 4;                            // per slot
      static_assert(kHalves == 2, "descriptor words are kept for two halves");
      auto mma_s = [&](int kt, int h) {
        if (lane == 0 && !failed) {
          tc_fence_after();
          const uint32_t klo = k_lo + slot_of(kt, 0) * SLOT_STEP, qlo = h ? q_lo1 : q_lo0;
          const uint32_t d = tmem + h * Tm::HALF + Tm::SP;
          mma_ss<0>(d, qlo, DHI, klo, DHI, IDESC_S);
#pragma unroll
          for (int ks = 1; ks < KSTEPS_S; ++ks) {
            const uint32_t qo = ((ks >> 2) * Lay::Q_ATOM + (ks & 3) * 32) >> 4;
            const uint32_t ko = ((ks >> 2) * Lay::KV_ATOM + (ks & 3) * 32) >> 4;
            mma_ss<1>(d, qlo + qo, DHI, klo + ko, DHI, IDESC_S);
          }
          tc_commit(bar_s + 8 * h);
          if (h == last_reader(kt)) tc_commit(bar_empty + 8 * slot_of(kt, 0));
        }
        __syncwarp();
      };
      wait_or_fail(bar_q, n_q & 1u, failed);
      ++n_q;
      if (nkt > 0) {
        wait_or_fail(bar_full + 8 * slot_of(0, 0), full_parity(0, 0), failed);
#pragma unroll
        for (int h = 0; h < kHalves; ++h)
          if (nkt_h[h] > 0) mma_s(0, h);
      }
      for (int kt = 0; kt < nkt; ++kt) {
        const uint32_t vslot = slot_of(kt, 1);
#pragma unroll
        for (int h = 0; h < kHalves; ++h) {
          if (kt >= nkt_h[h]) continue;
          wait_or_fail(bar_p + 8 * h, (ph[h] + kt) & 1u, failed);  // P(kt) is in place
          if (h == first_reader(kt)) {
            wait_or_fail(bar_full + 8 * vslot, full_parity(kt, 1), failed);
            const int key0 = kt * kKeyTile;
            if (!failed && key0 + kKeyTile > kv_end) {
              // rows of keys past kv_end may hold anything (even NaN): zero them in V
              const uint32_t sV = sRing + vslot * Lay::KV_BYTES;
              const int vr0 = kv_end - key0;
              const int n = (kKeyTile - vr0) * (D / 8);
              for (int i = lane; i < n; i += 32) {
                const int rr = vr0 + i / (D / 8), c = i % (D / 8);
                asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};\n" ::"r"(sV + Lay::off(rr, c, Lay::KV_ATOM)),
                             "r"(0u)
                             : "memory");
              }
              fence_proxy_async_smem();
            }
            __syncwarp();
          }
          if (lane == 0 && !failed) {
            tc_fence_after();
            const uint32_t vlo = v_lo + vslot * SLOT_STEP;
            const uint32_t t = tmem + h * Tm::HALF;
            // K step ks reads P at columns PCOLS / 2 * ks (+ 8 for the lo half of a pair)
            if (kt == 0)
              mma_ts<0>(t + Tm::O, t + Tm::SP, vlo, DHI, IDESC_O);  // the unit's first product overwrites O
            else
              mma_ts<1>(t + Tm::O, t + Tm::SP, vlo, DHI, IDESC_O);
            if (SPLIT) mma_ts<1>(t + Tm::O, t + Tm::SP + 8, vlo, DHI, IDESC_O);
#pragma unroll
            for (int ks = 1; ks < KSTEPS_O; ++ks) {
              const uint32_t vo = (ks * 2048) >> 4;  // 16 keys x 128 B per K step
              mma_ts<1>(t + Tm::O, t + Tm::SP + (PCOLS / 2) * ks, vlo + vo, DHI, IDESC_O);
              if (SPLIT) mma_ts<1>(t + Tm::O, t + Tm::SP + 16 * ks + 8, vlo + vo, DHI, IDESC_O);
            }
            tc_commit(bar_o + 8 * h);
            if (h == last_reader(kt)) tc_commit(bar_empty + 8 * vslot);
          }
          __syncwarp();
          if (kt + 1 < nkt_h[h]) {
            if (h == first_reader(kt + 1))
              wait_or_fail(bar_full + 8 * slot_of(kt + 1, 0), full_parity(kt + 1, 0), failed);
            wait_or_fail(bar_o + 8 * h, (ph[h] + kt) & 1u, failed);  // P V(kt) has read P(kt)
            mma_s(kt + 1, h);
          }
        }
      }
    } else {
      // ---------------- softmax: one row per thread (its TMEM lane) ----------------
      const int h = warp / 4;
      const int r = tid % kHalfRows;  // row within the half = TMEM lane
      const uint32_t t_lane = tmem + h * Tm::HALF + (static_cast<uint32_t>((warp % 4) * 32) << 16);
      const int qi = h * POS_PER_HALF + r / G, g = r % G;
      const bool row_valid = qi < npos;
      const int nk = nkt_h[h];
      float sl2 = p.scale_log2;  // > 0: the max of raw scores gives the max of scaled ones
      {  // Q of the half: row r = (position, head), K-major, swizzled
        const uint32_t sQ = sQ0 + h * Lay::Q_BYTES;
        const bf16 *qrow =
            p.q + static_cast<int64_t>(row0 + (row_valid ? qi : 0)) * p.q_stride + static_cast<int64_t>(kvh * G + g) * D;
        // q is only required to be 4-byte aligned: 16-byte loads when rows allow them
        const bool q16 = (reinterpret_cast<uintptr_t>(p.q) & 15u) == 0 && (p.q_stride & 7) == 0;
        auto load_q = [&](int c) {
          uint4 w = make_uint4(0u, 0u, 0u, 0u);
          if (row_valid) {
            if (q16) {
              w = __ldg(reinterpret_cast<const uint4 *>(qrow) + c);
            } else {
              const uint32_t *q32 = reinterpret_cast<const uint32_t *>(qrow) + 4 * c;
              w = make_uint4(__ldg(q32), __ldg(q32 + 1), __ldg(q32 + 2), __ldg(q32 + 3));
            }
          }
          return w;
        };
        // bf16 rows over 8-bit caches: 2^-e, e > 0 only when the row's largest |q| reaches 2^15
        float qmul = 1.f;
        if constexpr (KV8 && std::is_same<E, ElemBf16>::value) {
          float amax = 0.f;
#pragma unroll 4
          for (int c = 0; c < D / 8; ++c) {
            const uint4 w = load_q(c);
            const uint32_t v[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int k = 0; k < 4; ++k)
              amax = fmaxf(amax, fmaxf(fabsf(ElemBf16::lo(v[k])), fabsf(ElemBf16::hi(v[k]))));
          }
          const int ex = static_cast<int>((__float_as_uint(amax) >> 23) & 0xffu) - 127;  // floor(log2(amax))
          const int e = ex >= 15 ? min(ex - 14, 120) : 0;
          qmul = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
          sl2 *= __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
        }
#pragma unroll 4
        for (int c = 0; c < D / 8; ++c) {
          uint4 w = load_q(c);
          if constexpr (KV8 && std::is_same<E, ElemBf16>::value) {
            w = make_uint4(ElemFp16::pack(ElemBf16::lo(w.x) * qmul, ElemBf16::hi(w.x) * qmul),
                           ElemFp16::pack(ElemBf16::lo(w.y) * qmul, ElemBf16::hi(w.y) * qmul),
                           ElemFp16::pack(ElemBf16::lo(w.z) * qmul, ElemBf16::hi(w.z) * qmul),
                           ElemFp16::pack(ElemBf16::lo(w.w) * qmul, ElemBf16::hi(w.w) * qmul));
          }
          asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};\n" ::"r"(sQ + Lay::off(r, c, Lay::Q_ATOM)),
                       "r"(w.x), "r"(w.y), "r"(w.z), "r"(w.w)
                       : "memory");
        }
        fence_proxy_async_smem();  // the MMA reads Q through the async proxy
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_q);
      }
      float m_used = -INFINITY, l = 0.f;
      const int lim = row_valid ? pos0 + qi + 1 : 0;  // keys j < lim are visible to this row
      for (int kt = 0; kt < nk; ++kt) {
        const int key0 = kt * kKeyTile;
        const uint32_t sp = t_lane + Tm::SP;
        wait_or_fail(bar_s + 8 * h, (ph[h] + kt) & 1u, failed);
        tc_fence_after();
        // One pass over the range, 32 keys at a time: each chunk's maximum is
        // checked against the running one before its probabilities are taken.
        // One pass over the range, 32 keys at a time: each chunk's maximum is
        // checked against the running one before its probabilities are taken.
        float sum = 0.f;     // this range's probabilities, against m_used
        float alpha = 1.f;   // factor owed by O and l for growth within this range
#pragma unroll 1
        for (int c = 0; c < kKeyTile / 32; ++c) {
          const int ck0 = key0 + 32 * c;
          uint32_t sv[32], u[32];
          tmem_ld32_wait(sp + 32 * c, sv);
          // The chunk's maximum, rounded, and its growth over m_used, as separately
          // rounded operations (no contraction into one fused multiply-add): the
          // exponents below are bounded by exactly this difference.
          const float cm = __fmul_rn(sl2, masked_max32(sv, ck0, lim));
          const bool grow = cm > -INFINITY && (m_used == -INFINITY || __fsub_rn(cm, m_used) > kRescaleLog2);
          if (__any_sync(0xffffffffu, grow)) {
            // The row's maximum grew past the threshold (always in a row's
            // first visible chunk, rarely after): what was taken against the
            // old maximum (this range's sum and stored chunks, and O and l)
            // is scaled by 2^(old - new). TMEM accesses are warp-wide, so the
            // warp does it together (factor 1 in rows that did not grow).
            const float a = grow && m_used > -INFINITY ? ex2_approx(__fsub_rn(m_used, cm)) : 1.f;
            if (grow) m_used = cm;
            sum *= a;
            alpha *= a;
            if (c > 0) {
              tmem_wait_st();  // the chunks stored so far are read back
#pragma unroll 1
              for (int cc = 0; cc < c; ++cc) {
                if constexpr (SPLIT)
                  rescale_p32<M>(sp + 32 * cc, a);
                else
                  rescale_p16<M>(sp + 16 * cc, a);
              }
            }
          }
          const float ms = m_used == -INFINITY ? 0.f : m_used;
          if (__any_sync(0xffffffffu, fabsf(ms) > 4096.f))
            probs32<M, true, SPLIT>(sv, ck0, lim, sl2, ms, sum, u);
          else
            probs32<M, false, SPLIT>(sv, ck0, lim, sl2, ms, sum, u);
          // P over the scores it came from (single pairs: chunk c at columns 16c, over
          // scores of chunks <= c that have been read already)
          if constexpr (SPLIT) {
            tmem_st32u(sp + 32 * c, u);
          } else {
            uint32_t u16[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) u16[i] = u[i];
            tmem_st16u(sp + 16 * c, u16);
          }
        }
        // O holds P V(0 .. kt-1), all complete (S(kt) was issued after the
        // last of them finished).
        if (kt > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
          for (int ch = 0; ch < (D + 31) / 32; ++ch) {  // head_dim 80: also 16 unused columns
            uint32_t t[32];
            tmem_ld32_wait(t_lane + Tm::O + ch * 32, t);
#pragma unroll
            for (int i = 0; i < 32; ++i) t[i] = __float_as_uint(__uint_as_float(t[i]) * alpha);
            tmem_st32u(t_lane + Tm::O + ch * 32, t);
          }
        }
        l = l * alpha + sum;
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_p + 8 * h);
      }
      if (nk > 0) {
        // epilogue: the half's last P V product, normalised
        wait_or_fail(bar_o + 8 * h, (ph[h] + nk - 1) & 1u, failed);
        tc_fence_after();
        const float inv = l > 0.f ? p.out_scale / l : 0.f;
        bf16 *dst = p.out + static_cast<int64_t>(row0 + (row_valid ? qi : 0)) * p.num_heads * D +
                    static_cast<int64_t>(kvh * G + g) * D;
#pragma unroll
        for (int ch = 0; ch < (D + 31) / 32; ++ch) {
          uint32_t t[32];
          tmem_ld32_wait(t_lane + Tm::O + ch * 32, t);
          if (row_valid && !failed) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              if (32 * ch + 8 * c >= D) continue;  // head_dim 80: the last 16 columns are padding
              const float *f = reinterpret_cast<const float *>(&t[8 * c]);
              const uint4 v = make_uint4(E::pack(f[0] * inv, f[1] * inv), E::pack(f[2] * inv, f[3] * inv),
                                         E::pack(f[4] * inv, f[5] * inv), E::pack(f[6] * inv, f[7] * inv));
              *reinterpret_cast<uint4 *>(dst + ch * 32 + 8 * c) = v;
            }
          }
        }
      }
      tc_fence_before();  // O is overwritten by the next unit's first product after the unit barrier
    }
    // every role advances the phase bookkeeping alike
#pragma unroll
    for (int hh = 0; hh < kHalves; ++hh) ph[hh] += nkt_h[hh];
    ring0 += 2 * nkt;
  }

  // Every thread left the loop at the same unit barrier. Before tensor memory
  // and shared memory go away, wait (bounded) for work still in flight: the
  // MMA thread's products (one last commit) and, after a timeout, the
  // producer's loads that no product consumed (loads into a buffer complete
  // in order, so waiting for the last one issued suffices).
  if (warp == kMmaWarp && lane == 0) {
    tc_commit(bar_drain);
    if (!mbar_wait_bounded(bar_drain, 0, kTcWaitTimeoutNs)) failed = true;
  }
  if (warp == kTmaWarp && lane == 0) {
    const uint32_t landed = KV8 ? bar_raw : bar_full;  // where the loads' completion is counted
    for (uint32_t g = issued > SLOTS ? issued - SLOTS : 0; g < issued; ++g)
      if (!mbar_wait_bounded(landed + 8 * (g % SLOTS), (g / SLOTS) & 1u, kTcWaitTimeoutNs)) failed = true;
  }
  if (failed) flag_error(p.status, PA_FLAG_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

template <int D, int G, typename E, bool KV8>
cudaError_t launch_prefill_tiles(const CUtensorMap &kmap, const CUtensorMap &vmap, const TileParams &tp, int sm_count,
                                 cudaStream_t stream) {
  constexpr int smem = TcLayout<D>::REQUEST;
  auto kern = prefill_tile_kernel<D, G, E, KV8>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  err = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (err != cudaSuccess) return err;
  int64_t grid = sm_count;  // one CTA per SM: it holds all of the SM's tensor memory
  const int64_t units = static_cast<int64_t>(tp.max_tiles) * tp.num_kv_heads;
  if (grid > units) grid = units;
  if (grid < 1) grid = 1;
  return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(KV8 ? kTileThreads8 : kTileThreads), smem, stream,
                    kmap, vmap, tp);
}

#define PA_TILE_INST1(DD, GG, EE, K8)                                                                   \
  template cudaError_t launch_prefill_tiles<DD, GG, EE, K8>(const CUtensorMap &, const CUtensorMap &,     \
                                                            const TileParams &, int, cudaStream_t);
#define PA_TILE_INST(DD, GG)                                                                              \
  PA_TILE_INST1(DD, GG, ElemBf16, false)                                                                  \
  PA_TILE_INST1(DD, GG, ElemFp16, false)                                                                  \
  PA_TILE_INST1(DD, GG, ElemBf16, true)                                                                   \
  PA_TILE_INST1(DD, GG, ElemFp16, true)
PA_TILE_INST(128, 1)
PA_TILE_INST(128, 2)
PA_TILE_INST(128, 4)
PA_TILE_INST(128, 8)
PA_TILE_INST(64, 1)
PA_TILE_INST(64, 2)
PA_TILE_INST(64, 4)
PA_TILE_INST(64, 8)
PA_TILE_INST(96, 1)
PA_TILE_INST(96, 2)
PA_TILE_INST(96, 4)
PA_TILE_INST(96, 8)
PA_TILE_INST(80, 1)
PA_TILE_INST(80, 2)
PA_TILE_INST(80, 4)
PA_TILE_INST(80, 8)
#undef PA_TILE_INST
#undef PA_TILE_INST1

}  // namespace pa
