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
// One CTA per SM runs a stream of units. A unit is a tile of 256 "packed
// rows" = (query position, head of the GQA group) pairs of one request and
// one KV head, as two halves A and B of 128 rows (the UMMA M) that share
// every K/V range staged for the tile, so each K/V byte serves 2 x 128 rows.
// The keys are walked in ranges of 128 (an M128 x N128 product runs at close
// to the tensor cores' peak; N64 at half) by warps that hand work over
// through mbarriers only (every wait bounded):
//   * a producer warp claims units from the global queue and publishes each
//     in a two-slot record ring, then issues TMA loads of its K and V ranges
//     through the block table into one ring of K(0), V(0), K(1), V(1), ...
//     (five 32 KB slots at D = 128), running on into the next unit while the
//     current one finishes: a unit's first loads are in flight before the
//     previous unit's last products. K arrives as per-atom boxes of 16 rows
//     (the K-major operand wants rows 128 bytes apart); at head_dim 128, V
//     arrives one box per cache block holding both 64-element atoms (4-D
//     tensor map), fewer and larger boxes, which the TMA engine moves faster;
//   * an MMA warp issues tcgen05.mma. Each half owns one score buffer in
//     tensor memory: S(r) = Q K(r)^T lands there, the softmax overwrites it
//     in place with P(r), and O += P(r) V(r) reads P from there (V an
//     MN-major shared-memory operand). The order is P V_A(r), S_A(r+1),
//     P V_B(r), S_B(r+1): while one half's softmax runs, the tensor cores
//     work on the other half. S_A(r+1) is issued right behind P V_A(r),
//     whose operand it overwrites: the products one thread issues execute in
//     issue order, and the commit that signals S_A(r+1) complete also covers
//     every product issued before it. The warp zeroes V rows past the last
//     key before the first product reads them (over bf16 caches the
//     converter warps do);
//   * two converter warps rewrite staged ranges in place: 8-bit codes widened
//     exactly to fp16, and bf16 V rewritten as fp16 so that P can be one
//     fp16 value per key (a range holding a magnitude of 65536 or more goes
//     back to bf16 and takes a bf16 hi + lo pair for P);
//   * sixteen softmax warps, two per TMEM lane quadrant and half: each thread
//     owns one row (its TMEM lane) and 64 of the 128 keys of every range,
//     whose probabilities it computes in a loop of K steps that reads 16
//     scores from TMEM each (a small hot loop: the twenty warps share the
//     SM's instruction cache). The
//     two warps of a row exchange their maxima through shared memory (an
//     mbarrier pair), so both take the range's probabilities against the
//     same running maximum; each keeps its own partial row sum, rescales its
//     own half of O, and writes its own half of the output. O accumulates in
//     tensor memory and is rescaled only when a row's maximum grows by more
//     than 2^8. At the end of a unit the warps load the next unit's Q (its
//     record is already published) before they write the current output, so
//     the next unit's first product overlaps this unit's epilogue.
// Half A holds the earlier positions, so it may stop some ranges before half
// B (its keys end sooner); a half without valid rows does no work at all.
// One CTA per SM (all 512 TMEM columns, 256 per half). All shared state is in
// the dynamic segment, whose start must be 1024-byte aligned for the swizzled
// tiles (checked). On a timeout the warp records it, stops, and the kernel
// waits (bounded) for its loads and products in flight before it releases
// tensor memory. Head dim 256 has its own one-half kernel at the end of the
// file (S and O of two halves would not fit the 512 TMEM columns).
#include <type_traits>

#include "attention_internal.cuh"

namespace pa {

constexpr int kHalfRows = 128;  // UMMA M: rows per half
constexpr int kHalves = kPrefillTileRows / kHalfRows;
static_assert(kHalves == 2, "the pipeline interleaves exactly two halves");
constexpr int kParts = 2;        // softmax warps per TMEM lane quadrant and half (64 keys of a range each)
constexpr int kKeyTile = 128;    // keys per range (UMMA N of S, K of P V)
constexpr int kMaxSlots = 8;     // K/V ring slots (as many as shared memory holds)
constexpr int kUnitSlots = 2;    // published unit records
// Warp roles. The MMA warp is warp 0: its issue rate sets the tensor cores'
// (they queue only a couple of products) and it shares a scheduler with
// softmax warps; the schedulers favour lower-numbered warps when several are
// ready. Warp 1 loads K/V; warps 2 and 3 widen 8-bit codes (idle otherwise);
// warps 4 .. 19 run the softmax (warp % 4 is their TMEM lane quadrant).
constexpr int kSoftmaxWarps = 4 * kHalves * kParts, kMmaWarp = 0, kTmaWarp = 1, kSoftmaxWarp0 = 4;
constexpr int kTileThreads = 32 * (kSoftmaxWarp0 + kSoftmaxWarps);
// 8-bit caches: two more warps widen each staged range to fp16 in place.
constexpr int kConvWarp = 2, kConvWarps = 2;
constexpr int kTileThreads8 = kTileThreads;
constexpr int kRawBoxRows = 32;  // 8-bit boxes: min(block_size, 32) rows
constexpr uint64_t kTcWaitTimeoutNs = 2000000000;
constexpr uint32_t kTmemCols = 512;

// Tensor memory columns of half A: the score buffer SP [0, 128) and O
// [128, 128 + D); half B's are the same plus HALF. SP holds S (fp32, column
// = key) and then P. With P as a bf16 hi + lo pair, the 16 keys of UMMA K
// step k occupy columns [16k, 16k + 16) (8 columns of hi pairs, then 8 of lo
// pairs); with one 16-bit P per key, K step k occupies 8 columns at 8k for
// k < 4 and at 8k + 32 for k >= 4, so that each softmax warp's probabilities
// stay inside the 64 score columns it reads (the other warp of its row may
// still be reading its own).
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
  // mbarriers (8 bytes each): per ring slot full, empty, raw (8-bit codes
  // landed; bf16 caches: V range g % kMaxSlots put back to bf16) and conv
  // (8-bit caches: both converter warps hold a slot's codes; bf16 caches: V
  // range g % kMaxSlots rewritten); per half s
  // (S complete), p (P written), o (P V complete), qf (Q stored), qe (the MMA
  // warp has seen qf); per unit slot uf (record published), ue (record read);
  // per (half, lane quadrant) the softmax pair's exchange; drain
  static constexpr int B_FULL = 0, B_EMPTY = kMaxSlots, B_RAW = 2 * kMaxSlots, B_CONV = 3 * kMaxSlots;
  static constexpr int B_S = 4 * kMaxSlots, B_P = B_S + kHalves, B_O = B_P + kHalves, B_QF = B_O + kHalves;
  static constexpr int B_QE = B_QF + kHalves, B_UF = B_QE + kHalves, B_UE = B_UF + kUnitSlots;
  static constexpr int B_X = B_UE + kUnitSlots, B_DRAIN = B_X + 4 * kHalves, NBARS = B_DRAIN + 1;
  static constexpr int XCH_BYTES = kHalves * kParts * kHalfRows * 4;  // one float per (half, part, row)
  static constexpr int UNIT_BYTES = kUnitSlots * 32;                  // records of eight ints
  static constexpr int VF_BYTES = kMaxSlots * 8;                      // per V range and converter warp: kept bf16
  static constexpr int FIXED = kHalves * Q_BYTES + XCH_BYTES + UNIT_BYTES + VF_BYTES + 8 * NBARS + 16;
  static constexpr int FIT = (227 * 1024 - FIXED) / KV_BYTES;
  static constexpr int SLOTS = FIT < kMaxSlots ? FIT : kMaxSlots;
  static_assert(SLOTS >= 4, "the ring holds at least K and V of two ranges");
  static constexpr int Q_OFF = 0;                                // Q of halves A and B
  static constexpr int RING_OFF = Q_OFF + kHalves * Q_BYTES;     // K(0), V(0), K(1), V(1), ... in SLOTS slots
  static constexpr int XCH_OFF = RING_OFF + SLOTS * KV_BYTES;    // the softmax pairs' exchange
  static constexpr int UNIT_OFF = XCH_OFF + XCH_BYTES;           // unit records
  static constexpr int VF_OFF = UNIT_OFF + UNIT_BYTES;           // V range flags (bf16 V rewritten as fp16)
  static constexpr int BAR_OFF = VF_OFF + VF_BYTES;
  static constexpr int TMEM_OFF = BAR_OFF + 8 * NBARS;
  static constexpr int BYTES = TMEM_OFF + 16;
  // Shared memory requested per CTA: more than half an SM's, so that a second
  // CTA (which would wait for TMEM) never lands on the same SM.
  static constexpr int REQUEST = BYTES > 116 * 1024 ? BYTES : 116 * 1024;
  // byte offset of 16-byte chunk c of row r in a swizzled tile with `atom` bytes per atom column
  static __device__ __forceinline__ uint32_t off(int r, int c, int atom) {
    return (c >> 3) * atom + r * 128 + (((c & 7) ^ (r & 7)) << 4);
  }
};
static_assert(TcLayout<128>::BYTES <= 227 * 1024, "shared memory of one CTA");
static_assert(TcLayout<128>::SLOTS >= 5, "loads run two ranges ahead at head_dim 128");

// Bounded wait by a whole warp; the outcome is made warp-uniform, so a warp
// that gives up leaves its loops together (no lane is left inside a
// warp-collective instruction). A warp waits out at most one timeout.
__device__ __forceinline__ void wait_warp(uint32_t bar, uint32_t parity, bool &failed) {
  if (!failed) failed = !mbar_wait_bounded(bar, parity, kTcWaitTimeoutNs);
  failed = __any_sync(0xffffffffu, failed);
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

// 32 consecutive 32-bit columns of this thread's TMEM lane; the wait is in
// the same statement, so no use of the registers can be scheduled before it.
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

// Store 8 32-bit columns (raw bits) of this thread's TMEM lane.
__device__ __forceinline__ void tmem_st8u(uint32_t taddr, const uint32_t (&v)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};\n" ::"r"(taddr), "r"(v[0]),
      "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
      : "memory");
}

// P for the 16 keys of one UMMA K step (scores s[0..16), key k0 + i visible
// while k0 + i < lim): p = 2^(s * sl2 - ms), summed into *sum and stored at
// TMEM column `col` of this thread's lane. SPLIT (bf16 P, 8 significant
// bits): a hi + lo pair per key, 8 columns of hi pairs then 8 of lo pairs;
// otherwise (fp16, 11 bits: a weight's relative rounding error of at most
// 2^-11 moves the output by at most 2^-11 max|V|, and far less when the
// roundings are independent) 8 columns, one pair of keys each. The exponent
// is one fused multiply-add, whose unrounded product differs from the
// rounded one ms was taken from by at most half an ulp of ms: below 2^-12
// while |ms| <= 2^12. EXACT rows (larger |ms|) round the product first (scalar
// round-to-nearest intrinsics, never merged into a fused multiply-add), so the
// row maximum's exponent is exactly zero and none exceeds the growth the
// caller allowed.
template <typename E, bool EXACT, bool SPLIT>
__device__ __forceinline__ void probs16_store(const uint32_t *s, int k0, int lim, float sl2, float ms, float &sum,
                                              uint32_t col) {
  const bool full = k0 + 16 <= lim;
  float acc0 = 0.f, acc1 = 0.f;
  uint32_t hv[8], lv[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float x0 = __uint_as_float(s[2 * i]), x1 = __uint_as_float(s[2 * i + 1]);
    if (!full) {
      x0 = k0 + 2 * i < lim ? x0 : -INFINITY;
      x1 = k0 + 2 * i + 1 < lim ? x1 : -INFINITY;
    }
    float e0, e1;
    if (EXACT) {
      e0 = __fsub_rn(__fmul_rn(x0, sl2), ms);
      e1 = __fsub_rn(__fmul_rn(x1, sl2), ms);
    } else {
      fma2(e0, e1, x0, x1, sl2, sl2, -ms, -ms);
    }
    const float p0 = ex2_approx(e0), p1 = ex2_approx(e1);
    add2(acc0, acc1, acc0, acc1, p0, p1);
    hv[i] = E::pack(p0, p1);
    if (SPLIT) {
      float l0, l1;
      sub2(l0, l1, p0, p1, E::lo(hv[i]), E::hi(hv[i]));
      lv[i] = E::pack(l0, l1);
    }
  }
  sum += acc0 + acc1;
  tmem_st8u(col, hv);
  if (SPLIT) tmem_st8u(col + 8, lv);
}

// P of one softmax warp's 64 keys of a range, from column sp of its lane,
// the scores read again from TMEM 32 at a time (P of the first 32 keys never
// covers the columns of the second). PAIR: a bf16 hi + lo pair per key, 16
// columns per UMMA K step in place; else one fp16 P per key, 8 columns per
// K step from sp. The rare cases (exact exponents, a bf16 V range) take this
// path; the common one is the loop in the kernel.
template <bool PAIR>
__device__ __forceinline__ void range_probs(uint32_t sp, int ck0, int lim, float sl2, float ms, bool exact,
                                            float &sum) {
  using PT = typename std::conditional<PAIR, ElemBf16, ElemFp16>::type;
  constexpr uint32_t PSTEP = PAIR ? 16 : 8;
  uint32_t s0[32], s1[32];
  tmem_ld32_wait(sp, s0);
  if (exact) {
    probs16_store<PT, true, PAIR>(s0, ck0, lim, sl2, ms, sum, sp);
    probs16_store<PT, true, PAIR>(s0 + 16, ck0 + 16, lim, sl2, ms, sum, sp + PSTEP);
  } else {
    probs16_store<PT, false, PAIR>(s0, ck0, lim, sl2, ms, sum, sp);
    probs16_store<PT, false, PAIR>(s0 + 16, ck0 + 16, lim, sl2, ms, sum, sp + PSTEP);
  }
  tmem_ld32_wait(sp + 32, s1);
  if (exact) {
    probs16_store<PT, true, PAIR>(s1, ck0 + 32, lim, sl2, ms, sum, sp + 2 * PSTEP);
    probs16_store<PT, true, PAIR>(s1 + 16, ck0 + 48, lim, sl2, ms, sum, sp + 3 * PSTEP);
  } else {
    probs16_store<PT, false, PAIR>(s1, ck0 + 32, lim, sl2, ms, sum, sp + 2 * PSTEP);
    probs16_store<PT, false, PAIR>(s1 + 16, ck0 + 48, lim, sl2, ms, sum, sp + 3 * PSTEP);
  }
}

// Two 32-column loads of this thread's TMEM lane, then one wait.
__device__ __forceinline__ void tmem_ld32x2_wait(uint32_t taddr, uint32_t (&a)[32], uint32_t (&b)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n"
      : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]), "=r"(a[7]), "=r"(a[8]), "=r"(a[9]), "=r"(a[10]), "=r"(a[11]), "=r"(a[12]), "=r"(a[13]), "=r"(a[14]), "=r"(a[15]), "=r"(a[16]), "=r"(a[17]), "=r"(a[18]), "=r"(a[19]), "=r"(a[20]), "=r"(a[21]), "=r"(a[22]), "=r"(a[23]), "=r"(a[24]), "=r"(a[25]), "=r"(a[26]), "=r"(a[27]), "=r"(a[28]), "=r"(a[29]), "=r"(a[30]), "=r"(a[31])
      : "r"(taddr)
      : "memory");
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3]), "=r"(b[4]), "=r"(b[5]), "=r"(b[6]), "=r"(b[7]), "=r"(b[8]), "=r"(b[9]), "=r"(b[10]), "=r"(b[11]), "=r"(b[12]), "=r"(b[13]), "=r"(b[14]), "=r"(b[15]), "=r"(b[16]), "=r"(b[17]), "=r"(b[18]), "=r"(b[19]), "=r"(b[20]), "=r"(b[21]), "=r"(b[22]), "=r"(b[23]), "=r"(b[24]), "=r"(b[25]), "=r"(b[26]), "=r"(b[27]), "=r"(b[28]), "=r"(b[29]), "=r"(b[30]), "=r"(b[31])
      : "r"(taddr + 32)
      : "memory");
}

// A published unit: a tile of one request and one KV head, or the end of the stream.
struct TileUnit {
  int b, row0, npos, pos0, kv_end, kvh, stop;
};

// A bf16 V range in shared memory, rewritten by the two converter warps:
// converter warp w takes its 16-byte chunks c = w * PER * 32 + lane + 32 i
// (i < PER); the chunk at byte offset o holds key row key_of(o), and with
// MASKED rows at or past nvalid are not the request's keys (they are zeroed).
// A chunk all of whose values have magnitudes below 65536 (bf16 bits
// 0x4780: no larger bf16 value rounds to a finite fp16 one; inf and NaN come
// after it) is rewritten as fp16; the others stay bf16. Returns bit i set for
// each chunk i that stayed bf16.
template <int PER, bool MASKED, typename Mask, typename KeyOf>
__device__ __forceinline__ Mask vrange_to_fp16(uint32_t sV, int c0, int nvalid, KeyOf key_of) {
  constexpr int BATCH = 8;
  static_assert(PER <= 8 * static_cast<int>(sizeof(Mask)) && PER % BATCH == 0, "a bit per chunk, whole batches");
  Mask kept = 0;
  // One batch of code, not unrolled: the twenty warps' hot loops share the
  // SM's instruction cache, and unrolling this loop four times made the
  // whole kernel 20 % slower.
#pragma unroll 1
  for (int b0 = 0; b0 < PER; b0 += BATCH) {
    uint4 w[BATCH];
#pragma unroll
    for (int i = 0; i < BATCH; ++i)
      asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];\n"
                   : "=r"(w[i].x), "=r"(w[i].y), "=r"(w[i].z), "=r"(w[i].w)
                   : "r"(sV + 16u * static_cast<uint32_t>(c0 + 32 * (b0 + i))));
#pragma unroll
    for (int i = 0; i < BATCH; ++i) {
      const uint32_t o = 16u * static_cast<uint32_t>(c0 + 32 * (b0 + i));
      const uint4 v = w[i];
      const uint32_t m = __vmaxu2(__vmaxu2(v.x & 0x7fff7fffu, v.y & 0x7fff7fffu),
                                  __vmaxu2(v.z & 0x7fff7fffu, v.w & 0x7fff7fffu));
      const bool big = max(m >> 16, m & 0xffffu) >= 0x4780u;
      const bool zero = MASKED && key_of(o) >= nvalid;
      uint4 h = make_uint4(0u, 0u, 0u, 0u);
      if (!zero)
        h = make_uint4(ElemFp16::pack(bf16_lo(v.x), bf16_hi(v.x)), ElemFp16::pack(bf16_lo(v.y), bf16_hi(v.y)),
                       ElemFp16::pack(bf16_lo(v.z), bf16_hi(v.z)), ElemFp16::pack(bf16_lo(v.w), bf16_hi(v.w)));
      if (zero || !big)
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};\n" ::"r"(sV + o), "r"(h.x), "r"(h.y), "r"(h.z),
                     "r"(h.w)
                     : "memory");
      else
        kept |= static_cast<Mask>(1) << (b0 + i);
    }
  }
  return kept;
}

// Back to bf16: the chunks vrange_to_fp16 rewrote (not in `kept`, not
// zeroed). Exact for every value of magnitude 2^-17 or more (and zero); a
// smaller one comes back within 2^-25 of the value it was.
template <int PER, bool MASKED, typename Mask, typename KeyOf>
__device__ __forceinline__ void vrange_back_to_bf16(uint32_t sV, int c0, int nvalid, Mask kept, KeyOf key_of) {
#pragma unroll 4
  for (int i = 0; i < PER; ++i) {
    const uint32_t o = 16u * static_cast<uint32_t>(c0 + 32 * i);
    if (((kept >> i) & 1u) || (MASKED && key_of(o) >= nvalid)) continue;
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];\n"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(sV + o));
    v = make_uint4(pack_bf16x2(ElemFp16::lo(v.x), ElemFp16::hi(v.x)), pack_bf16x2(ElemFp16::lo(v.y), ElemFp16::hi(v.y)),
                   pack_bf16x2(ElemFp16::lo(v.z), ElemFp16::hi(v.z)), pack_bf16x2(ElemFp16::lo(v.w), ElemFp16::hi(v.w)));
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};\n" ::"r"(sV + o), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
  }
}

// 8-bit caches (KV8): the producer stages a range's codes in the back half of
// its ring slot (kKeyTile x D bytes, the TMA boxes' own 128- or 64-byte
// swizzle); two converter warps load them, meet at the slot's conv barrier
// (the fp16 rows they then write overlap the codes), widen them exactly to
// fp16 in the layout the 16-bit path's TMA writes, and arrive on the slot's
// full barrier. The tensor cores then take fp16 operands whatever q is: a
// bf16 Q row is stored as fp16, scaled first by a power of two when its
// largest |q| reaches 2^15, and its row's softmax factor is scaled back.
//
// bf16 caches (VCONV): S takes bf16 Q and K as they are; V is rewritten as
// fp16 in place, so that P is one fp16 value per key (11 significant bits)
// instead of a bf16 hi + lo pair, halving the P V products. Each V range is
// rewritten by both converter warps in one pass: every value of magnitude
// below 65536 is an fp16 value (exactly so from 2^-17 up, within 2^-25
// below). A range holding a larger magnitude (or inf, NaN) is put back to
// bf16 and its flags send the softmax warps and the MMA warp to the hi + lo
// pair for that range. Either way the rows past the unit's last key are
// zeroed.
template <int D, int G, typename E, bool KV8>
// Twenty warps (two of them idle over fp16 caches), one CTA per SM.
__global__ void __launch_bounds__(KV8 ? kTileThreads8 : kTileThreads, 1)
    prefill_tile_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                        const __grid_constant__ CUtensorMap vmapb, const TileParams p) {
  using Lay = TcLayout<D>;
  using Tm = TcTmem<D>;
  using M = typename std::conditional<KV8, ElemFp16, E>::type;  // operand type of S = Q K^T
  constexpr bool VCONV = !KV8 && std::is_same<E, ElemBf16>::value;  // bf16 V rewritten as fp16
  // P and V are fp16 in every case but a bf16 range that does not fit fp16 (P then a bf16 hi + lo pair)
  // V staged one cache block per box, both atoms (4-D map): 16-bit caches at head_dim 128
  constexpr bool VBLK = D == 128 && !KV8;
  constexpr int NTHREADS = KV8 ? kTileThreads8 : kTileThreads;
  constexpr int RAW_ROW = D <= 64 ? 64 : 128;      // bytes per staged row of codes (padded past head_dim)
  constexpr int RAW_BYTES = kKeyTile * RAW_ROW;    // 8-bit codes of one range
  constexpr uint32_t RAW_OFF = Lay::KV_BYTES / 2;  // staged in the back half of the slot
  static_assert(RAW_BYTES == Lay::KV_BYTES / 2, "a range's codes fill half of its 16-bit slot");
  constexpr int KSTEPS_S = D / 16;         // UMMA K steps of S = Q K^T
  constexpr int KSTEPS_O = kKeyTile / 16;  // UMMA K steps of O = P V
  constexpr int POS_PER_HALF = kHalfRows / G;
  constexpr int PART_KEYS = kKeyTile / kParts;  // keys of a range per softmax warp
  constexpr int NCH = (D + 31) / 32;            // 32-column chunks of O (head_dim 80: 16 padding columns)
  constexpr uint32_t IDESC_S = f16_idesc(kHalfRows, kKeyTile, 0, M::kUmmaFormat);
  constexpr uint32_t IDESC_O = f16_idesc(kHalfRows, D, 1, ElemFp16::kUmmaFormat);
  constexpr uint32_t IDESC_OB = f16_idesc(kHalfRows, D, 1, ElemBf16::kUmmaFormat);  // a range kept bf16
  // O stays in TMEM and is rescaled only when a row's running maximum grows
  // by more than 2^8 (log2 domain); in between, probabilities are taken
  // against the older maximum and stay below 256.
  constexpr float kRescaleLog2 = 8.f;
  constexpr unsigned FULL = 0xffffffffu;
  (void)NTHREADS;

  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t base = smem_u32(smem_raw);
  if (base & 1023u) {  // the swizzled tiles need 1024-byte alignment; never touch misaligned tiles
    if (tid == 0) flag_error(p.status, PA_FLAG_LENGTHS);
    griddep_wait();  // completion still implies the decode kernel's
    return;
  }
  constexpr int SLOTS = Lay::SLOTS;
  const uint32_t sQ0 = base + Lay::Q_OFF, sRing = base + Lay::RING_OFF;
  auto bar = [&](int i) { return base + Lay::BAR_OFF + 8u * static_cast<uint32_t>(i); };
  uint32_t *tmem_base_s = reinterpret_cast<uint32_t *>(smem_raw + Lay::TMEM_OFF);
  volatile int *units = reinterpret_cast<volatile int *>(smem_raw + Lay::UNIT_OFF);
  volatile float *xch = reinterpret_cast<volatile float *>(smem_raw + Lay::XCH_OFF);
  volatile int *vkeep = reinterpret_cast<volatile int *>(smem_raw + Lay::VF_OFF);  // bf16 V range kept bf16

  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_base_s), kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < kMaxSlots; ++i) {
      // full: the producer's TMA (16-bit caches) or one arrival per converter warp (8-bit)
      mbar_init(bar(Lay::B_FULL + i), KV8 ? kConvWarps : 1);
      mbar_init(bar(Lay::B_EMPTY + i), 1);  // the MMA warp's commit after the range's last product
      // bf16 caches: conv and raw count one arrival per converter warp
      mbar_init(bar(Lay::B_RAW + i), KV8 ? 1 : kConvWarps);
      mbar_init(bar(Lay::B_CONV + i), KV8 ? 32 * kConvWarps : kConvWarps);
    }
    for (int h = 0; h < kHalves; ++h) {
      mbar_init(bar(Lay::B_S + h), 1);
      mbar_init(bar(Lay::B_P + h), 4 * kParts);  // the half's softmax warps
      mbar_init(bar(Lay::B_O + h), 1);
      mbar_init(bar(Lay::B_QF + h), 4 * kParts);
      mbar_init(bar(Lay::B_QE + h), 1);
    }
    for (int i = 0; i < kUnitSlots; ++i) {
      mbar_init(bar(Lay::B_UF + i), 1);
      mbar_init(bar(Lay::B_UE + i), 1 + kSoftmaxWarps + (KV8 || VCONV ? kConvWarps : 0));
    }
    for (int i = 0; i < 4 * kHalves; ++i) mbar_init(bar(Lay::B_X + i), 32 * kParts);
    mbar_init(bar(Lay::B_DRAIN), 1);
    prefetch_tmap(&kmap);
    prefetch_tmap(&vmap);
    if (VBLK) prefetch_tmap(&vmapb);
  }
  fence_mbar_init();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // No griddepcontrol.wait here: this kernel follows the split-KV decode
  // kernel, which lets it start as its CTAs exit; it reads only what the
  // kernels before that one wrote (the plan's tiles, q, the caches), all
  // complete before the decode kernel let it start. It waits for the decode
  // kernel at its end, so its own completion still orders later work.
  const uint32_t tmem = *tmem_base_s;

  const int Hkv = p.num_kv_heads;
  const int bs = p.block_size;
  bool failed = false;
  uint32_t issued = 0;  // producer: loads issued (the final drain waits for them)

  // Record j of the stream sits in slot j % kUnitSlots; every consumer warp
  // reads each record once and releases the slot.
  auto read_unit = [&](uint32_t j, TileUnit &r) {
    const uint32_t s = j % kUnitSlots;
    wait_warp(bar(Lay::B_UF + s), (j / kUnitSlots) & 1u, failed);
    r.stop = 1;
    if (!failed) {
      const volatile int *u = units + 8 * s;
      r.b = u[0];
      r.row0 = u[1];
      r.npos = u[2];
      r.pos0 = u[3];
      r.kv_end = u[4];
      r.kvh = u[5];
      r.stop = u[6];
    }
    __syncwarp();
    if (lane == 0 && !failed) mbar_arrive(bar(Lay::B_UE + s));
  };
  // key ranges of the unit, and of each half: up to its last valid position (0 = no valid rows)
  auto ranges = [&](const TileUnit &r, int (&nh)[kHalves]) {
#pragma unroll
    for (int h = 0; h < kHalves; ++h) {
      const int last = min(r.npos, (h + 1) * POS_PER_HALF);  // positions [h * POS_PER_HALF, last)
      nh[h] = last > h * POS_PER_HALF ? (r.pos0 + last + kKeyTile - 1) / kKeyTile : 0;
    }
    return (r.kv_end + kKeyTile - 1) / kKeyTile;
  };
  // V in shared memory. VBLK: block after block of R = block_size rows, each
  // [atom][R rows][128 B]; else [atom][128 keys][128 B] (per-atom boxes).
  const int vshift = p.block_shift;  // log2(R)
  auto v_off = [&](int rr, int c) -> uint32_t {  // 16-byte chunk c of key row rr of a range
    if constexpr (VBLK) {
      const int blk = rr >> vshift, r = rr & (bs - 1);
      return static_cast<uint32_t>(blk * bs * 256 + (c >> 3) * bs * 128 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
    } else {
      return Lay::off(rr, c, Lay::KV_ATOM);
    }
  };

  if (warp == kTmaWarp) {
    // ---------------- producer: unit records, then K(j), V(j) of each range ----------------
    const int total_units = min(max(ld_cg(p.tile_count), 0), p.max_tiles) * Hkv;
    constexpr int MAXROWS = KV8 ? kRawBoxRows : kTileKeys;
    const int box_rows = bs < MAXROWS ? bs : MAXROWS;  // K boxes (and V boxes unless VBLK)
    const int nbk = kKeyTile / box_rows;                // 4 .. 16
    const int nbv = VBLK ? kKeyTile / bs : nbk;         // VBLK: one box per block
    uint32_t j = 0, g = 0;
    for (;;) {
      int u = 0;
      if (lane == 0) u = atomicAdd(p.tile_counter, 1);
      u = __shfl_sync(FULL, u, 0);
      TileUnit r{0, 0, 0, 0, 0, 0, u >= total_units ? 1 : 0};
      if (!r.stop) {
        const int item = u / Hkv;
        r.kvh = u - item * Hkv;
        const int4 r0 = ld_cg(p.tiles + 2 * item);
        const int4 r1 = ld_cg(p.tiles + 2 * item + 1);
        r.b = r0.x;
        r.row0 = r0.y;
        r.npos = r0.z;
        r.pos0 = r0.w;
        r.kv_end = r1.y;
        const bool sane = r.b >= 0 && r.b < p.num_seqs && r.npos >= 1 && r.npos <= kPrefillTileRows / G &&
                          r.row0 >= 0 && r.row0 + r.npos <= p.total_q && r.pos0 >= 0 &&
                          r.kv_end == r.pos0 + r.npos &&
                          r.kv_end <= static_cast<int64_t>(p.max_blocks_per_seq) * bs;
        if (!sane) {
          if (lane == 0) flag_error(p.status, PA_FLAG_LENGTHS);
          continue;
        }
      }
      const uint32_t s = j % kUnitSlots;
      if (j >= kUnitSlots) wait_warp(bar(Lay::B_UE + s), (j / kUnitSlots - 1) & 1u, failed);
      if (failed) break;
      if (lane == 0) {
        volatile int *d = units + 8 * s;
        d[0] = r.b;
        d[1] = r.row0;
        d[2] = r.npos;
        d[3] = r.pos0;
        d[4] = r.kv_end;
        d[5] = r.kvh;
        d[6] = r.stop;
        mbar_arrive(bar(Lay::B_UF + s));  // release: the record is visible to whoever sees the phase
      }
      __syncwarp();
      ++j;
      if (r.stop) break;
      const int32_t *table = p.block_tables + static_cast<int64_t>(r.b) * p.max_blocks_per_seq;
      // First cache row of the box of `rows` keys starting at `key`: a block-table
      // lookup (block sizes are powers of two); keys past the end, or a block id
      // out of range, read at -rows (zero fill).
      auto box_z = [&](int key, int rows) {
        if (key >= r.kv_end) return -rows;
        const int phys = __ldg(table + (key >> p.block_shift));
        if (phys < 0 || phys >= p.num_blocks) {
          flag_error(p.status, PA_FLAG_BLOCK_RANGE);
          return -rows;
        }
        return (phys << p.block_shift) + (key & (bs - 1));
      };
      int dummy[kHalves];
      const int nkt = ranges(r, dummy);
      for (int kt = 0; kt < nkt && !failed; ++kt) {
        // lane i computes the row coordinate of K box i and V box i of this
        // range, and issues those boxes itself once lane 0 has set the byte count
        const int zk = lane < nbk ? box_z(kt * kKeyTile + lane * box_rows, box_rows) : 0;
        const int zv = VBLK ? (lane < nbv ? box_z(kt * kKeyTile + lane * bs, bs) : 0) : zk;
        for (int v = 0; v < 2 && !failed; ++v) {
          const uint32_t slot = g % SLOTS, use = g / SLOTS;
          if (use > 0) wait_warp(bar(Lay::B_EMPTY + slot), (use - 1) & 1u, failed);
          if (failed) break;
          const void *map = v ? static_cast<const void *>(&vmap) : static_cast<const void *>(&kmap);
          const uint32_t dst = sRing + slot * Lay::KV_BYTES;
          if constexpr (KV8) {
            // the range's codes: boxes of box_rows x D bytes into the back half of the slot
            const uint32_t b8 = bar(Lay::B_RAW + slot);
            if (lane == 0) mbar_arrive_expect_tx(b8, RAW_BYTES);
            __syncwarp();
            if (lane < nbk) tma_load_3d(dst + RAW_OFF + lane * box_rows * RAW_ROW, map, b8, 0, r.kvh, zk);
          } else {
            const uint32_t bf = bar(Lay::B_FULL + slot);
            if (lane == 0) mbar_arrive_expect_tx(bf, Lay::KV_BYTES);
            __syncwarp();
            if (VBLK && v) {
              // one box per block: both atoms of bs rows, [atom][rows][128 B]
              if (lane < nbv) tma_load_4d(dst + lane * bs * 256, &vmapb, bf, 0, zv, 0, r.kvh);
            } else if (lane < nbk) {
              // per-atom boxes of box_rows rows: [atom][128 keys][128 B]
#pragma unroll
              for (int a = 0; a < Lay::ATOMS; ++a)
                tma_load_3d(dst + a * Lay::KV_ATOM + lane * box_rows * 128, map, bf, a * 64, r.kvh, v ? zv : zk);
            }
          }
          __syncwarp();
          issued = ++g;
        }
      }
      if (failed) break;
    }
  } else if (warp >= kConvWarp && warp < kSoftmaxWarp0) {
    // ---------------- 8-bit caches: widen staged codes to fp16 in place ----------------
    if constexpr (KV8) {
      // Lane l of converter warp w takes 16-byte code chunk c of rows
      // r0 + l % 8, so the eight lanes of one shared-memory phase touch eight
      // rows at one chunk: distinct bank groups in both swizzled layouts.
      constexpr int CPR = RAW_ROW / 16;         // code chunks per staged row (zeros past head_dim)
      constexpr int ROWS_PASS = 8 * (8 / CPR);  // rows per pass of the 64 threads
      constexpr int PASSES = kKeyTile / ROWS_PASS;
      const int ct = (warp - kConvWarp) * 32 + lane;
      const int q8 = ct >> 3, c = q8 % CPR, rsub = (q8 / CPR) * 8 + (ct & 7);
      uint32_t j = 0, g = 0;
      for (;;) {
        TileUnit r;
        read_unit(j++, r);
        if (failed || r.stop) break;
        int dummy[kHalves];
        const int nkt = ranges(r, dummy);
        for (int i = 0; i < 2 * nkt && !failed; ++i, ++g) {
          const uint32_t slot = g % SLOTS, use = g / SLOTS;
          wait_warp(bar(Lay::B_RAW + slot), use & 1u, failed);
          if (failed) break;
          const uint32_t sbase = sRing + slot * Lay::KV_BYTES;
          uint4 codes[PASSES];
#pragma unroll
          for (int i2 = 0; i2 < PASSES; ++i2) {
            const int rr = i2 * ROWS_PASS + rsub;
            const uint32_t a = sbase + RAW_OFF + (RAW_ROW == 128 ? rr * 128 + (((c ^ rr) & 7) << 4)
                                                                  : rr * 64 + (((c ^ (rr >> 1)) & 3) << 4));
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];\n"
                         : "=r"(codes[i2].x), "=r"(codes[i2].y), "=r"(codes[i2].z), "=r"(codes[i2].w)
                         : "r"(a));
          }
          // every code of the slot is in registers (both warps) before any fp16 row overwrites them
          mbar_arrive(bar(Lay::B_CONV + slot));
          wait_warp(bar(Lay::B_CONV + slot), use & 1u, failed);
          if (failed) break;
#pragma unroll
          for (int i2 = 0; i2 < PASSES; ++i2) {
            const int rr = i2 * ROWS_PASS + rsub;
            const uint32_t w[4] = {codes[i2].x, codes[i2].y, codes[i2].z, codes[i2].w};
            uint32_t hh[8];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              asm("{\n .reg .b16 l, u;\n mov.b32 {l, u}, %2;\n cvt.rn.f16x2.e4m3x2 %0, l;\n"
                  " cvt.rn.f16x2.e4m3x2 %1, u;\n}\n"
                  : "=r"(hh[2 * k]), "=r"(hh[2 * k + 1])
                  : "r"(w[k]));
            }
            // codes d = 16c .. 16c + 15 -> fp16 chunks 2c (d .. d + 7) and 2c + 1
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};\n" ::"r"(sbase + Lay::off(rr, 2 * c, Lay::KV_ATOM)),
                         "r"(hh[0]), "r"(hh[1]), "r"(hh[2]), "r"(hh[3])
                         : "memory");
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};\n" ::"r"(
                             sbase + Lay::off(rr, 2 * c + 1, Lay::KV_ATOM)),
                         "r"(hh[4]), "r"(hh[5]), "r"(hh[6]), "r"(hh[7])
                         : "memory");
          }
          fence_proxy_async_smem();  // the MMA reads the slot through the async proxy
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(Lay::B_FULL + slot));
        }
        if (failed) break;
      }
    } else if constexpr (VCONV) {
      // bf16 V ranges rewritten as fp16 in place, each by both converter
      // warps (half of its chunks each; one warp per range, the two taking
      // alternate ranges, measured 5 % slower). Range g (counted over the
      // CTA's units) uses conv barrier and flags g % kMaxSlots (the ring
      // keeps the converters fewer ranges ahead): each warp writes its flag
      // (a chunk stayed bf16) and arrives; the warps then read both flags,
      // and if either is set they put their fp16 chunks back to bf16 and
      // arrive on the range's raw barrier, which readers wait for only then.
      constexpr int PER = Lay::KV_BYTES / 16 / (32 * kConvWarps);  // chunks per lane
      using Mask = uint32_t;
      const int cw = warp - kConvWarp;
      const int c0 = cw * PER * 32 + lane;
      auto key_of = [&](uint32_t o) -> int {  // key row of the chunk at byte offset o of a V slot
        if constexpr (VBLK)
          return static_cast<int>(((o >> (vshift + 8)) << vshift) + ((o >> 7) & static_cast<uint32_t>(bs - 1)));
        else
          return static_cast<int>((o >> 7) & static_cast<uint32_t>(kKeyTile - 1));
      };
      uint32_t j = 0, ring = 0, gv = 0;
      for (;;) {
        TileUnit r;
        read_unit(j++, r);
        if (failed || r.stop) break;
        int dummy[kHalves];
        const int nkt = ranges(r, dummy);
        for (int kt = 0; kt < nkt && !failed; ++kt, ++gv) {
          const uint32_t pos = ring + 2 * kt + 1, slot = pos % SLOTS;  // V(kt) in the load ring
          wait_warp(bar(Lay::B_FULL + slot), (pos / SLOTS) & 1u, failed);
          if (failed) break;
          const uint32_t sV = sRing + slot * Lay::KV_BYTES;
          const int nvalid = min(r.kv_end - kt * kKeyTile, kKeyTile);
          const bool masked = nvalid < kKeyTile;
          const Mask kept = masked ? vrange_to_fp16<PER, true, Mask>(sV, c0, nvalid, key_of)
                                   : vrange_to_fp16<PER, false, Mask>(sV, c0, nvalid, key_of);
          const bool any_kept = __any_sync(FULL, kept != 0);
          const uint32_t fi = gv % kMaxSlots;
          fence_proxy_async_smem();  // the MMA reads the slot through the async proxy
          __syncwarp();
          if (lane == 0) {
            vkeep[2 * fi + cw] = any_kept ? 1 : 0;
            mbar_arrive(bar(Lay::B_CONV + fi));  // release: the flag and the rows
          }
          wait_warp(bar(Lay::B_CONV + fi), (gv / kMaxSlots) & 1u, failed);
          if (failed) break;
          if (vkeep[2 * fi] | vkeep[2 * fi + 1]) {
            if (masked)
              vrange_back_to_bf16<PER, true>(sV, c0, nvalid, kept, key_of);
            else
              vrange_back_to_bf16<PER, false>(sV, c0, nvalid, kept, key_of);
            fence_proxy_async_smem();
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(Lay::B_RAW + fi));
        }
        ring += 2 * nkt;
        if (failed) break;
      }
    }
  } else if (warp == kMmaWarp) {
    // ---------------- MMA issue ----------------
    // The whole warp follows the loops (it zeroes the tail of the last V
    // range); lane 0 alone issues tensor-core work and commits. Range r of a
    // unit is read by the halves with r < nkt_h: the first of them waits for
    // the K/V loads, the last one's commit releases the buffers.
    constexpr uint32_t DHI = desc_hi(1024);
    const uint32_t q_lo0 = desc_lo(sQ0, 16), q_lo1 = desc_lo(sQ0 + Lay::Q_BYTES, 16);
    const uint32_t k_lo = desc_lo(sRing, 16);  // slot 0
    // V (MN-major): LBO = distance between the two 64-element atoms along d,
    // SBO = distance between 8-key groups along K; VBLK blocks of 8 rows put
    // consecutive 8-key groups in consecutive blocks
    const uint32_t v_lo = VBLK ? desc_lo(sRing, static_cast<uint32_t>(bs) * 128u) : desc_lo(sRing, Lay::KV_ATOM);
    const uint32_t v_hi = VBLK && bs == 8 ? desc_hi(2048) : DHI;
    constexpr uint32_t SLOT_STEP = Lay::KV_BYTES >> 4;  // per slot
    uint32_t vks[KSTEPS_O];                              // byte offset >> 4 of V's K step ks
#pragma unroll
    for (int ks = 0; ks < KSTEPS_O; ++ks) {
      const int k16 = ks * 16;
      vks[ks] = VBLK ? static_cast<uint32_t>(((k16 >> vshift) * bs * 256 + (k16 & (bs - 1)) * 128) >> 4)
                     : static_cast<uint32_t>((ks * 2048) >> 4);
    }
    uint32_t ph[kHalves] = {0, 0};  // ranges each half has run so far (phases of its s, p, o barriers)
    uint32_t ring0 = 0;             // loads of earlier units
    for (uint32_t j = 0;; ++j) {
      TileUnit r;
      read_unit(j, r);
      if (failed || r.stop) break;
      int nkt_h[kHalves];
      const int nkt = ranges(r, nkt_h);
      auto first_reader = [&](int kt) { return kt < nkt_h[0] ? 0 : 1; };
      auto last_reader = [&](int kt) { return kt < nkt_h[1] ? 1 : 0; };
      // ring slot of K(kt) (v = 0) or V(kt) (v = 1), and the parity of its full barrier
      auto slot_of = [&](int kt, int v) { return (ring0 + 2 * kt + v) % SLOTS; };
      auto full_parity = [&](int kt, int v) { return ((ring0 + 2 * kt + v) / SLOTS) & 1u; };
      auto mma_s = [&](int kt, int h) {
        if (lane == 0) {
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
          tc_commit(bar(Lay::B_S + h));
          if (h == last_reader(kt)) tc_commit(bar(Lay::B_EMPTY + slot_of(kt, 0)));
        }
        __syncwarp();
      };
      // this unit's Q in both halves (the softmax warps store it); qe lets them store the next one
#pragma unroll
      for (int h = 0; h < kHalves; ++h) {
        wait_warp(bar(Lay::B_QF + h), j & 1u, failed);
        if (lane == 0 && !failed) mbar_arrive(bar(Lay::B_QE + h));
      }
      if (failed) break;
      if (nkt > 0) {
        wait_warp(bar(Lay::B_FULL + slot_of(0, 0)), full_parity(0, 0), failed);
#pragma unroll
        for (int h = 0; h < kHalves; ++h)
          if (nkt_h[h] > 0 && !failed) mma_s(0, h);
      }
      for (int kt = 0; kt < nkt && !failed; ++kt) {
        const uint32_t vslot = slot_of(kt, 1);
        bool vpair = false;  // this range's V kept bf16: P as a hi + lo pair
#pragma unroll
        for (int h = 0; h < kHalves; ++h) {
          if (kt >= nkt_h[h]) continue;
          wait_warp(bar(Lay::B_P + h), (ph[h] + kt) & 1u, failed);  // P(kt) is in place
          if (failed) break;
          if (VCONV && h == first_reader(kt)) {
            // the converter warp has rewritten V(kt) (and zeroed the rows past the last key)
            const uint32_t gv = ring0 / 2 + kt, fi = gv % kMaxSlots;
            wait_warp(bar(Lay::B_CONV + fi), (gv / kMaxSlots) & 1u, failed);
            if (failed) break;
            vpair = (vkeep[2 * fi] | vkeep[2 * fi + 1]) != 0;
            if (vpair) wait_warp(bar(Lay::B_RAW + fi), (gv / kMaxSlots) & 1u, failed);  // back in bf16
            if (failed) break;
          } else if (h == first_reader(kt)) {
            wait_warp(bar(Lay::B_FULL + vslot), full_parity(kt, 1), failed);
            if (failed) break;
            const int key0 = kt * kKeyTile;
            if (key0 + kKeyTile > r.kv_end) {
              // rows of keys past kv_end may hold anything (even NaN): zero them in V
              const uint32_t sV = sRing + vslot * Lay::KV_BYTES;
              const int vr0 = r.kv_end - key0;
              const int n = (kKeyTile - vr0) * (D / 8);
              for (int i = lane; i < n; i += 32) {
                const int rr = vr0 + i / (D / 8), c = i % (D / 8);
                asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};\n" ::"r"(sV + v_off(rr, c)), "r"(0u)
                             : "memory");
              }
              fence_proxy_async_smem();
            }
            __syncwarp();
          }
          if (lane == 0) {
            tc_fence_after();
            const uint32_t vlo = v_lo + vslot * SLOT_STEP;
            const uint32_t t = tmem + h * Tm::HALF;
            if (!vpair) {
              // one fp16 P per key: K step ks at column 8 ks (+ 32 for the second part's keys)
              auto pcol = [](int ks) { return 8 * ks + (ks >= 4 ? 32 : 0); };
              if (kt == 0)
                mma_ts<0>(t + Tm::O, t + Tm::SP, vlo, v_hi, IDESC_O);  // the unit's first product overwrites O
              else
                mma_ts<1>(t + Tm::O, t + Tm::SP, vlo, v_hi, IDESC_O);
#pragma unroll
              for (int ks = 1; ks < KSTEPS_O; ++ks)
                mma_ts<1>(t + Tm::O, t + Tm::SP + pcol(ks), vlo + vks[ks], v_hi, IDESC_O);
            } else {
              // a bf16 hi + lo pair per key: K step ks at columns 16 ks (hi) and 16 ks + 8 (lo)
              if (kt == 0)
                mma_ts<0>(t + Tm::O, t + Tm::SP, vlo, v_hi, IDESC_OB);
              else
                mma_ts<1>(t + Tm::O, t + Tm::SP, vlo, v_hi, IDESC_OB);
              mma_ts<1>(t + Tm::O, t + Tm::SP + 8, vlo, v_hi, IDESC_OB);
#pragma unroll
              for (int ks = 1; ks < KSTEPS_O; ++ks) {
                mma_ts<1>(t + Tm::O, t + Tm::SP + 16 * ks, vlo + vks[ks], v_hi, IDESC_OB);
                mma_ts<1>(t + Tm::O, t + Tm::SP + 16 * ks + 8, vlo + vks[ks], v_hi, IDESC_OB);
              }
            }
            tc_commit(bar(Lay::B_O + h));
            if (h == last_reader(kt)) tc_commit(bar(Lay::B_EMPTY + vslot));
          }
          __syncwarp();
          if (kt + 1 < nkt_h[h]) {
            if (h == first_reader(kt + 1))
              wait_warp(bar(Lay::B_FULL + slot_of(kt + 1, 0)), full_parity(kt + 1, 0), failed);
            if (failed) break;
            mma_s(kt + 1, h);
          }
        }
      }
      if (failed) break;
#pragma unroll
      for (int h = 0; h < kHalves; ++h) ph[h] += nkt_h[h];
      ring0 += 2 * nkt;
    }
  } else {
    // ---------------- softmax: one row per thread (its TMEM lane), 64 keys per range ----------------
    const int sw = warp - kSoftmaxWarp0;  // softmax warp index
    const int quad = sw & 3, h = (sw >> 2) & 1, part = sw / (4 * kHalves);
    const int r = quad * 32 + lane;  // row within the half = TMEM lane
    const uint32_t t_lane = tmem + h * Tm::HALF + (static_cast<uint32_t>(quad * 32) << 16);
    const uint32_t bx = bar(Lay::B_X + h * 4 + quad);  // exchange with the other warp of these rows
    volatile float *x_mine = xch + (h * kParts + part) * kHalfRows + r;
    volatile float *x_other = xch + (h * kParts + (kParts - 1 - part)) * kHalfRows + r;
    uint32_t nx = 0;  // exchanges so far
    // my value out, the other warp's value in (both warps of the rows call it alike)
    auto exchange = [&](float v) -> float {
      *x_mine = v;
      mbar_arrive(bx);  // every thread: release of its own store
      wait_warp(bx, nx & 1u, failed);
      ++nx;
      return failed ? v : *x_other;
    };
    // both warps of the rows have reached this point (no data)
    auto pair_sync = [&]() {
      mbar_arrive(bx);
      wait_warp(bx, nx & 1u, failed);
      ++nx;
    };
    const int ch0 = part ? (NCH + 1) / 2 : 0, ch1 = part ? NCH : (NCH + 1) / 2;  // this warp's O chunks
    const int g = r % G;
    uint32_t phh = 0;  // ranges this half has run so far
    uint32_t gvs = 0;  // ranges of the CTA's earlier units (both halves)

    // Q of the half for unit `u`: this warp stores its half of the row's 16-byte
    // chunks (row r = (position, head), K-major, swizzled); returns the row's
    // softmax factor (log2 domain, times 2^e for a scaled bf16 row over 8-bit caches)
    auto load_q = [&](const TileUnit &u) -> float {
      const int qi = h * POS_PER_HALF + r / G;
      const bool valid = qi < u.npos;
      const uint32_t sQ = sQ0 + h * Lay::Q_BYTES;
      const bf16 *qrow =
          p.q + static_cast<int64_t>(u.row0 + (valid ? qi : 0)) * p.q_stride + static_cast<int64_t>(u.kvh * G + g) * D;
      // q is only required to be 4-byte aligned: 16-byte loads when rows allow them
      const bool q16 = (reinterpret_cast<uintptr_t>(p.q) & 15u) == 0 && (p.q_stride & 7) == 0;
      auto ldq = [&](int c) {
        uint4 w = make_uint4(0u, 0u, 0u, 0u);
        if (valid) {
          if (q16) {
            w = __ldg(reinterpret_cast<const uint4 *>(qrow) + c);
          } else {
            const uint32_t *q32 = reinterpret_cast<const uint32_t *>(qrow) + 4 * c;
            w = make_uint4(__ldg(q32), __ldg(q32 + 1), __ldg(q32 + 2), __ldg(q32 + 3));
          }
        }
        return w;
      };
      float sl2 = p.scale_log2;  // > 0: the max of raw scores gives the max of scaled ones
      float qmul = 1.f;
      if constexpr (KV8 && std::is_same<E, ElemBf16>::value) {
        // bf16 rows over 8-bit caches: 2^-e, e > 0 only when the row's largest |q| reaches 2^15
        float amax = 0.f;
#pragma unroll 4
        for (int c = 0; c < D / 8; ++c) {
          const uint4 w = ldq(c);
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
      constexpr int CQ = D / 16;  // chunks per warp (D / 8 per row)
#pragma unroll 4
      for (int c = part * CQ; c < (part + 1) * CQ; ++c) {
        uint4 w = ldq(c);
        if constexpr (KV8 && std::is_same<E, ElemBf16>::value) {
          w = make_uint4(ElemFp16::pack(ElemBf16::lo(w.x) * qmul, ElemBf16::hi(w.x) * qmul),
                         ElemFp16::pack(ElemBf16::lo(w.y) * qmul, ElemBf16::hi(w.y) * qmul),
                         ElemFp16::pack(ElemBf16::lo(w.z) * qmul, ElemBf16::hi(w.z) * qmul),
                         ElemFp16::pack(ElemBf16::lo(w.w) * qmul, ElemBf16::hi(w.w) * qmul));
        }
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};\n" ::"r"(sQ + Lay::off(r, c, Lay::Q_ATOM)), "r"(w.x),
                     "r"(w.y), "r"(w.z), "r"(w.w)
                     : "memory");
      }
      fence_proxy_async_smem();  // the MMA reads Q through the async proxy
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(Lay::B_QF + h));
      return sl2;
    };

    TileUnit cur;
    read_unit(0, cur);
    float sl2 = 0.f;
    if (!failed && !cur.stop) sl2 = load_q(cur);
    for (uint32_t j = 0; !failed && !cur.stop; ++j) {
      int nkt_h[kHalves];
      const int nkt_all = ranges(cur, nkt_h);
      const int nk = nkt_h[h];
      const int qi = h * POS_PER_HALF + r / G;
      const bool row_valid = qi < cur.npos;
      const int lim = row_valid ? cur.pos0 + qi + 1 : 0;  // keys j < lim are visible to this row
      float m_used = -INFINITY, l = 0.f;
      for (int kt = 0; kt < nk; ++kt) {
        const int ck0 = kt * kKeyTile + part * PART_KEYS;  // this warp's first key of the range
        const uint32_t sp = t_lane + Tm::SP + part * PART_KEYS;
        wait_warp(bar(Lay::B_S + h), (phh + kt) & 1u, failed);
        if (failed) break;
        tc_fence_after();
        uint32_t s0[32], s1[32];
        tmem_ld32x2_wait(sp, s0, s1);
        // The range's maximum over both warps' keys, then its growth over
        // m_used, as separately rounded operations (no contraction into one
        // fused multiply-add): the exponents below are bounded by exactly this
        // difference. The other warp reads its scores before either writes P.
        const float mx = fmaxf(masked_max32(s0, ck0, lim), masked_max32(s1, ck0 + 32, lim));
        const float mo = exchange(mx);
        if (failed) break;
        const float cm = __fmul_rn(sl2, fmaxf(mx, mo));
        const bool grow = cm > -INFINITY && (m_used == -INFINITY || __fsub_rn(cm, m_used) > kRescaleLog2);
        float alpha = 1.f;  // factor owed by O and l for the growth
        if (grow) {
          alpha = m_used > -INFINITY ? ex2_approx(__fsub_rn(m_used, cm)) : 1.f;
          m_used = cm;
        }
        const float ms = m_used == -INFINITY ? 0.f : m_used;
        float sum = 0.f;
        const bool exact = __any_sync(FULL, fabsf(ms) > 4096.f);
        bool vpair = false;  // V(kt) kept bf16 (bf16 caches only): P as a hi + lo pair
        if constexpr (VCONV) {
          const uint32_t gv = gvs + kt, fi = gv % kMaxSlots;
          wait_warp(bar(Lay::B_CONV + fi), (gv / kMaxSlots) & 1u, failed);
          if (failed) break;
          vpair = (vkeep[2 * fi] | vkeep[2 * fi + 1]) != 0;
        }
        // P over the scores it came from, one UMMA K step (16 keys) at a
        // time, the scores read again from TMEM: a loop unrolled twice, not
        // four times (the hot code of twenty warps shares the instruction
        // cache; measured 5 % faster over bf16 caches than four steps inline
        // on scores kept in registers), no score registers live across it.
        // P of step ks (8 columns at 8 ks) covers only scores read by
        // earlier steps. Rare cases stay out of the loop (inside it, as a
        // branch per step, they cost 2 %).
        if (vpair) {
          range_probs<true>(sp, ck0, lim, sl2, ms, exact, sum);
        } else if (exact) {
          range_probs<false>(sp, ck0, lim, sl2, ms, true, sum);
        } else {
#pragma unroll 2
          for (int ks = 0; ks < PART_KEYS / 16; ++ks) {
            uint32_t t[16];
            tmem_ld16_wait(sp + 16 * ks, t);
            probs16_store<ElemFp16, false, false>(t, ck0 + 16 * ks, lim, sl2, ms, sum, sp + 8 * ks);
          }
        }
        // O holds P V(0 .. kt-1), all complete (they were issued before S(kt),
        // whose completion the wait above observed); each warp rescales its
        // own columns.
        if (kt > 0 && __any_sync(FULL, alpha != 1.f)) {
#pragma unroll 1
          for (int ch = ch0; ch < ch1; ++ch) {
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
        if (lane == 0) mbar_arrive(bar(Lay::B_P + h));
      }
      if (failed) break;
      // the next unit's record and Q (overlapping this unit's last products)
      TileUnit nxt;
      read_unit(j + 1, nxt);
      float nsl2 = sl2;
      if (!failed && !nxt.stop) {
        wait_warp(bar(Lay::B_QE + h), j & 1u, failed);  // the MMA warp has taken this unit's Q
        if (!failed) nsl2 = load_q(nxt);
      }
      if (failed) break;
      if (nk > 0) {
        // epilogue: the row sum over both warps' keys, then this warp's columns
        // of the half's last P V product, normalised
        pair_sync();  // both warps are past their last read of the maxima
        const float lt = l + exchange(l);
        pair_sync();  // both have read the sums
        wait_warp(bar(Lay::B_O + h), (phh + nk - 1) & 1u, failed);
        if (failed) break;
        tc_fence_after();
        const float inv = lt > 0.f ? p.out_scale / lt : 0.f;
        bf16 *dst = p.out + static_cast<int64_t>(cur.row0 + (row_valid ? qi : 0)) * p.num_heads * D +
                    static_cast<int64_t>(cur.kvh * G + g) * D;
#pragma unroll 1
        for (int ch = ch0; ch < ch1; ++ch) {
          uint32_t t[32];
          tmem_ld32_wait(t_lane + Tm::O + ch * 32, t);
          if (row_valid) {
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
        tc_fence_before();  // O is overwritten by a later unit's first product
      }
      phh += nk;
      gvs += nkt_all;
      cur = nxt;
      sl2 = nsl2;
    }
  }

  // Every warp has left its loop (normally at the end of the stream, or after
  // a timeout). Before tensor memory and shared memory go away, wait (bounded)
  // for work still in flight: the MMA thread's products (one last commit)
  // and the producer's loads (loads into a buffer complete in order, so
  // waiting for the last SLOTS issued suffices).
  if (warp == kMmaWarp && lane == 0) {
    tc_commit(bar(Lay::B_DRAIN));
    if (!mbar_wait_bounded(bar(Lay::B_DRAIN), 0, kTcWaitTimeoutNs)) failed = true;
  }
  if (warp == kTmaWarp && lane == 0) {
    const int landed = KV8 ? Lay::B_RAW : Lay::B_FULL;  // where the loads' completion is counted
    for (uint32_t g = issued > SLOTS ? issued - SLOTS : 0; g < issued; ++g)
      if (!mbar_wait_bounded(bar(landed + static_cast<int>(g % SLOTS)), (g / SLOTS) & 1u, kTcWaitTimeoutNs))
        failed = true;
  }
  if (failed) flag_error(p.status, PA_FLAG_TIMEOUT);
  griddep_wait();  // the decode kernel before this one has completed
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------------------
// head_dim 256: one 128-row half per tile. S (128 columns) and O (256) of a
// half take 384 of the 512 TMEM columns, so the tile has one half and two
// score buffers: S(r + 1) is computed while the softmax works on S(r), and
// the tensor cores run P V(r) and S(r + 2) behind it. A K or V range is
// staged as two units of 128 keys x 128 elements (d 0..127 and 128..255),
// each laid out like a head_dim-128 ring slot (so 8-bit codes are widened
// unit by unit exactly as there), four loads per range; S takes its first
// eight K steps from the first K unit and the rest from the second, and
// P V is two N = 128 products per K step, one per V unit, into O's two
// column halves. The roles, the record ring, the bounded waits and the exit
// path are those of the kernel above; eight softmax warps (two per TMEM lane
// quadrant, 64 keys of a range each).
// ---------------------------------------------------------------------------
constexpr int kWideD = 256;
constexpr int kWideSoftmaxWarps = 8;
constexpr int kWideThreads = 32 * (kSoftmaxWarp0 + kWideSoftmaxWarps);

struct WideTmem {
  static constexpr uint32_t SP0 = 0, O = 2 * kKeyTile;  // score buffers at 0 and 128, O at [256, 512)
};

struct WideLayout {
  static constexpr int Q_ATOM = kHalfRows * 128;   // 128 rows x 128 B
  static constexpr int Q_BYTES = 4 * Q_ATOM;       // one half, four 64-element atoms
  static constexpr int KV_ATOM = kKeyTile * 128;   // 128 keys x 128 B
  static constexpr int UNIT_BYTES = 2 * KV_ATOM;   // 128 keys x 128 elements: a ring slot
  // mbarriers: per ring slot full, empty, raw, conv; per score buffer s, p;
  // o, qf, qe; per record slot uf, ue; per lane quadrant x1 (values
  // written), x2 (values read); drain
  static constexpr int B_FULL = 0, B_EMPTY = kMaxSlots, B_RAW = 2 * kMaxSlots, B_CONV = 3 * kMaxSlots;
  static constexpr int B_S = 4 * kMaxSlots, B_P = B_S + 2, B_O = B_P + 2, B_QF = B_O + 1, B_QE = B_QF + 1;
  static constexpr int B_UF = B_QE + 1, B_UE = B_UF + kUnitSlots, B_X1 = B_UE + kUnitSlots, B_X2 = B_X1 + 4;
  static constexpr int B_DRAIN = B_X2 + 4, NBARS = B_DRAIN + 1;
  static constexpr int XCH_BYTES = kWideSoftmaxWarps * 32 * 4;
  static constexpr int REC_BYTES = kUnitSlots * 32;
  static constexpr int FIXED = Q_BYTES + XCH_BYTES + REC_BYTES + 8 * NBARS + 16;
  static constexpr int FIT = (227 * 1024 - FIXED) / UNIT_BYTES;
  static constexpr int SLOTS = FIT < kMaxSlots ? FIT : kMaxSlots;
  static_assert(SLOTS >= 5, "the ring holds a range's four loads and the next one's first");
  static constexpr int RING_OFF = Q_BYTES;
  static constexpr int XCH_OFF = RING_OFF + SLOTS * UNIT_BYTES;
  static constexpr int REC_OFF = XCH_OFF + XCH_BYTES;
  static constexpr int BAR_OFF = REC_OFF + REC_BYTES;
  static constexpr int TMEM_OFF = BAR_OFF + 8 * NBARS;
  static constexpr int BYTES = TMEM_OFF + 16;
};
static_assert(WideLayout::BYTES <= 227 * 1024, "shared memory of one CTA");

template <int G, typename E, bool KV8>
__global__ void __launch_bounds__(kWideThreads, 1)
    prefill_tile_wide_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                             const TileParams p) {
  using Lay = WideLayout;
  using Tm = WideTmem;
  using TL = TcLayout<128>;  // a ring slot: the layout of a head_dim-128 range
  constexpr int D = kWideD;
  using M = typename std::conditional<KV8, ElemFp16, E>::type;  // tensor-core operand type
  constexpr bool SPLIT = std::is_same<M, ElemBf16>::value;      // P as a hi + lo pair (bf16 operands only)
  constexpr int RAW_ROW = 128;
  constexpr int RAW_BYTES = kKeyTile * RAW_ROW;    // 8-bit codes of one unit
  constexpr uint32_t RAW_OFF = Lay::UNIT_BYTES / 2;
  constexpr int LPR = 4;                           // loads per range: K lo, K hi, V lo, V hi
  constexpr int KSTEPS_S = D / 16;
  constexpr int KSTEPS_O = kKeyTile / 16;
  constexpr int POS = kHalfRows / G;               // positions per tile
  constexpr uint32_t IDESC_S = f16_idesc(kHalfRows, kKeyTile, 0, M::kUmmaFormat);
  constexpr uint32_t IDESC_O = f16_idesc(kHalfRows, 128, 1, M::kUmmaFormat);
  constexpr float kRescaleLog2 = 8.f;
  constexpr unsigned FULL = 0xffffffffu;
  constexpr int SLOTS = Lay::SLOTS;

  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t base = smem_u32(smem_raw);
  if (base & 1023u) {
    if (tid == 0) flag_error(p.status, PA_FLAG_LENGTHS);
    griddep_wait();
    return;
  }
  const uint32_t sQ = base, sRing = base + Lay::RING_OFF;
  auto bar = [&](int i) { return base + Lay::BAR_OFF + 8u * static_cast<uint32_t>(i); };
  uint32_t *tmem_base_s = reinterpret_cast<uint32_t *>(smem_raw + Lay::TMEM_OFF);
  volatile int *units = reinterpret_cast<volatile int *>(smem_raw + Lay::REC_OFF);
  volatile float *xch = reinterpret_cast<volatile float *>(smem_raw + Lay::XCH_OFF);

  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_base_s), kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < kMaxSlots; ++i) {
      mbar_init(bar(Lay::B_FULL + i), KV8 ? kConvWarps : 1);
      mbar_init(bar(Lay::B_EMPTY + i), 1);
      mbar_init(bar(Lay::B_RAW + i), 1);
      mbar_init(bar(Lay::B_CONV + i), 32 * kConvWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(Lay::B_S + b), 1);
      mbar_init(bar(Lay::B_P + b), kWideSoftmaxWarps);
    }
    mbar_init(bar(Lay::B_O), 1);
    mbar_init(bar(Lay::B_QF), kWideSoftmaxWarps);
    mbar_init(bar(Lay::B_QE), 1);
    for (int i = 0; i < kUnitSlots; ++i) {
      mbar_init(bar(Lay::B_UF + i), 1);
      mbar_init(bar(Lay::B_UE + i), 1 + kWideSoftmaxWarps + (KV8 ? kConvWarps : 0));
    }
    for (int q = 0; q < 4; ++q) {
      mbar_init(bar(Lay::B_X1 + q), 64);  // the two softmax warps of a lane quadrant
      mbar_init(bar(Lay::B_X2 + q), 64);
    }
    mbar_init(bar(Lay::B_DRAIN), 1);
    prefetch_tmap(&kmap);
    prefetch_tmap(&vmap);
  }
  fence_mbar_init();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // No griddepcontrol.wait here: this kernel follows the split-KV decode
  // kernel, which lets it start as its CTAs exit; it reads only what the
  // kernels before that one wrote (the plan's tiles, q, the caches), all
  // complete before the decode kernel let it start. It waits for the decode
  // kernel at its end, so its own completion still orders later work.
  const uint32_t tmem = *tmem_base_s;

  const int Hkv = p.num_kv_heads;
  const int bs = p.block_size;
  bool failed = false;
  uint32_t issued = 0;

  auto read_unit = [&](uint32_t j, TileUnit &r) {
    const uint32_t s = j % kUnitSlots;
    wait_warp(bar(Lay::B_UF + s), (j / kUnitSlots) & 1u, failed);
    r.stop = 1;
    if (!failed) {
      const volatile int *u = units + 8 * s;
      r.b = u[0];
      r.row0 = u[1];
      r.npos = u[2];
      r.pos0 = u[3];
      r.kv_end = u[4];
      r.kvh = u[5];
      r.stop = u[6];
    }
    __syncwarp();
    if (lane == 0 && !failed) mbar_arrive(bar(Lay::B_UE + s));
  };
  auto nranges = [&](const TileUnit &r) { return (r.kv_end + kKeyTile - 1) / kKeyTile; };

  if (warp == kTmaWarp) {
    // ---------------- producer ----------------
    const int total_units = min(max(ld_cg(p.tile_count), 0), p.max_tiles) * Hkv;
    constexpr int MAXROWS = KV8 ? kRawBoxRows : kTileKeys;
    const int box_rows = bs < MAXROWS ? bs : MAXROWS;
    const int nbk = kKeyTile / box_rows;
    uint32_t j = 0, g = 0;
    for (;;) {
      int u = 0;
      if (lane == 0) u = atomicAdd(p.tile_counter, 1);
      u = __shfl_sync(FULL, u, 0);
      TileUnit r{0, 0, 0, 0, 0, 0, u >= total_units ? 1 : 0};
      if (!r.stop) {
        const int item = u / Hkv;
        r.kvh = u - item * Hkv;
        const int4 r0 = ld_cg(p.tiles + 2 * item);
        const int4 r1 = ld_cg(p.tiles + 2 * item + 1);
        r.b = r0.x;
        r.row0 = r0.y;
        r.npos = r0.z;
        r.pos0 = r0.w;
        r.kv_end = r1.y;
        const bool sane = r.b >= 0 && r.b < p.num_seqs && r.npos >= 1 && r.npos <= POS && r.row0 >= 0 &&
                          r.row0 + r.npos <= p.total_q && r.pos0 >= 0 && r.kv_end == r.pos0 + r.npos &&
                          r.kv_end <= static_cast<int64_t>(p.max_blocks_per_seq) * bs;
        if (!sane) {
          if (lane == 0) flag_error(p.status, PA_FLAG_LENGTHS);
          continue;
        }
      }
      const uint32_t s = j % kUnitSlots;
      if (j >= kUnitSlots) wait_warp(bar(Lay::B_UE + s), (j / kUnitSlots - 1) & 1u, failed);
      if (failed) break;
      if (lane == 0) {
        volatile int *d = units + 8 * s;
        d[0] = r.b;
        d[1] = r.row0;
        d[2] = r.npos;
        d[3] = r.pos0;
        d[4] = r.kv_end;
        d[5] = r.kvh;
        d[6] = r.stop;
        mbar_arrive(bar(Lay::B_UF + s));
      }
      __syncwarp();
      ++j;
      if (r.stop) break;
      const int32_t *table = p.block_tables + static_cast<int64_t>(r.b) * p.max_blocks_per_seq;
      auto box_z = [&](int key, int rows) {
        if (key >= r.kv_end) return -rows;
        const int phys = __ldg(table + (key >> p.block_shift));
        if (phys < 0 || phys >= p.num_blocks) {
          flag_error(p.status, PA_FLAG_BLOCK_RANGE);
          return -rows;
        }
        return (phys << p.block_shift) + (key & (bs - 1));
      };
      const int nkt = nranges(r);
      for (int kt = 0; kt < nkt && !failed; ++kt) {
        const int z = lane < nbk ? box_z(kt * kKeyTile + lane * box_rows, box_rows) : 0;
        for (int v = 0; v < LPR && !failed; ++v) {
          const uint32_t slot = g % SLOTS, use = g / SLOTS;
          if (use > 0) wait_warp(bar(Lay::B_EMPTY + slot), (use - 1) & 1u, failed);
          if (failed) break;
          const void *map = v >= 2 ? static_cast<const void *>(&vmap) : static_cast<const void *>(&kmap);
          const int x0 = (v & 1) * 128;  // first element of the unit's half of d
          const uint32_t dst = sRing + slot * Lay::UNIT_BYTES;
          if constexpr (KV8) {
            const uint32_t b8 = bar(Lay::B_RAW + slot);
            if (lane == 0) mbar_arrive_expect_tx(b8, RAW_BYTES);
            __syncwarp();
            if (lane < nbk) tma_load_3d(dst + RAW_OFF + lane * box_rows * RAW_ROW, map, b8, x0, r.kvh, z);
          } else {
            const uint32_t bf = bar(Lay::B_FULL + slot);
            if (lane == 0) mbar_arrive_expect_tx(bf, Lay::UNIT_BYTES);
            __syncwarp();
            if (lane < nbk) {
#pragma unroll
              for (int a = 0; a < 2; ++a)
                tma_load_3d(dst + a * Lay::KV_ATOM + lane * box_rows * 128, map, bf, x0 + a * 64, r.kvh, z);
            }
          }
          __syncwarp();
          issued = ++g;
        }
      }
      if (failed) break;
    }
  } else if (warp >= kConvWarp && warp < kSoftmaxWarp0) {
    // ---------------- 8-bit caches: widen staged codes to fp16 in place (unit by unit) ----------------
    if constexpr (KV8) {
      constexpr int CPR = RAW_ROW / 16;
      constexpr int ROWS_PASS = 8 * (8 / CPR);
      constexpr int PASSES = kKeyTile / ROWS_PASS;
      const int ct = (warp - kConvWarp) * 32 + lane;
      const int q8 = ct >> 3, c = q8 % CPR, rsub = (q8 / CPR) * 8 + (ct & 7);
      uint32_t j = 0, g = 0;
      for (;;) {
        TileUnit r;
        read_unit(j++, r);
        if (failed || r.stop) break;
        const int nkt = nranges(r);
        for (int i = 0; i < LPR * nkt && !failed; ++i, ++g) {
          const uint32_t slot = g % SLOTS, use = g / SLOTS;
          wait_warp(bar(Lay::B_RAW + slot), use & 1u, failed);
          if (failed) break;
          const uint32_t sbase = sRing + slot * Lay::UNIT_BYTES;
          uint4 codes[PASSES];
#pragma unroll
          for (int i2 = 0; i2 < PASSES; ++i2) {
            const int rr = i2 * ROWS_PASS + rsub;
            const uint32_t a = sbase + RAW_OFF + rr * 128 + (((c ^ rr) & 7) << 4);
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];\n"
                         : "=r"(codes[i2].x), "=r"(codes[i2].y), "=r"(codes[i2].z), "=r"(codes[i2].w)
                         : "r"(a));
          }
          mbar_arrive(bar(Lay::B_CONV + slot));
          wait_warp(bar(Lay::B_CONV + slot), use & 1u, failed);
          if (failed) break;
#pragma unroll
          for (int i2 = 0; i2 < PASSES; ++i2) {
            const int rr = i2 * ROWS_PASS + rsub;
            const uint32_t w[4] = {codes[i2].x, codes[i2].y, codes[i2].z, codes[i2].w};
            uint32_t hh[8];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              asm("{\n .reg .b16 l, u;\n mov.b32 {l, u}, %2;\n cvt.rn.f16x2.e4m3x2 %0, l;\n"
                  " cvt.rn.f16x2.e4m3x2 %1, u;\n}\n"
                  : "=r"(hh[2 * k]), "=r"(hh[2 * k + 1])
                  : "r"(w[k]));
            }
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};\n" ::"r"(sbase + TL::off(rr, 2 * c, TL::KV_ATOM)),
                         "r"(hh[0]), "r"(hh[1]), "r"(hh[2]), "r"(hh[3])
                         : "memory");
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};\n" ::"r"(
                             sbase + TL::off(rr, 2 * c + 1, TL::KV_ATOM)),
                         "r"(hh[4]), "r"(hh[5]), "r"(hh[6]), "r"(hh[7])
                         : "memory");
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(Lay::B_FULL + slot));
        }
        if (failed) break;
      }
    }
  } else if (warp == kMmaWarp) {
    // ---------------- MMA issue ----------------
    // Ranges run S(0), S(1), then per range r: P V(r) (once P(r) is written)
    // and S(r + 2) into the score buffer P V(r) read (the products one thread
    // issues execute in issue order). Range number gr = (ranges of earlier
    // units) + r counts across units: its score buffer is gr % 2 and that
    // buffer's barriers complete once per use, phase gr / 2.
    constexpr uint32_t DHI = desc_hi(1024);
    const uint32_t q_lo = desc_lo(sQ, 16);
    const uint32_t k_lo = desc_lo(sRing, 16), v_lo = desc_lo(sRing, Lay::KV_ATOM);
    constexpr uint32_t SLOT_STEP = Lay::UNIT_BYTES >> 4;
    uint32_t ph = 0, ring0 = 0;
    for (uint32_t j = 0;; ++j) {
      TileUnit r;
      read_unit(j, r);
      if (failed || r.stop) break;
      const int nkt = nranges(r);
      auto slot_of = [&](int kt, int u) { return (ring0 + LPR * kt + u) % SLOTS; };
      auto full_parity = [&](int kt, int u) { return ((ring0 + LPR * kt + u) / SLOTS) & 1u; };
      auto mma_s = [&](int kt) {
        wait_warp(bar(Lay::B_FULL + slot_of(kt, 0)), full_parity(kt, 0), failed);
        wait_warp(bar(Lay::B_FULL + slot_of(kt, 1)), full_parity(kt, 1), failed);
        if (failed) return;
        if (lane == 0) {
          tc_fence_after();
          const uint32_t gr = ph + kt;
          const uint32_t d = tmem + Tm::SP0 + (gr & 1u) * kKeyTile;
          const uint32_t klo0 = k_lo + slot_of(kt, 0) * SLOT_STEP, klo1 = k_lo + slot_of(kt, 1) * SLOT_STEP;
#pragma unroll
          for (int ks = 0; ks < KSTEPS_S; ++ks) {
            const uint32_t qo = ((ks >> 2) * Lay::Q_ATOM + (ks & 3) * 32) >> 4;
            const uint32_t ko = (((ks >> 2) & 1) * Lay::KV_ATOM + (ks & 3) * 32) >> 4;
            const uint32_t kb = ks < 8 ? klo0 : klo1;
            if (ks == 0)
              mma_ss<0>(d, q_lo + qo, DHI, kb + ko, DHI, IDESC_S);
            else
              mma_ss<1>(d, q_lo + qo, DHI, kb + ko, DHI, IDESC_S);
          }
          tc_commit(bar(Lay::B_S + (gr & 1u)));
          tc_commit(bar(Lay::B_EMPTY + slot_of(kt, 0)));
          tc_commit(bar(Lay::B_EMPTY + slot_of(kt, 1)));
        }
        __syncwarp();
      };
      wait_warp(bar(Lay::B_QF), j & 1u, failed);
      if (lane == 0 && !failed) mbar_arrive(bar(Lay::B_QE));
      if (failed) break;
      if (nkt > 0) mma_s(0);
      if (nkt > 1) mma_s(1);
      for (int kt = 0; kt < nkt && !failed; ++kt) {
        const uint32_t gr = ph + kt;
        wait_warp(bar(Lay::B_P + (gr & 1u)), (gr >> 1) & 1u, failed);  // P(kt) is in place
        const uint32_t vs0 = slot_of(kt, 2), vs1 = slot_of(kt, 3);
        wait_warp(bar(Lay::B_FULL + vs0), full_parity(kt, 2), failed);
        wait_warp(bar(Lay::B_FULL + vs1), full_parity(kt, 3), failed);
        if (failed) break;
        const int key0 = kt * kKeyTile;
        if (key0 + kKeyTile > r.kv_end) {
          // rows of keys past kv_end may hold anything (even NaN): zero them in both V units
          const int vr0 = r.kv_end - key0;
          const int n = (kKeyTile - vr0) * 16;  // 16 chunks of 16 bytes per row and unit
          for (int i = lane; i < 2 * n; i += 32) {
            const int unit = i / n, ii = i - unit * n;
            const int rr = vr0 + ii / 16, c = ii % 16;
            const uint32_t sV = sRing + (unit ? vs1 : vs0) * Lay::UNIT_BYTES;
            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};\n" ::"r"(sV + TL::off(rr, c, TL::KV_ATOM)),
                         "r"(0u)
                         : "memory");
          }
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) {
          tc_fence_after();
          const uint32_t sp = tmem + Tm::SP0 + (gr & 1u) * kKeyTile;
          const uint32_t v0 = v_lo + vs0 * SLOT_STEP, v1 = v_lo + vs1 * SLOT_STEP;
          // P of K step ks: SPLIT hi at 16 ks, lo at 16 ks + 8; else 8 ks (+ 32 for the second warp's keys)
          auto pcol = [](int ks) { return SPLIT ? 16 * ks : 8 * ks + (ks >= 4 ? 32 : 0); };
#pragma unroll
          for (int ks = 0; ks < KSTEPS_O; ++ks) {
            const uint32_t vo = (ks * 2048) >> 4;
            const uint32_t a = sp + pcol(ks);
            if (kt == 0 && ks == 0) {  // the unit's first products overwrite O
              mma_ts<0>(tmem + Tm::O, a, v0 + vo, DHI, IDESC_O);
              mma_ts<0>(tmem + Tm::O + 128, a, v1 + vo, DHI, IDESC_O);
            } else {
              mma_ts<1>(tmem + Tm::O, a, v0 + vo, DHI, IDESC_O);
              mma_ts<1>(tmem + Tm::O + 128, a, v1 + vo, DHI, IDESC_O);
            }
            if (SPLIT) {
              mma_ts<1>(tmem + Tm::O, a + 8, v0 + vo, DHI, IDESC_O);
              mma_ts<1>(tmem + Tm::O + 128, a + 8, v1 + vo, DHI, IDESC_O);
            }
          }
          tc_commit(bar(Lay::B_O));
          tc_commit(bar(Lay::B_EMPTY + vs0));
          tc_commit(bar(Lay::B_EMPTY + vs1));
        }
        __syncwarp();
        if (kt + 2 < nkt) mma_s(kt + 2);
      }
      if (failed) break;
      ph += nkt;
      ring0 += LPR * nkt;
    }
  } else if (warp >= kSoftmaxWarp0) {
    // ---------------- softmax: one row per thread, 64 keys of each range per warp ----------------
    const int sw = warp - kSoftmaxWarp0;
    const int quad = sw & 3, part = sw >> 2;
    const int r = quad * 32 + lane;  // row = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t bx1 = bar(Lay::B_X1 + quad), bx2 = bar(Lay::B_X2 + quad);
    volatile float *x_mine = xch + (part * 4 + quad) * 32 + lane;
    volatile float *x_other = xch + ((1 - part) * 4 + quad) * 32 + lane;
    uint32_t nx = 0;
    // my value out, the other warp's value in; x2 (its read of the last
    // exchange) is waited for only before the next write
    auto exchange = [&](float v) -> float {
      if (nx > 0) wait_warp(bx2, (nx - 1) & 1u, failed);
      *x_mine = v;
      mbar_arrive(bx1);
      wait_warp(bx1, nx & 1u, failed);
      const float o = failed ? v : *x_other;
      mbar_arrive(bx2);
      ++nx;
      return o;
    };
    const int g = r % G;
    const int qi = r / G;
    auto load_q = [&](const TileUnit &u) -> float {
      const bool valid = qi < u.npos;
      const bf16 *qrow = p.q + static_cast<int64_t>(u.row0 + (valid ? qi : 0)) * p.q_stride +
                         static_cast<int64_t>(u.kvh * G + g) * D;
      const bool q16 = (reinterpret_cast<uintptr_t>(p.q) & 15u) == 0 && (p.q_stride & 7) == 0;
      auto ldq = [&](int c) {
        uint4 w = make_uint4(0u, 0u, 0u, 0u);
        if (valid) {
          if (q16) {
            w = __ldg(reinterpret_cast<const uint4 *>(qrow) + c);
          } else {
            const uint32_t *q32 = reinterpret_cast<const uint32_t *>(qrow) + 4 * c;
            w = make_uint4(__ldg(q32), __ldg(q32 + 1), __ldg(q32 + 2), __ldg(q32 + 3));
          }
        }
        return w;
      };
      float sl2 = p.scale_log2;
      float qmul = 1.f;
      if constexpr (KV8 && std::is_same<E, ElemBf16>::value) {
        float amax = 0.f;
#pragma unroll 4
        for (int c = 0; c < D / 8; ++c) {
          const uint4 w = ldq(c);
          const uint32_t v[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int k = 0; k < 4; ++k)
            amax = fmaxf(amax, fmaxf(fabsf(ElemBf16::lo(v[k])), fabsf(ElemBf16::hi(v[k]))));
        }
        const int ex = static_cast<int>((__float_as_uint(amax) >> 23) & 0xffu) - 127;
        const int e = ex >= 15 ? min(ex - 14, 120) : 0;
        qmul = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
        sl2 *= __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
      }
      constexpr int CQ = D / 16;  // this warp's half of the row's 16-byte chunks
#pragma unroll 4
      for (int c = part * CQ; c < (part + 1) * CQ; ++c) {
        uint4 w = ldq(c);
        if constexpr (KV8 && std::is_same<E, ElemBf16>::value) {
          w = make_uint4(ElemFp16::pack(ElemBf16::lo(w.x) * qmul, ElemBf16::hi(w.x) * qmul),
                         ElemFp16::pack(ElemBf16::lo(w.y) * qmul, ElemBf16::hi(w.y) * qmul),
                         ElemFp16::pack(ElemBf16::lo(w.z) * qmul, ElemBf16::hi(w.z) * qmul),
                         ElemFp16::pack(ElemBf16::lo(w.w) * qmul, ElemBf16::hi(w.w) * qmul));
        }
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};\n" ::"r"(sQ + TL::off(r, c, Lay::Q_ATOM)),
                     "r"(w.x), "r"(w.y), "r"(w.z), "r"(w.w)
                     : "memory");
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(Lay::B_QF));
      return sl2;
    };

    uint32_t ph = 0;
    TileUnit cur;
    read_unit(0, cur);
    float sl2 = 0.f;
    if (!failed && !cur.stop) sl2 = load_q(cur);
    for (uint32_t j = 0; !failed && !cur.stop; ++j) {
      const int nk = nranges(cur);
      const bool row_valid = qi < cur.npos;
      const int lim = row_valid ? cur.pos0 + qi + 1 : 0;
      float m_used = -INFINITY, l = 0.f;
      for (int kt = 0; kt < nk; ++kt) {
        const uint32_t gr = ph + kt;
        const int ck0 = kt * kKeyTile + part * 64;
        const uint32_t sp = tmem + lane_off + Tm::SP0 + (gr & 1u) * kKeyTile + part * 64;
        wait_warp(bar(Lay::B_S + (gr & 1u)), (gr >> 1) & 1u, failed);
        if (failed) break;
        tc_fence_after();
        uint32_t s0[32], s1[32];
        tmem_ld32x2_wait(sp, s0, s1);
        const float mx = fmaxf(masked_max32(s0, ck0, lim), masked_max32(s1, ck0 + 32, lim));
        const float mo = exchange(mx);
        if (failed) break;
        const float cm = __fmul_rn(sl2, fmaxf(mx, mo));
        const bool grow = cm > -INFINITY && (m_used == -INFINITY || __fsub_rn(cm, m_used) > kRescaleLog2);
        float alpha = 1.f;
        if (grow) {
          alpha = m_used > -INFINITY ? ex2_approx(__fsub_rn(m_used, cm)) : 1.f;
          m_used = cm;
        }
        const float ms = m_used == -INFINITY ? 0.f : m_used;
        float sum = 0.f;
        constexpr uint32_t PSTEP = SPLIT ? 16 : 8;
        if (__any_sync(FULL, fabsf(ms) > 4096.f)) {
          probs16_store<M, true, SPLIT>(s0, ck0, lim, sl2, ms, sum, sp);
          probs16_store<M, true, SPLIT>(s0 + 16, ck0 + 16, lim, sl2, ms, sum, sp + PSTEP);
        } else {
          probs16_store<M, false, SPLIT>(s0, ck0, lim, sl2, ms, sum, sp);
          probs16_store<M, false, SPLIT>(s0 + 16, ck0 + 16, lim, sl2, ms, sum, sp + PSTEP);
        }
        tmem_ld32_wait(sp + 32, s1);
        if (__any_sync(FULL, fabsf(ms) > 4096.f)) {
          probs16_store<M, true, SPLIT>(s1, ck0 + 32, lim, sl2, ms, sum, sp + 2 * PSTEP);
          probs16_store<M, true, SPLIT>(s1 + 16, ck0 + 48, lim, sl2, ms, sum, sp + 3 * PSTEP);
        } else {
          probs16_store<M, false, SPLIT>(s1, ck0 + 32, lim, sl2, ms, sum, sp + 2 * PSTEP);
          probs16_store<M, false, SPLIT>(s1 + 16, ck0 + 48, lim, sl2, ms, sum, sp + 3 * PSTEP);
        }
        // O holds P V(0 .. kt-1) once P V(kt-1) completes (S(kt) may have been
        // issued before it): wait for it only when O must be rescaled
        if (kt > 0 && __any_sync(FULL, alpha != 1.f)) {
          wait_warp(bar(Lay::B_O), (gr - 1) & 1u, failed);
          if (failed) break;
          tc_fence_after();
#pragma unroll 1
          for (int ch = part * 4; ch < part * 4 + 4; ++ch) {
            uint32_t t[32];
            tmem_ld32_wait(tmem + lane_off + Tm::O + ch * 32, t);
#pragma unroll
            for (int i = 0; i < 32; ++i) t[i] = __float_as_uint(__uint_as_float(t[i]) * alpha);
            tmem_st32u(tmem + lane_off + Tm::O + ch * 32, t);
          }
        }
        l = l * alpha + sum;
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(Lay::B_P + (gr & 1u)));
      }
      if (failed) break;
      TileUnit nxt;
      read_unit(j + 1, nxt);
      float nsl2 = sl2;
      if (!failed && !nxt.stop) {
        wait_warp(bar(Lay::B_QE), j & 1u, failed);
        if (!failed) nsl2 = load_q(nxt);
      }
      if (failed) break;
      if (nk > 0) {
        const float lt = l + exchange(l);
        wait_warp(bar(Lay::B_O), (ph + nk - 1) & 1u, failed);
        if (failed) break;
        tc_fence_after();
        const float inv = lt > 0.f ? p.out_scale / lt : 0.f;
        bf16 *dst = p.out + static_cast<int64_t>(cur.row0 + (row_valid ? qi : 0)) * p.num_heads * D +
                    static_cast<int64_t>(cur.kvh * G + g) * D;
#pragma unroll 1
        for (int ch = part * 4; ch < part * 4 + 4; ++ch) {
          uint32_t t[32];
          tmem_ld32_wait(tmem + lane_off + Tm::O + ch * 32, t);
          if (row_valid) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const float *f = reinterpret_cast<const float *>(&t[8 * c]);
              const uint4 v = make_uint4(E::pack(f[0] * inv, f[1] * inv), E::pack(f[2] * inv, f[3] * inv),
                                         E::pack(f[4] * inv, f[5] * inv), E::pack(f[6] * inv, f[7] * inv));
              *reinterpret_cast<uint4 *>(dst + ch * 32 + 8 * c) = v;
            }
          }
        }
        tc_fence_before();
      }
      ph += nk;
      cur = nxt;
      sl2 = nsl2;
    }
  }

  if (warp == kMmaWarp && lane == 0) {
    tc_commit(bar(Lay::B_DRAIN));
    if (!mbar_wait_bounded(bar(Lay::B_DRAIN), 0, kTcWaitTimeoutNs)) failed = true;
  }
  if (warp == kTmaWarp && lane == 0) {
    const int landed = KV8 ? Lay::B_RAW : Lay::B_FULL;
    for (uint32_t g = issued > SLOTS ? issued - SLOTS : 0; g < issued; ++g)
      if (!mbar_wait_bounded(bar(landed + static_cast<int>(g % SLOTS)), (g / SLOTS) & 1u, kTcWaitTimeoutNs))
        failed = true;
  }
  if (failed) flag_error(p.status, PA_FLAG_TIMEOUT);
  griddep_wait();  // the decode kernel before this one has completed
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

template <int D, int G, typename E, bool KV8>
cudaError_t launch_prefill_tiles(const CUtensorMap &kmap, const CUtensorMap &vmap, const CUtensorMap &vmapb,
                                 const TileParams &tp, int sm_count, cudaStream_t stream) {
  if constexpr (D == kWideD) {
    (void)vmapb;
    constexpr int smem = WideLayout::BYTES;
    auto kern = prefill_tile_wide_kernel<G, E, KV8>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (err != cudaSuccess) return err;
    int64_t grid = sm_count;
    const int64_t units = static_cast<int64_t>(tp.max_tiles) * tp.num_kv_heads;
    if (grid > units) grid = units;
    if (grid < 1) grid = 1;
    return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(kWideThreads), smem, stream, kmap, vmap, tp);
  } else {
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
    return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(KV8 ? kTileThreads8 : kTileThreads), smem,
                      stream, kmap, vmap, vmapb, tp);
  }
}

#define PA_TILE_INST1(DD, GG, EE, K8)                                                                   \
  template cudaError_t launch_prefill_tiles<DD, GG, EE, K8>(const CUtensorMap &, const CUtensorMap &,     \
                                                            const CUtensorMap &, const TileParams &, int, \
                                                            cudaStream_t);
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
PA_TILE_INST(256, 1)
PA_TILE_INST(256, 2)
PA_TILE_INST(256, 4)
PA_TILE_INST(256, 8)
#undef PA_TILE_INST
#undef PA_TILE_INST1

}  // namespace pa
