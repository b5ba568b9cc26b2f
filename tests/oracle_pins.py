"""Checks that pin the CPU oracle to facts other than itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError on a
mismatch. ``test_oracle_pins.py`` runs them against the oracle; the mutant test
runs them against deliberately broken copies of it and expects each copy to
fail at least one pin.

What pins what:
  * dense brute force: scaled_dot_product_attention from PyTorch (float64, CPU,
    explicit causal mask, GQA by repeat-interleave) on contiguous K/V, against
    the oracle reading the same rows scattered into a shuffled block pool;
  * closed forms: seq_len 1 gives the V row, constant V gives V, q = 0 gives
    the mean of the visible V rows, two keys give logistic weights;
  * invariants: physical block permutation, causal future perturbation, GQA
    equals MHA with replicated KV heads, weights sum to one;
  * the slot address formula, from the golden fixture;
  * the element decoders: fp16 against numpy's IEEE binary16 on all 65536 bit
    patterns, bf16 at values the format fixes (1, -2, pi rounded, the largest
    finite, the smallest subnormal, signed zero, infinities, NaN); the dense
    brute force and the seq_len-1 closed form are repeated on fp16 data;
  * 8-bit (E4M3) cache codes: decoding against PyTorch's float8_e4m3fn on all
    256 codes; rounding against PyTorch's cast inside the finite range (random
    values, every tie, values next to every tie) and against the format's
    closed forms at saturation, zero, signed zero, subnormal ties and NaN; the
    quantiser against a numpy binary32 division followed by that cast; the
    quantising scatter against a numpy scatter; attention over 8-bit caches
    against float64 SDPA over the decoded values times the scales.
"""

from __future__ import annotations

import math
import os

import numpy as np
import torch

from paged_kv_cache_55_gb300.workloads import (NAN_BITS, bf16_bits_to_f32, bits_to_f32, f32_to_bf16_bits, f32_to_bits,
                                               rope_cos_sin_cache)

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_golden(name: str) -> np.ndarray:
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([int(x) for x in line.split()])
    return np.array(rows, dtype=np.int64)


# --------------------------------------------------------------------------
# A test-local problem builder: dense per-request K/V first, then a paged pool
# --------------------------------------------------------------------------

class DenseProblem:
    """Contiguous K/V per request plus the same rows scattered into a shuffled pool."""

    def __init__(self, rng, ctx_lens, q_lens, H, Hkv, D, bs=16, extra_blocks=3, q_scale=1.0,
                 perm=None, dtype="bf16"):
        self.H, self.Hkv, self.D, self.bs = H, Hkv, D, bs
        self.dtype = dtype
        self.ctx = list(ctx_lens)
        self.ql = list(q_lens)
        self.L = [c + q for c, q in zip(self.ctx, self.ql)]
        B = len(self.L)
        nblk = [(x + bs - 1) // bs for x in self.L]
        self.num_blocks = sum(nblk) + extra_blocks
        self.kd = [f32_to_bits(rng.standard_normal((x, Hkv, D)).astype(np.float32), dtype) for x in self.L]
        self.vd = [f32_to_bits(rng.standard_normal((x, Hkv, D)).astype(np.float32), dtype) for x in self.L]
        T = sum(self.ql)
        self.q = f32_to_bits((q_scale * rng.standard_normal((T, H, D))).astype(np.float32), dtype)
        self.qsl = np.zeros(B + 1, dtype=np.int32)
        self.qsl[1:] = np.cumsum(self.ql)
        self.seq_lens = np.array(self.L, dtype=np.int32)
        self.perm = rng.permutation(self.num_blocks) if perm is None else np.asarray(perm)
        self.max_blocks = max(nblk + [1]) + 1
        self.scale = float(np.float32(1.0 / math.sqrt(D)))
        self.repack()

    def repack(self):
        """Write the dense rows into a pool whose unowned slots hold NaN."""
        bs = self.bs
        self.bt = np.full((len(self.L), self.max_blocks), -7, dtype=np.int32)
        self.kc = np.full((self.num_blocks, bs, self.Hkv, self.D), NAN_BITS[self.dtype], dtype=np.uint16)
        self.vc = np.full_like(self.kc, NAN_BITS[self.dtype])
        cursor = 0
        for b, L in enumerate(self.L):
            for i in range((L + bs - 1) // bs):
                self.bt[b, i] = self.perm[cursor]
                cursor += 1
            for j in range(L):
                blk = self.bt[b, j // bs]
                self.kc[blk, j % bs] = self.kd[b][j]
                self.vc[blk, j % bs] = self.vd[b][j]

    def run(self, oracle, num_threads=2):
        return oracle.attention(self.q, self.kc, self.vc, self.bt, self.seq_lens, self.qsl,
                                self.H, self.scale, num_threads=num_threads, dtype=self.dtype)

    def sdpa(self):
        """PyTorch SDPA per request in float64 with a bottom-right causal mask."""
        out = np.zeros((int(self.qsl[-1]), self.H, self.D), dtype=np.float64)
        for b, L in enumerate(self.L):
            q0, ql = int(self.qsl[b]), self.ql[b]
            if ql == 0:
                continue
            qb = torch.from_numpy(bits_to_f32(self.q[q0:q0 + ql], self.dtype).astype(np.float64)).transpose(0, 1)
            kb = torch.from_numpy(bits_to_f32(self.kd[b], self.dtype).astype(np.float64)).transpose(0, 1)
            vb = torch.from_numpy(bits_to_f32(self.vd[b], self.dtype).astype(np.float64)).transpose(0, 1)
            i = torch.arange(ql).unsqueeze(1)
            j = torch.arange(L).unsqueeze(0)
            mask = j <= (L - ql) + i
            o = torch.nn.functional.scaled_dot_product_attention(
                qb.unsqueeze(0), kb.unsqueeze(0), vb.unsqueeze(0), attn_mask=mask,
                scale=self.scale, enable_gqa=(self.H != self.Hkv))
            out[q0:q0 + ql] = o[0].transpose(0, 1).numpy()
        return out


# --------------------------------------------------------------------------
# The pins
# --------------------------------------------------------------------------

DENSE_CASES = [
    # (ctx_lens, q_lens, H, Hkv, D, bs)
    ([0, 6, 15, 32], [1, 1, 1, 1], 4, 1, 64, 16),
    ([3, 17, 0], [5, 2, 9], 8, 2, 8, 16),
    ([30, 1], [10, 4], 8, 8, 4, 16),
    ([12, 0, 21], [3, 0, 7], 16, 2, 8, 8),
    ([33], [7], 8, 1, 4, 4),
]


def pin_dense_vs_sdpa(oracle, dtype="bf16"):
    rng = np.random.default_rng(11)
    for ctx, ql, H, Hkv, D, bs in DENSE_CASES:
        p = DenseProblem(rng, ctx, ql, H, Hkv, D, bs, dtype=dtype)
        got = p.run(oracle)
        ref = p.sdpa()
        err = float(np.max(np.abs(got - ref))) if got.size else 0.0
        assert err <= 1e-12, f"oracle vs SDPA max |diff| {err} for case {(ctx, ql, H, Hkv, D, bs)} ({dtype})"


def pin_dense_vs_sdpa_fp16(oracle):
    pin_dense_vs_sdpa(oracle, dtype="fp16")


def pin_sampled_equals_full(oracle):
    """attention_sampled, the reference of the full-size GPU checks, equals attention at every
    (token, head) pair asked for in any order, bit for bit (the same definition, evaluated the
    same way), on the dense shapes above (so it inherits their agreement with SDPA)."""
    rng = np.random.default_rng(15)
    for k, (ctx, ql, H, Hkv, D, bs) in enumerate(DENSE_CASES):
        dtype = "fp16" if k % 2 else "bf16"
        p = DenseProblem(rng, ctx, ql, H, Hkv, D, bs, dtype=dtype)
        full = p.run(oracle)
        T = int(p.qsl[-1])
        if T == 0:
            continue
        order = rng.permutation(T * H)
        tokens, heads = (order // H).astype(np.int64), (order % H).astype(np.int32)
        got = oracle.attention_sampled(p.q, p.kc, p.vc, p.bt, p.seq_lens, p.qsl, H, p.scale, tokens, heads,
                                       dtype=dtype)
        assert np.array_equal(got, full[tokens, heads]), f"sampled != full for case {(ctx, ql, H, Hkv, D, bs)}"


def pin_block_permutation_invariance(oracle):
    rng = np.random.default_rng(12)
    p = DenseProblem(rng, [40, 9, 70], [3, 1, 6], 8, 2, 8, bs=16, extra_blocks=5)
    a = p.run(oracle)
    p.perm = np.random.default_rng(99).permutation(p.num_blocks)
    p.repack()
    b = p.run(oracle)
    assert np.array_equal(a, b), "output changed under a permutation of physical block ids"


def pin_seq_len_one_is_v_row(oracle, dtype="bf16"):
    rng = np.random.default_rng(13)
    p = DenseProblem(rng, [0, 0], [1, 1], 4, 2, 64, dtype=dtype)
    out = p.run(oracle)
    for b in range(2):
        for h in range(4):
            v = bits_to_f32(p.vd[b][0, h // 2], dtype).astype(np.float64)
            assert np.array_equal(out[b, h], v), f"seq_len 1 must return the V row exactly ({dtype})"


def pin_seq_len_one_is_v_row_fp16(oracle):
    pin_seq_len_one_is_v_row(oracle, dtype="fp16")


def pin_fp16_decoding_matches_ieee(oracle):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode_elements(bits, "fp16")
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan), "fp16 NaN patterns must decode to NaN"
    assert np.array_equal(got[~nan], ref[~nan]), "fp16 decoding must match IEEE binary16"
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan])), "fp16 signs (incl. -0)"


def pin_bf16_decoding_special_values(oracle):
    cases = [(0x3F80, 1.0), (0xC000, -2.0), (0x4049, 3.140625), (0x0001, 2.0 ** -133),
             (0x7F7F, (2.0 - 2.0 ** -7) * 2.0 ** 127), (0x0080, 2.0 ** -126), (0x0000, 0.0), (0x8000, -0.0),
             (0x7F80, math.inf), (0xFF80, -math.inf)]
    bits = np.array([c[0] for c in cases] + [0x7FC0], dtype=np.uint16)
    got = oracle.decode_elements(bits, "bf16")
    for (h, v), g in zip(cases, got[:-1]):
        assert g == v and math.copysign(1.0, g) == math.copysign(1.0, v), f"bf16 {h:#06x} must be {v}, got {g}"
    assert math.isnan(got[-1]), "bf16 0x7FC0 is a NaN"


def pin_constant_v(oracle):
    rng = np.random.default_rng(14)
    p = DenseProblem(rng, [25, 3], [4, 1], 4, 1, 8)
    c = f32_to_bf16_bits(rng.standard_normal(8).astype(np.float32))
    for b in range(2):
        p.vd[b][:] = c
    p.repack()
    out = p.run(oracle)
    cv = bf16_bits_to_f32(c).astype(np.float64)
    assert np.max(np.abs(out - cv)) <= 1e-14, "constant V must give V"


def pin_zero_q_mean(oracle):
    rng = np.random.default_rng(15)
    p = DenseProblem(rng, [19, 5], [3, 2], 4, 2, 8)
    p.q[:] = 0
    out = p.run(oracle)
    for b in range(2):
        q0, ql, L = int(p.qsl[b]), p.ql[b], p.L[b]
        for i in range(ql):
            n = L - ql + i + 1
            for h in range(4):
                mean = bf16_bits_to_f32(p.vd[b][:n, h // 2]).astype(np.float64).mean(axis=0)
                assert np.max(np.abs(out[q0 + i, h] - mean)) <= 1e-14, "q = 0 must average the visible V rows"


def pin_two_keys_logistic(oracle):
    # One head, D = 4, scale 1: scores are q . k exactly (bf16-exact values),
    # so the weights are the logistic function of the score gap.
    for a, c in [(1.0, 0.0), (2.5, -1.25), (-3.0, 4.0), (0.0, 0.0), (10.0, -6.0)]:
        q = f32_to_bf16_bits(np.array([[[1, 0, 0, 0]]], dtype=np.float32))
        kc = np.full((2, 4, 1, 4), 0x7FC0, dtype=np.uint16)
        vc = np.full_like(kc, 0x7FC0)
        kc[1, 0, 0] = f32_to_bf16_bits(np.array([a, 0, 0, 0], dtype=np.float32))
        kc[1, 1, 0] = f32_to_bf16_bits(np.array([c, 0, 0, 0], dtype=np.float32))
        vc[1, 0, 0] = f32_to_bf16_bits(np.array([1, 0, 0, 0], dtype=np.float32))
        vc[1, 1, 0] = f32_to_bf16_bits(np.array([0, 1, 0, 0], dtype=np.float32))
        bt = np.array([[1, 0]], dtype=np.int32)
        out = oracle.attention(q, kc, vc, bt, np.array([2], np.int32), np.array([0, 1], np.int32),
                               1, 1.0, num_threads=1)
        w0 = 1.0 / (1.0 + math.exp(-(a - c)))
        assert abs(out[0, 0, 0] - w0) <= 1e-15 and abs(out[0, 0, 1] - (1.0 - w0)) <= 1e-15, \
            f"two-key weights must be logistic in the score gap ({a}, {c})"
        assert out[0, 0, 2] == 0.0 and out[0, 0, 3] == 0.0


def pin_weights_sum_to_one(oracle):
    rng = np.random.default_rng(16)
    p = DenseProblem(rng, [50, 7], [5, 1], 8, 2, 16, q_scale=4.0)
    for tok in range(int(p.qsl[-1])):
        for h in (0, 3, 7):
            w = oracle.attention_weights(p.q, p.kc, p.vc, p.bt, p.seq_lens, p.qsl, p.H, p.scale, tok, h)
            assert (w >= 0).all()
            assert abs(w.sum() - 1.0) <= 1e-12, "softmax weights must sum to one"
    # the number of visible keys follows the causal rule
    w = oracle.attention_weights(p.q, p.kc, p.vc, p.bt, p.seq_lens, p.qsl, p.H, p.scale, 2, 0)
    assert w.shape[0] == 50 + 2 + 1


def pin_causal_future_perturbation(oracle):
    rng = np.random.default_rng(17)
    p = DenseProblem(rng, [20], [8], 4, 2, 8)
    base = p.run(oracle)
    i = 3
    pos = 20 + i  # query i sees keys 0 .. 23
    p.kd[0][pos + 1:] = f32_to_bf16_bits(rng.standard_normal(p.kd[0][pos + 1:].shape).astype(np.float32))
    p.vd[0][pos + 1:] = f32_to_bf16_bits(rng.standard_normal(p.vd[0][pos + 1:].shape).astype(np.float32))
    p.repack()
    after = p.run(oracle)
    assert np.array_equal(base[:i + 1], after[:i + 1]), "future keys must not affect a query"
    assert not np.array_equal(base[i + 1:], after[i + 1:]), "later queries must see the changed keys"


def pin_gqa_equals_replicated_mha(oracle):
    rng = np.random.default_rng(18)
    G = 4
    p = DenseProblem(rng, [30, 12], [2, 5], 8, 2, 8)
    gqa = p.run(oracle)
    m = DenseProblem(rng, [30, 12], [2, 5], 8, 8, 8, perm=p.perm)
    m.q = p.q.copy()
    m.kd = [np.repeat(k, G, axis=1) for k in p.kd]
    m.vd = [np.repeat(v, G, axis=1) for v in p.vd]
    m.repack()
    mha = m.run(oracle)
    assert np.array_equal(gqa, mha), "GQA must equal MHA with each KV head repeated for its group"


def pin_slot_formula_golden(oracle):
    rows = read_golden("slot_address.txt")
    for bs, blk, off, slot in rows:
        nb = blk + 2
        kc = np.zeros((nb, bs, 1, 8), dtype=np.uint16)
        vc = np.zeros_like(kc)
        key = np.arange(1, 9, dtype=np.uint16).reshape(1, 1, 8)
        val = key + 100
        oracle.reshape_and_cache(key, val, kc, vc, np.array([slot]), int(bs))
        assert np.array_equal(kc[blk, off, 0], key[0, 0]) and np.array_equal(vc[blk, off, 0], val[0, 0]), \
            f"slot {slot} must land in block {blk} offset {off} (block_size {bs})"
        assert int(np.count_nonzero(kc)) == 8, "exactly one row may change"


def pin_reshape_matches_numpy_scatter(oracle):
    rng = np.random.default_rng(19)
    nb, bs, hkv, d = 20, 16, 3, 8
    kc = np.full((nb, bs, hkv, d), 0x7FC0, dtype=np.uint16)
    vc = kc.copy()
    T = 37
    slots = rng.choice(nb * bs, size=T, replace=False).astype(np.int64)
    slots[5] = -1
    slots[30] = -4
    key = rng.integers(0, 65535, size=(T, hkv, d), dtype=np.uint16)
    val = rng.integers(0, 65535, size=(T, hkv, d), dtype=np.uint16)
    ek, ev = kc.copy(), vc.copy()
    keep = slots >= 0
    ek.reshape(nb * bs, hkv, d)[slots[keep]] = key[keep]
    ev.reshape(nb * bs, hkv, d)[slots[keep]] = val[keep]
    oracle.reshape_and_cache(key, val, kc, vc, slots, bs)
    assert np.array_equal(kc, ek) and np.array_equal(vc, ev), "scatter must match numpy fancy assignment"


def pin_copy_blocks_matches_numpy(oracle):
    rng = np.random.default_rng(20)
    nb, bs, hkv, d = 40, 16, 2, 8
    kc = rng.integers(0, 65535, size=(nb, bs, hkv, d), dtype=np.uint16)
    vc = rng.integers(0, 65535, size=(nb, bs, hkv, d), dtype=np.uint16)
    ids = rng.permutation(nb)
    src, dst = ids[:9], ids[9:18]  # disjoint: no destination is also a source
    ek, ev = kc.copy(), vc.copy()
    ek[dst] = kc[src]
    ev[dst] = vc[src]
    oracle.copy_blocks(kc, vc, np.stack([src, dst], axis=1))
    assert np.array_equal(kc, ek) and np.array_equal(vc, ev), "block copy must match numpy assignment"


def pin_round_fp16_matches_numpy(oracle):
    rng = np.random.default_rng(21)
    x = np.concatenate([
        rng.standard_normal(20000) * 10.0 ** rng.integers(-9, 5, size=20000),
        # exact halfway points between neighbouring fp16 values, and one ulp of a double either side
        (np.arange(1, 2048) + 0.5) * 2.0 ** -24, (np.arange(1024, 2048) + 0.5) * 2.0 ** -9,
        np.nextafter((np.arange(1024, 2048) + 0.5) * 2.0 ** -9, np.inf),
        np.nextafter((np.arange(1024, 2048) + 0.5) * 2.0 ** -9, -np.inf),
        [65504.0, 65519.99, 65520.0, 1e6, -1e6, 0.0, -0.0, np.inf, -np.inf]])
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    got = oracle.round_elements(x, "fp16")
    assert np.array_equal(got, ref), "fp16 rounding must match numpy's float64 -> float16"


def pin_round_bf16_definition_cases(oracle):
    # round to nearest, ties to even, straight from the double (8 significant bits)
    cases = [(1 + 2.0 ** -8, 0x3F80), (1 + 2.0 ** -8 + 2.0 ** -40, 0x3F81), (1 + 3 * 2.0 ** -8, 0x3F82),
             (-(1 + 2.0 ** -9), 0xBF80), (3.4e38, 0x7F80), (2.0 ** -133, 0x0001), (2.0 ** -134, 0x0000),
             (3 * 2.0 ** -135, 0x0001), (-2.0, 0xC000), (np.inf, 0x7F80), (-0.0, 0x8000), (0.1, 0x3DCD)]
    got = oracle.round_elements(np.array([c[0] for c in cases]), "bf16")
    for (x, want), g in zip(cases, got):
        assert int(g) == want, f"bf16 rounding of {x!r}: want {want:#06x}, got {int(g):#06x}"
    # values exact in float32 agree with the float32 -> bf16 rounding of the generator
    f = np.random.default_rng(22).standard_normal(5000).astype(np.float32)
    assert np.array_equal(oracle.round_elements(f.astype(np.float64), "bf16"), f32_to_bf16_bits(f))


class RopeProblem:
    """q, key, value rows of T tokens, a cache to scatter into, positions and a table."""

    def __init__(self, rng, T=6, H=4, Hkv=2, D=32, rot=32, dtype="bf16", table=None, positions=None):
        self.dtype, self.D = dtype, D
        self.q = f32_to_bits(rng.standard_normal((T, H, D)).astype(np.float32), dtype)
        self.k = f32_to_bits(rng.standard_normal((T, Hkv, D)).astype(np.float32), dtype)
        self.v = f32_to_bits(rng.standard_normal((T, Hkv, D)).astype(np.float32), dtype)
        self.nb, self.bs = 4, 4
        self.slots = rng.permutation(self.nb * self.bs)[:T].astype(np.int64)
        self.table = rope_cos_sin_cache(64, rot) if table is None else table
        self.pos = rng.integers(0, self.table.shape[0], size=T) if positions is None else np.asarray(positions)

    def run(self, oracle, is_neox=True):
        q = self.q.copy()
        kc = np.zeros((self.nb, self.bs, self.k.shape[1], self.D), dtype=np.uint16)
        vc = np.zeros_like(kc)
        oracle.rope_reshape_and_cache(q, self.k, self.v, kc, vc, self.slots, self.pos, self.table, is_neox,
                                      self.bs, self.dtype)
        flat_k = kc.reshape(-1, self.k.shape[1], self.D)[self.slots]
        flat_v = vc.reshape(-1, self.k.shape[1], self.D)[self.slots]
        return q, flat_k, flat_v


def pin_rope_position_zero_is_identity(oracle):
    rng = np.random.default_rng(23)
    for dtype in ("bf16", "fp16"):
        p = RopeProblem(rng, dtype=dtype, positions=[0] * 6)
        for neox in (True, False):
            q, k, v = p.run(oracle, neox)
            assert np.array_equal(q, p.q) and np.array_equal(k, p.k) and np.array_equal(v, p.v), \
                "position 0 (cos 1, sin 0) leaves q and k as they are and caches them"


def pin_rope_quarter_turn(oracle):
    # a table row with cos 0 and sin 1 turns every pair (x1, x2) into (-x2, x1)
    rng = np.random.default_rng(24)
    D, rot, half = 32, 16, 8
    table = np.zeros((2, rot), dtype=np.float32)
    table[0, :half] = 1.0
    table[1, half:] = 1.0
    p = RopeProblem(rng, D=D, rot=rot, table=table, positions=[1] * 6)
    x = bits_to_f32(p.q, "bf16")
    kx = bits_to_f32(p.k, "bf16")
    for neox in (True, False):
        q, k, v = p.run(oracle, neox)
        a = np.arange(half) if neox else 2 * np.arange(half)
        b = a + half if neox else a + 1
        for got, src in ((bits_to_f32(q, "bf16"), x), (bits_to_f32(k, "bf16"), kx)):
            assert np.array_equal(got[..., a], -src[..., b]) and np.array_equal(got[..., b], src[..., a]), \
                "a quarter turn maps (x1, x2) to (-x2, x1) for q and k"
            assert np.array_equal(got[..., rot:], src[..., rot:]), "elements past rotary_dim pass through"
        assert np.array_equal(v, p.v), "value rows are cached unchanged"


def pin_rope_interleaved_is_permuted_neox(oracle):
    # pairing (2i, 2i + 1) on x equals pairing (i, i + rot/2) on x with those dims moved together
    rng = np.random.default_rng(25)
    D, rot = 64, 48
    p = RopeProblem(rng, D=D, rot=rot, dtype="fp16")
    perm = np.concatenate([np.arange(0, rot, 2), np.arange(1, rot, 2), np.arange(rot, D)])
    qi, ki, _ = p.run(oracle, is_neox=False)
    pp = RopeProblem(rng, D=D, rot=rot, dtype="fp16", table=p.table, positions=p.pos)
    pp.q, pp.k, pp.v, pp.slots = p.q[..., perm].copy(), p.k[..., perm].copy(), p.v.copy(), p.slots
    qn, kn, _ = pp.run(oracle, is_neox=True)
    inv = np.argsort(perm)
    assert np.array_equal(qi, qn[..., inv]) and np.array_equal(ki, kn[..., inv]), \
        "interleaved pairing must be the neox pairing under the index permutation"


def pin_rope_relative_positions(oracle):
    # RoPE's defining property: after rotation, q(p) . k(p') depends only on p - p'
    rng = np.random.default_rng(26)
    D = rot = 64
    q0 = rng.standard_normal((1, 1, D)).astype(np.float32)
    k0 = rng.standard_normal((1, 1, D)).astype(np.float32)
    table = rope_cos_sin_cache(200, rot)
    dots = []
    for shift in (0, 17, 90):
        pq = RopeProblem(rng, T=1, H=1, Hkv=1, D=D, rot=rot, table=table, positions=[30 + shift], dtype="fp16")
        pq.q = f32_to_bits(q0, "fp16")
        pq.k = f32_to_bits(k0, "fp16")
        pq.slots = np.array([0], dtype=np.int64)
        q_rot, _, _ = pq.run(oracle)
        pk = RopeProblem(rng, T=1, H=1, Hkv=1, D=D, rot=rot, table=table, positions=[12 + shift], dtype="fp16")
        pk.q = f32_to_bits(q0, "fp16")
        pk.k = f32_to_bits(k0, "fp16")
        pk.slots = np.array([0], dtype=np.int64)
        _, k_rot, _ = pk.run(oracle)
        dots.append(float(np.dot(bits_to_f32(q_rot, "fp16").ravel().astype(np.float64),
                                 bits_to_f32(k_rot, "fp16").ravel().astype(np.float64))))
    scale = float(np.linalg.norm(q0) * np.linalg.norm(k0))
    assert max(dots) - min(dots) <= 4e-3 * scale, f"q.k must depend on the position gap only: {dots}"


PINS = [
    pin_dense_vs_sdpa,
    pin_sampled_equals_full,
    pin_dense_vs_sdpa_fp16,
    pin_seq_len_one_is_v_row_fp16,
    pin_fp16_decoding_matches_ieee,
    pin_bf16_decoding_special_values,
    pin_block_permutation_invariance,
    pin_seq_len_one_is_v_row,
    pin_constant_v,
    pin_zero_q_mean,
    pin_two_keys_logistic,
    pin_weights_sum_to_one,
    pin_causal_future_perturbation,
    pin_gqa_equals_replicated_mha,
    pin_slot_formula_golden,
    pin_reshape_matches_numpy_scatter,
    pin_copy_blocks_matches_numpy,
    pin_round_fp16_matches_numpy,
    pin_round_bf16_definition_cases,
    pin_rope_position_zero_is_identity,
    pin_rope_quarter_turn,
    pin_rope_interleaved_is_permuted_neox,
    pin_rope_relative_positions,
]


# --------------------------------------------------------------------------
# 8-bit (E4M3) cache codes
# --------------------------------------------------------------------------

def _torch_e4m3_codes(x32: np.ndarray) -> np.ndarray:
    """PyTorch's float32 -> float8_e4m3fn cast (round to nearest even inside the finite range)."""
    return torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32)).to(torch.float8_e4m3fn).view(
        torch.uint8).numpy()


def _torch_e4m3_values(codes: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn).to(
        torch.float64).numpy()


def pin_fp8_decode_matches_torch(oracle):
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.fp8_decode(codes)
    ref = _torch_e4m3_values(codes)
    nan = np.isnan(ref)
    assert list(np.flatnonzero(nan)) == [0x7F, 0xFF], "E4M3 has exactly two NaN codes"
    assert np.array_equal(np.isnan(got), nan), "E4M3 NaN codes"
    assert np.array_equal(got[~nan], ref[~nan]), "E4M3 decoding must match PyTorch's float8_e4m3fn"
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan])), "E4M3 signs (incl. -0)"
    # values the format fixes: 1.0, the largest finite, the smallest subnormal and normal
    assert got[0x38] == 1.0 and got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x08] == 2.0 ** -6


def pin_fp8_round_matches_torch(oracle):
    rng = np.random.default_rng(41)
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = _torch_e4m3_values(finite)
    pos = np.unique(vals[vals >= 0])
    mids = (pos[:-1] + pos[1:]) / 2.0  # exact ties, ties to the even code
    mag = np.exp2(rng.uniform(-12.0, np.log2(448.0), size=20000))
    x = np.concatenate([vals, mids, -mids, mids * (1 + 2.0 ** -20), mids * (1 - 2.0 ** -20),
                        mag * rng.choice([-1.0, 1.0], size=mag.size)]).astype(np.float32)
    got = oracle.fp8_round(x.astype(np.float64))
    ref = _torch_e4m3_codes(x)
    bad = np.flatnonzero(got != ref)
    assert bad.size == 0, f"E4M3 rounding differs from PyTorch at {x[bad[:5]]}: {got[bad[:5]]} vs {ref[bad[:5]]}"
    assert np.array_equal(oracle.fp8_round(vals), finite), "every finite code must round-trip"


def pin_fp8_round_saturates_and_specials(oracle):
    cases = [(448.0, 0x7E), (449.0, 0x7E), (464.0, 0x7E), (480.0, 0x7E), (1e6, 0x7E), (math.inf, 0x7E),
             (-448.0, 0xFE), (-1e30, 0xFE), (-math.inf, 0xFE), (0.0, 0x00), (-0.0, 0x80),
             (2.0 ** -10, 0x00),        # half the smallest subnormal: tie to the even code 0
             (3 * 2.0 ** -10, 0x02),    # 1.5 quanta: tie to 2 quanta
             (5 * 2.0 ** -10, 0x02),    # 2.5 quanta: tie to 2 quanta
             (1.0625, 0x38),            # between 1 and 1.125: tie to 1.0 (even fraction 0)
             (1.1875, 0x3A),            # between 1.125 and 1.25: tie to 1.25 (fraction 2)
             (440.0, 0x7E),             # between 416 and 448: tie to 448 (fraction 6)
             (math.nan, 0x7F)]
    x = np.array([c[0] for c in cases], dtype=np.float64)
    got = oracle.fp8_round(x)
    want = np.array([c[1] for c in cases], dtype=np.uint8)
    assert np.array_equal(got, want), f"E4M3 special cases: {list(zip(x, got, want))}"


def pin_fp8_quantize_is_float32_quotient(oracle):
    rng = np.random.default_rng(42)
    for dtype in ("bf16", "fp16"):
        bits = f32_to_bits((4.0 * rng.standard_normal(50000)).astype(np.float32), dtype)
        for scale in (0.0371, 0.0625, 1.7):
            s32 = np.float32(scale)
            q = bits_to_f32(bits, dtype) / s32  # numpy binary32 division
            keep = np.abs(q) < 448.0
            got = oracle.fp8_quantize(bits, float(s32), dtype)
            ref = _torch_e4m3_codes(q)
            assert np.array_equal(got[keep], ref[keep]), f"quantiser vs float32 quotient + cast ({dtype}, {scale})"
            big = ~keep
            assert np.all((got[big] & 0x7F) == 0x7E), "quotients beyond 448 saturate"


def pin_fp8_reshape_matches_numpy_scatter(oracle):
    rng = np.random.default_rng(43)
    nb, bs, hkv, d, T = 6, 8, 2, 16, 20
    slots = rng.permutation(nb * bs)[:T].astype(np.int64)
    slots[3] = -1
    key = f32_to_bits(rng.standard_normal((T, hkv, d)).astype(np.float32), "bf16")
    value = f32_to_bits(rng.standard_normal((T, hkv, d)).astype(np.float32), "bf16")
    ks, vs = np.float32(0.05), np.float32(0.03)
    kc = np.full((nb, bs, hkv, d), 0x7F, dtype=np.uint8)
    vc = kc.copy()
    oracle.reshape_and_cache_fp8(key, value, kc, vc, slots, bs, float(ks), float(vs), "bf16")
    kref = np.full_like(kc, 0x7F).reshape(nb * bs, hkv, d)
    vref = kref.copy()
    ok = slots >= 0
    kref[slots[ok]] = _torch_e4m3_codes(bf16_bits_to_f32(key[ok]) / ks)
    vref[slots[ok]] = _torch_e4m3_codes(bf16_bits_to_f32(value[ok]) / vs)
    assert np.array_equal(kc.reshape(nb * bs, hkv, d), kref), "8-bit K scatter"
    assert np.array_equal(vc.reshape(nb * bs, hkv, d), vref), "8-bit V scatter"


def pin_fp8_attention_vs_sdpa(oracle):
    """Attention over 8-bit caches: dense float64 SDPA over the decoded values times the scales."""
    from paged_kv_cache_55_gb300.workloads import fp8_codes
    rng = np.random.default_rng(44)
    ks, vs = float(np.float32(0.0625 * 1.1)), float(np.float32(0.0437))
    for ctx, ql, H, Hkv, D, bs in DENSE_CASES:
        p = DenseProblem(rng, ctx, ql, H, Hkv, D, bs)
        p.kd = [fp8_codes(rng, (x, Hkv, D)) for x in p.L]
        p.vd = [fp8_codes(rng, (x, Hkv, D)) for x in p.L]
        bt = np.full((len(p.L), p.max_blocks), -7, dtype=np.int32)
        kc = np.full((p.num_blocks, bs, Hkv, D), 0x7F, dtype=np.uint8)
        vc = kc.copy()
        cursor = 0
        for b, L in enumerate(p.L):
            for i in range((L + bs - 1) // bs):
                bt[b, i] = p.perm[cursor]
                cursor += 1
            for j in range(L):
                kc[bt[b, j // bs], j % bs] = p.kd[b][j]
                vc[bt[b, j // bs], j % bs] = p.vd[b][j]
        got = oracle.attention(p.q, kc, vc, bt, p.seq_lens, p.qsl, H, p.scale, num_threads=2,
                               k_scale=ks, v_scale=vs)
        ref = np.zeros_like(got)
        for b, L in enumerate(p.L):
            q0, n = int(p.qsl[b]), p.ql[b]
            if n == 0:
                continue
            qb = torch.from_numpy(bf16_bits_to_f32(p.q[q0:q0 + n]).astype(np.float64)).transpose(0, 1)
            kb = torch.from_numpy(_torch_e4m3_values(p.kd[b]) * ks).transpose(0, 1)
            vb = torch.from_numpy(_torch_e4m3_values(p.vd[b]) * vs).transpose(0, 1)
            mask = torch.arange(L).unsqueeze(0) <= (L - n) + torch.arange(n).unsqueeze(1)
            o = torch.nn.functional.scaled_dot_product_attention(
                qb.unsqueeze(0), kb.unsqueeze(0), vb.unsqueeze(0), attn_mask=mask, scale=p.scale,
                enable_gqa=(H != Hkv))
            ref[q0:q0 + n] = o[0].transpose(0, 1).numpy()
        err = float(np.max(np.abs(got - ref))) if got.size else 0.0
        assert err <= 1e-12, f"8-bit cache attention vs SDPA max |diff| {err} for {(ctx, ql, H, Hkv, D, bs)}"


def pin_rope_fp8_identity_and_quarter_turn(oracle):
    """The rotary scatter into 8-bit caches: at position 0 the codes are PyTorch's cast of
    k / k_scale and v / v_scale; with a row (cos 0, sin 1) K's rotated pairs become
    (-x2, x1) exactly, so their codes are the cast of those over k_scale."""
    rng = np.random.default_rng(45)
    ks, vs = np.float32(0.07), np.float32(0.05)
    D, rot, half = 32, 16, 8
    quarter = np.zeros((2, rot), dtype=np.float32)
    quarter[0, :half] = 1.0
    quarter[1, half:] = 1.0
    for dtype in ("bf16", "fp16"):
        for table, pos in ((rope_cos_sin_cache(64, rot), [0] * 6), (quarter, [1] * 6)):
            p = RopeProblem(rng, D=D, rot=rot, dtype=dtype, table=table, positions=pos)
            q = p.q.copy()
            kc = np.full((p.nb, p.bs, p.k.shape[1], D), 0x7F, dtype=np.uint8)
            vc = kc.copy()
            oracle.rope_reshape_and_cache_fp8(q, p.k, p.v, kc, vc, p.slots, p.pos, p.table, True, p.bs,
                                              float(ks), float(vs), dtype)
            kx = bits_to_f32(p.k, dtype)
            if pos[0] == 1:  # neox pairs (i, i + half), i < half: (x1, x2) -> (-x2, x1)
                kr = kx.copy()
                kr[..., :half] = -kx[..., half:rot]
                kr[..., half:rot] = kx[..., :half]
                kx = kr
            want_k = _torch_e4m3_codes(kx / ks)
            want_v = _torch_e4m3_codes(bits_to_f32(p.v, dtype) / vs)
            got_k = kc.reshape(-1, p.k.shape[1], D)[p.slots]
            got_v = vc.reshape(-1, p.k.shape[1], D)[p.slots]
            assert np.array_equal(got_k, want_k), f"8-bit rotary K codes ({dtype}, position {pos[0]})"
            assert np.array_equal(got_v, want_v), f"8-bit rotary V codes ({dtype})"


PINS += [
    pin_rope_fp8_identity_and_quarter_turn,
    pin_fp8_decode_matches_torch,
    pin_fp8_round_matches_torch,
    pin_fp8_round_saturates_and_specials,
    pin_fp8_quantize_is_float32_quotient,
    pin_fp8_reshape_matches_numpy_scatter,
    pin_fp8_attention_vs_sdpa,
]
