"""Rotary embedding fused with the cache scatter, against the oracle (needs a GB300).

The kernel rotates in fp32 and the oracle in fp64, each rounding once to the
element type, so rotated q and K elements may differ by one unit in the last
place; V rows and every untouched element must match bit for bit. A whole step
(rotary scatter, then attention) must meet the attention tolerance.
"""

import numpy as np
import pytest
import torch

from paged_kv_cache_55_gb300 import binding as B
from paged_kv_cache_55_gb300 import workloads as W
from paged_kv_cache_55_gb300.runner import DeviceStep, bf16_tensor, bf16_to_float64, bf16_to_numpy_bits

from test_gpu_parity import assert_attention_close

pytestmark = pytest.mark.gpu


def positions_of(w):
    """Token i of request b sits at position context_b + i."""
    pos = np.empty(w.total_q, dtype=np.int64)
    qsl = np.asarray(w.query_start_loc)
    for b in range(w.num_seqs):
        ctx = int(w.seq_lens[b]) - int(qsl[b + 1] - qsl[b])
        pos[qsl[b]:qsl[b + 1]] = ctx + np.arange(qsl[b + 1] - qsl[b])
    return pos


def within_one_ulp(g: np.ndarray, o: np.ndarray) -> np.ndarray:
    """Element-wise: equal bits, or neighbours of the same sign (one unit in the last place)."""
    gi, oi = g.astype(np.int64), o.astype(np.int64)
    same_sign = (gi >> 15) == (oi >> 15)
    return (gi == oi) | (same_sign & (np.abs((gi & 0x7FFF) - (oi & 0x7FFF)) <= 1))


def rope_case(w, rot, neox, oracle):
    table = W.rope_cos_sin_cache(int(w.max_seq_len) + 8, rot)
    pos = positions_of(w)
    st = DeviceStep(w)
    B.pa_rope_reshape_and_cache(st.q, st.key, st.value, st.key_cache, st.value_cache, st.slot_mapping,
                                torch.from_numpy(pos).cuda(), torch.from_numpy(table).cuda(), is_neox=neox)
    torch.cuda.synchronize()
    assert B.pa_debug_status() == 0
    q = w.q.copy()
    kc, vc = w.key_cache.copy(), w.value_cache.copy()
    oracle.rope_reshape_and_cache(q, w.key, w.value, kc, vc, w.slot_mapping, pos, table, neox, w.block_size, w.dtype)
    return st, q, kc, vc, table, pos


CASES = [(128, 128, 8, 2), (128, 64, 32, 8), (64, 32, 16, 2)]  # (D, rotary_dim, H, Hkv)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("neox", [True, False])
@pytest.mark.parametrize("case", CASES)
def test_rope_reshape_matches_oracle(oracle, dtype, neox, case):
    D, rot, H, Hkv = case
    w = W.make_workload("rope", context_lens=[0, 37, 500, 3], query_lens=[40, 1, 9, 1], num_heads=H,
                        num_kv_heads=Hkv, head_dim=D, seed=12, dtype=dtype)
    st, q, kc, vc, _, _ = rope_case(w, rot, neox, oracle)
    gq = bf16_to_numpy_bits(st.q)
    gk = bf16_to_numpy_bits(st.key_cache)
    gv = bf16_to_numpy_bits(st.value_cache)
    assert np.array_equal(gv, vc), "value rows are copied bit for bit"
    assert np.array_equal(gq[..., rot:], q[..., rot:]), "q elements past rotary_dim pass through"
    ok_q, ok_k = within_one_ulp(gq, q), within_one_ulp(gk, kc)
    assert ok_q.all() and ok_k.all(), f"{int((~ok_q).sum())} q and {int((~ok_k).sum())} K elements off by > 1 ulp"
    assert (gq == q).mean() > 0.99 and (gk == kc).mean() > 0.99  # a one-ulp difference is the exception


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_rope_then_attention_matches_oracle(oracle, dtype):
    w = W.make_workload("rope_step", context_lens=[0, 37, 600, 20, 1000], query_lens=[40, 2, 1, 129, 1],
                        num_heads=32, num_kv_heads=8, head_dim=128, seed=13, dtype=dtype)
    st, q, kc, vc, _, _ = rope_case(w, 128, True, oracle)
    st.attention()
    torch.cuda.synchronize()
    assert B.pa_debug_status() == 0
    ref = oracle.attention(q, kc, vc, w.block_tables, w.seq_lens, w.query_start_loc, w.num_heads, w.scale,
                           dtype=w.dtype)
    gpu = bf16_to_float64(st.out)
    assert np.isfinite(gpu).all()
    assert_attention_close(gpu, ref, f"rope step {dtype}")


def test_rope_q_with_token_stride_and_bad_position(oracle):
    """q as a slice of a fused QKV buffer; a token whose position is past the table is
    skipped (q row untouched, nothing cached) and flagged."""
    H, Hkv, D = 8, 2, 128
    w = W.make_workload("rope_stride", context_lens=[10, 3], query_lens=[5, 2], num_heads=H, num_kv_heads=Hkv,
                        head_dim=D, seed=14)
    table = W.rope_cos_sin_cache(16, 128)
    pos = positions_of(w)
    bad = 3
    pos[bad] = 16  # one past the table
    st = DeviceStep(w)
    fused = torch.zeros((w.total_q, H + 2 * Hkv, D), dtype=torch.bfloat16, device="cuda")
    fused[:, :H] = st.q
    qv = fused[:, :H]
    B.pa_rope_reshape_and_cache(qv, st.key, st.value, st.key_cache, st.value_cache, st.slot_mapping,
                                torch.from_numpy(pos).cuda(), torch.from_numpy(table).cuda(), is_neox=True)
    torch.cuda.synchronize()
    assert B.pa_debug_status() == B.FLAG_POSITION_RANGE
    gq = bf16_to_numpy_bits(qv.contiguous())
    assert np.array_equal(gq[bad], w.q[bad]), "the flagged token's q is left as it was"
    gk = bf16_to_numpy_bits(st.key_cache).reshape(-1, Hkv, D)
    assert np.array_equal(gk[w.slot_mapping[bad]], w.key_cache.reshape(-1, Hkv, D)[w.slot_mapping[bad]])
    keep = np.arange(w.total_q) != bad
    q = w.q[keep].copy()
    kc, vc = w.key_cache.copy(), w.value_cache.copy()
    oracle.rope_reshape_and_cache(q, w.key[keep], w.value[keep], kc, vc, w.slot_mapping[keep], pos[keep], table,
                                  True, w.block_size)
    assert within_one_ulp(gq[keep], q).all() and within_one_ulp(gk.reshape(kc.shape), kc).all()
    assert np.array_equal(bf16_to_numpy_bits(fused[:, H:]), np.zeros((w.total_q, 2 * Hkv, D), np.uint16)), \
        "the rest of the fused buffer is not touched"


def within_one_code(g: np.ndarray, o: np.ndarray) -> np.ndarray:
    """E4M3 codes: equal, or neighbours of the same sign (the rotated element they quantise may
    differ by one unit in the last place between the fp32 kernel and the fp64 oracle)."""
    gi, oi = g.astype(np.int64), o.astype(np.int64)
    return (gi == oi) | (((gi >> 7) == (oi >> 7)) & (np.abs((gi & 0x7F) - (oi & 0x7F)) <= 1))


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("neox", [True, False])
@pytest.mark.parametrize("case", CASES)
def test_rope_fp8_matches_oracle(oracle, dtype, neox, case):
    D, rot, H, Hkv = case
    w = W.make_workload("rope_fp8", context_lens=[0, 30, 900, 5], query_lens=[40, 1, 3, 17], num_heads=H,
                        num_kv_heads=Hkv, head_dim=D, seed=5, dtype=dtype, kv_dtype=W.FP8_E4M3)
    table = W.rope_cos_sin_cache(int(w.max_seq_len) + 8, rot)
    pos = positions_of(w)
    st = DeviceStep(w)
    B.pa_rope_reshape_and_cache_fp8(st.q, st.key, st.value, st.key_cache, st.value_cache, st.slot_mapping,
                                    torch.from_numpy(pos).cuda(), torch.from_numpy(table).cuda(), w.k_scale,
                                    w.v_scale, is_neox=neox)
    torch.cuda.synchronize()
    assert B.pa_debug_status() == 0
    q = w.q.copy()
    kc, vc = w.key_cache.copy(), w.value_cache.copy()
    oracle.rope_reshape_and_cache_fp8(q, w.key, w.value, kc, vc, w.slot_mapping, pos, table, neox, w.block_size,
                                      w.k_scale, w.v_scale, w.dtype)
    assert within_one_ulp(bf16_to_numpy_bits(st.q), q).all(), "rotated q"
    assert np.array_equal(st.value_cache.cpu().numpy(), vc), "V codes must match bit for bit"
    gk = st.key_cache.cpu().numpy()
    assert within_one_code(gk, kc).all(), "rotated K codes within one step"
    rows = w.slot_mapping
    gk_rows = gk.reshape(-1, Hkv, D)[rows]
    ok_rows = kc.reshape(-1, Hkv, D)[rows]
    assert np.array_equal(gk_rows[..., rot:], ok_rows[..., rot:]), "K past rotary_dim must match bit for bit"
    assert (gk_rows == ok_rows).mean() > 0.99
    # everything outside the written slots is untouched
    untouched = np.ones(gk.reshape(-1, Hkv, D).shape[0], dtype=bool)
    untouched[rows] = False
    assert np.array_equal(gk.reshape(-1, Hkv, D)[untouched], w.key_cache.reshape(-1, Hkv, D)[untouched])


def test_rope_fp8_step_matches_oracle(oracle):
    """A whole step over 8-bit caches: rotary scatter, then attention, against the oracle's."""
    w = W.make_workload("rope_fp8_step", context_lens=[0, 37, 600, 20, 1000], query_lens=[40, 2, 1, 129, 1],
                        num_heads=32, num_kv_heads=8, head_dim=128, seed=6, kv_dtype=W.FP8_E4M3)
    table = W.rope_cos_sin_cache(int(w.max_seq_len) + 8, 128)
    pos = positions_of(w)
    st = DeviceStep(w, rope=(table, pos, True))
    st.run()
    torch.cuda.synchronize()
    assert B.pa_debug_status() == 0
    q = w.q.copy()
    kc, vc = w.key_cache.copy(), w.value_cache.copy()
    oracle.rope_reshape_and_cache_fp8(q, w.key, w.value, kc, vc, w.slot_mapping, pos, table, True, w.block_size,
                                      w.k_scale, w.v_scale, w.dtype)
    # attention on the GPU's own caches and rotated q (isolates the attention step from 1-ulp rotations)
    gq = bf16_to_numpy_bits(st.q)
    gk, gv = st.key_cache.cpu().numpy(), st.value_cache.cpu().numpy()
    ref = oracle.attention(gq, gk, gv, w.block_tables, w.seq_lens, w.query_start_loc, w.num_heads, w.scale,
                           dtype=w.dtype, k_scale=w.k_scale, v_scale=w.v_scale)
    assert_attention_close(bf16_to_float64(st.out), ref, w.name)
    assert within_one_code(gk, kc).all() and np.array_equal(gv, vc)
