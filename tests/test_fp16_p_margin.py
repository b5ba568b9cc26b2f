"""Margin of one fp16 P per key, the tensor-core tiles' rounding of the
probabilities, against the attention tolerance (CPU only).

The tile kernel stores each probability as one fp16 value (11 significant
bits) for the P V products: for fp16 elements, for 8-bit caches (widened to
fp16), and for bf16 caches, whose V it rewrites as fp16 (exactly, for values
of magnitude 2^-17 up to 65535). This test models that rounding alone: P
computed in fp64 against the row maximum, rounded to fp16, the products and
the normalising sum in fp64. It compares the model with the fp64 oracle on
chunked-prefill shapes (every query row of requests that take the tiles)
and requires the error to stay within half of the tolerance the GPU tests
apply, |err| <= 2e-3 + 1e-2 |ref|. The kernel's lazy rescale takes P against
a maximum up to 2^8 below the running one, which moves P within fp16's
normal range and leaves its relative rounding unchanged.
"""

import numpy as np
import pytest

from paged_kv_cache_55_gb300 import workloads as W

import oracle

ATOL, RTOL = 2e-3, 1e-2

CASES = {
    "chunks_g4_d128": dict(context_lens=[0, 300, 77], query_lens=[130, 200, 1], num_heads=16, num_kv_heads=4,
                           head_dim=128),
    "chunks_g1_d64_sharp": dict(context_lens=[40, 0], query_lens=[100, 64], num_heads=4, num_kv_heads=4,
                                head_dim=64, q_scale=3.0),
    "chunks_g8_d96_bs8": dict(context_lens=[500], query_lens=[48], num_heads=16, num_kv_heads=2, head_dim=96,
                              block_size=8),
}


def p16_model(orc, w, kc, vc):
    """Attention of the tile kernel's requests with P rounded to fp16; rows of other requests are NaN."""
    q = orc.decode_elements(w.q, w.dtype)
    if w.kv_fp8:
        K = orc.fp8_decode(kc) * np.float64(np.float32(w.k_scale))
        V = orc.fp8_decode(vc) * np.float64(np.float32(w.v_scale))
    else:
        K = orc.decode_elements(kc, w.dtype)
        V = orc.decode_elements(vc, w.dtype)
    bs, G = w.block_size, w.num_heads // w.num_kv_heads
    out = np.full((w.total_q, w.num_heads, w.head_dim), np.nan)
    scale = np.float64(np.float32(w.scale))
    for b in range(w.num_seqs):
        q0, q1 = int(w.query_start_loc[b]), int(w.query_start_loc[b + 1])
        ql, L = q1 - q0, int(w.seq_lens[b])
        if ql * G <= 8:  # decode items: the split-KV kernel, not the tiles
            continue
        j = np.arange(L)
        phys = w.block_tables[b, j // bs]
        Kb, Vb = K[phys, j % bs], V[phys, j % bs]
        visible = j[None, :] <= (L - ql + np.arange(ql))[:, None]
        for h in range(w.num_heads):
            kvh = h // G
            s = (q[q0:q1, h] @ Kb[:, kvh].T) * scale
            s = np.where(visible, s, -np.inf)
            p = np.exp(s - s.max(axis=1, keepdims=True))
            p16 = p.astype(np.float16).astype(np.float64)
            out[q0:q1, h] = (p16 @ Vb[:, kvh]) / p.sum(axis=1, keepdims=True)
    return out


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("dtype,kv_dtype", [("bf16", ""), ("fp16", ""), ("bf16", W.FP8_E4M3),
                                            ("fp16", W.FP8_E4M3)])
def test_fp16_p_uses_at_most_half_the_tolerance(name, dtype, kv_dtype):
    orc = oracle.default()
    w = W.make_workload(name, seed=7, dtype=dtype, kv_dtype=kv_dtype, **CASES[name])
    kc, vc, ref = orc.run_step(w)
    model = p16_model(orc, w, kc, vc)
    rows = ~np.isnan(model[:, 0, 0])
    assert rows.any()
    err = np.abs(model[rows] - ref[rows])
    ratio = err / (ATOL + RTOL * np.abs(ref[rows]))
    assert ratio.max() <= 0.5, f"fp16 P alone reaches {ratio.max():.3f} of the tolerance"
    # and the rounding is visible at all (the model is not the oracle in disguise)
    assert err.max() > 0.0
