"""The bench's algorithmic bytes and FLOPs (the numerators of its roofline
fractions) against a brute-force count over every (query, key) pair and every
cache slot a step reads, on small workloads with a shared prefix, prefill
chunks and decode tokens (CPU only)."""

import os
import sys

import pytest

from paged_kv_cache_55_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
import bench  # noqa: E402


def brute_force(w, rope=False):
    """Walk every request's keys and queries one by one."""
    H, Hkv, D, bs = w.num_heads, w.num_kv_heads, w.head_dim, w.block_size
    elem = 1 if w.kv_fp8 else 2
    slots = set()      # physical (block, row) slots read by the step
    pairs = 0          # visible (query, key) pairs
    tile_pairs = 0     # of requests longer than one decode item (the tensor-core tiles)
    rows_per_item = 8 // (H // Hkv)
    for b in range(w.num_seqs):
        L = int(w.seq_lens[b])
        n = int(w.query_start_loc[b + 1] - w.query_start_loc[b])
        for j in range(L):
            slots.add((int(w.block_tables[b, j // bs]), j % bs))
        ctx = L - n
        for i in range(n):
            vis = ctx + i + 1  # keys 0 .. ctx + i
            pairs += vis
            if n > rows_per_item:
                tile_pairs += vis
    T = int(w.query_start_loc[-1])
    kv = len(slots) * 2 * Hkv * D * elem
    tables = sum(-(-int(L) // bs) for L in w.seq_lens) * 4
    meta = (2 * w.num_seqs + 1) * 4
    q_out = 2 * T * H * D * 2
    scatter = T * 2 * Hkv * D * 2 + T * 2 * Hkv * D * elem + T * 8
    if rope:
        scatter += 2 * T * H * D * 2 + T * 8 + T * D * 4
    return {
        "kv_bytes": kv,
        "attention_bytes": kv + q_out + tables + meta,
        "step_bytes": kv + q_out + tables + meta + scatter,
        "scatter_bytes": scatter,
        "flops": 4 * H * D * pairs,
        "tile_flops": 4 * H * D * tile_pairs,
        "query_tokens": T,
    }


CASES = {
    "mixed_shared": dict(context_lens=[64, 64, 300, 0, 17, 128], query_lens=[1, 1, 40, 33, 1, 9],
                         num_heads=8, num_kv_heads=2, head_dim=64, shared_prefix_requests=[0, 1],
                         shared_prefix_blocks=4),
    "decode_g8": dict(context_lens=[5, 99, 1000, 16], query_lens=[1, 1, 1, 1], num_heads=16, num_kv_heads=2,
                      head_dim=128, block_size=8),
    "chunks_g1": dict(context_lens=[0, 200, 31], query_lens=[50, 7, 12], num_heads=4, num_kv_heads=4, head_dim=80,
                      block_size=32),
}


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("kv_dtype", ["", "fp8_e4m3"])
@pytest.mark.parametrize("rope", [False, True])
def test_step_accounting_matches_brute_force(name, kv_dtype, rope):
    w = W.make_workload(name, seed=3, kv_dtype=kv_dtype, **CASES[name])
    got = bench.step_accounting(w, rope=rope)
    want = brute_force(w, rope=rope)
    for k, v in want.items():
        assert got[k] == v, (k, got[k], v)


def test_shared_prefix_is_counted_once():
    kw = CASES["mixed_shared"]
    w = W.make_workload("mixed_shared", seed=3, **kw)
    acct = bench.step_accounting(w)
    assert acct["kv_bytes"] < acct["kv_bytes_logical"]
    # the two sharing requests read 4 blocks of 16 rows each once between them
    saved = (acct["kv_bytes_logical"] - acct["kv_bytes"]) // (2 * w.num_kv_heads * w.head_dim * 2)
    assert saved == 4 * 16
