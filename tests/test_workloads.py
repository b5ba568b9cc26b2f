"""Host logic of the seeded input generator (no GPU)."""

import numpy as np
import pytest

from oracle_pins import read_golden
from paged_kv_cache_55_gb300 import workloads as W


def test_page_count_matches_diagram():
    for tokens, page, pages in read_golden("page_alloc_diagram.txt"):
        assert W.blocks_needed(int(tokens), int(page)) == pages
    assert W.blocks_needed(0, 16) == 0
    assert W.blocks_needed(1, 16) == 1
    assert W.blocks_needed(16, 16) == 1
    assert W.blocks_needed(17, 16) == 2


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-8, -2.5, 65504.0, 1e-30], dtype=np.float32)
    h = W.f32_to_bf16_bits(x)
    back = W.bf16_bits_to_f32(h)
    assert back[0] == 1.0
    assert back[1] == 1.0                    # tie rounds to even (down)
    assert back[2] == 1.0 + 4 * 2**-8        # tie rounds to even (up)
    assert back[3] == -2.5
    import torch
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(h, ref)


def _check_consistent(w: W.Workload):
    B = w.num_seqs
    ql = w.query_lens
    assert w.query_start_loc[0] == 0 and (ql >= 0).all()
    assert (w.seq_lens >= ql).all()
    assert w.q.shape == (w.total_q, w.num_heads, w.head_dim)
    assert w.key.shape == (w.total_q, w.num_kv_heads, w.head_dim)
    s = w.slot_mapping[w.slot_mapping >= 0]
    assert np.unique(s).size == s.size, "slots must be unique"
    assert (s < w.num_blocks * w.block_size).all()
    for b in range(B):
        nb = W.blocks_needed(int(w.seq_lens[b]), w.block_size)
        ids = w.block_tables[b, :nb]
        assert ((ids >= 0) & (ids < w.num_blocks)).all()


@pytest.mark.parametrize("name,kw", [("tiny_decode", {}), ("mha_decode", {"batch": 4}),
                                     ("gqa_decode", {"batch": 6}),
                                     ("long_decode", {"batch": 2, "seq_len": 300})])
def test_named_small_workloads(name, kw):
    a = W.by_name(name, seed=3, **kw)
    b = W.by_name(name, seed=3, **kw)
    _check_consistent(a)
    assert np.array_equal(a.q, b.q) and np.array_equal(a.key_cache, b.key_cache)
    assert np.array_equal(a.block_tables, b.block_tables)
    c = W.by_name(name, seed=4, **kw)
    assert not np.array_equal(a.q, c.q)


def test_tiny_decode_shape():
    w = W.tiny_decode()
    assert list(w.seq_lens) == [1, 7, 16, 33]
    assert w.num_blocks == 32 and w.num_heads == 4 and w.num_kv_heads == 1 and w.head_dim == 64
    assert w.scale == np.float32(1 / 8)


def test_mha_pool_has_ten_percent_slack():
    w = W.mha_decode(seed=1, batch=6)
    need = sum(W.blocks_needed(int(L), 16) for L in w.seq_lens)
    assert w.num_blocks == int(np.ceil(need * 1.1))
    assert ((w.seq_lens >= 128) & (w.seq_lens <= 2048)).all()


def test_gqa_lengths_lognormal_clipped():
    L = W.gqa_seq_lens(0, 4096)
    assert L.min() >= 16 and L.max() <= 8192
    med = np.median(L)
    assert 900 < med < 1150


def test_mixed_step_shared_prefix_is_copy_on_write_safe():
    w = W.mixed_step(seed=0, n_prefill=3, chunk=40, n_decode=12, n_shared=5, shared_blocks=4)
    _check_consistent(w)
    shared = set(int(x) for x in w.shared_blocks)
    assert len(shared) == 4
    users = [b for b in range(w.num_seqs) if set(int(x) for x in w.block_tables[b, :4]) == shared]
    assert len(users) == 5
    # no new token of this step writes into a shared block
    blocks_written = set(int(s) // w.block_size for s in w.slot_mapping)
    assert not (blocks_written & shared)
    assert w.total_q == 3 * 40 + 12


def test_unowned_slots_hold_nan_sentinel():
    w = W.tiny_decode()
    owned = np.zeros(w.num_blocks * w.block_size, dtype=bool)
    for b in range(w.num_seqs):
        for j in range(int(w.seq_lens[b]) - int(w.query_lens[b])):
            owned[int(w.block_tables[b, j // 16]) * 16 + j % 16] = True
    flat = w.key_cache.reshape(-1, w.num_kv_heads * w.head_dim)
    assert (flat[~owned] == 0x7FC0).all()
    assert not (flat[owned] == 0x7FC0).any()


def test_fp16_workload_rounds_the_same_draws():
    """dtype="fp16" rounds the very draws the bf16 workload rounds (numpy's IEEE
    binary16 conversion), keeps the structure, and fills unowned slots with the
    fp16 NaN."""
    kw = dict(context_lens=[5, 40, 0], query_lens=[1, 3, 9], num_heads=8, num_kv_heads=2, head_dim=64, seed=4)
    wb = W.make_workload("b", **kw)
    wh = W.make_workload("h", dtype="fp16", **kw)
    assert wh.dtype == "fp16" and wb.dtype == "bf16"
    for f in ("slot_mapping", "block_tables", "seq_lens", "query_start_loc"):
        assert np.array_equal(getattr(wb, f), getattr(wh, f))
    qb = W.bf16_bits_to_f32(wb.q).astype(np.float64)
    qh = wh.q.view(np.float16).astype(np.float64)
    assert np.all(np.abs(qb - qh) <= 2.0 ** -8 * np.abs(qh) + 1e-7)  # both round one float32 draw
    own = np.zeros(wh.key_cache.shape[0] * wh.block_size, dtype=bool)
    for b in range(wh.num_seqs):
        L = int(wh.seq_lens[b])
        j = np.arange(L)
        own[wh.block_tables[b, j // wh.block_size].astype(np.int64) * wh.block_size + j % wh.block_size] = True
    flat = wh.key_cache.reshape(-1, wh.num_kv_heads, wh.head_dim)
    assert (flat[~own] == 0x7E00).all() and np.isnan(flat[~own].view(np.float16)).all()
