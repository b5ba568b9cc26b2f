"""Shape checks of the Python binding (no GPU).

The C ABI takes plain pointers, so the binding is the last place where a
tensor of the wrong size can be refused before a kernel reads or writes past
its end. These tests build the device buffers of real workloads on PyTorch's
``meta`` device (shapes without storage), check that every shape the step
passes is accepted, and that each kind of mismatch is refused.
"""

import pytest
import torch

from paged_kv_cache_55_gb300 import binding as B
from paged_kv_cache_55_gb300 import build as build_mod
from paged_kv_cache_55_gb300 import workloads as W
from paged_kv_cache_55_gb300.runner import DeviceStep


@pytest.fixture(scope="module", autouse=True)
def _library():
    build_mod.build()  # DeviceStep sizes its workspace through the library (host arithmetic only)


def meta(*shape, dtype=torch.bfloat16):
    return torch.empty(shape, dtype=dtype, device="meta")


def meta_step(w, rope=None):
    return DeviceStep(w, device="meta", rope=rope)


WORKLOADS = [
    lambda: W.tiny_decode(seed=0),
    lambda: W.make_workload("mixed", context_lens=[0, 7, 300, 33], query_lens=[40, 1, 1, 9], num_heads=32,
                            num_kv_heads=8, head_dim=128, seed=2),
    lambda: W.make_workload("fp8", context_lens=[200, 35], query_lens=[1, 12], num_heads=8, num_kv_heads=2,
                            head_dim=96, block_size=32, kv_dtype=W.FP8_E4M3, seed=4),
    lambda: W.make_workload("fp16_bs8", context_lens=[17, 0], query_lens=[1, 5], num_heads=4, num_kv_heads=4,
                            head_dim=64, block_size=8, dtype="fp16", seed=5),
]


@pytest.mark.parametrize("make", WORKLOADS, ids=["tiny", "mixed", "fp8_d96_bs32", "fp16_bs8"])
def test_shapes_of_a_step_are_accepted(make):
    w = make()
    st = meta_step(w)
    B._scatter_shapes(st.key, st.value, st.key_cache, st.value_cache, st.slot_mapping)
    B._attention_shapes(st.q, st.key_cache, st.value_cache, st.block_tables, st.seq_lens, st.query_start_loc,
                        st.out)
    B._cache_pair_shapes(st.key_cache, st.value_cache)
    # the gather of each request into [seq_len, Hkv, D] buffers
    for b in range(w.num_seqs):
        L = int(w.seq_lens[b])
        out = meta(L, w.num_kv_heads, w.head_dim, dtype=st.key_cache.dtype)
        B._gather_shapes(st.key_cache, st.value_cache, st.block_tables[b], L, out, out)
    # the rotary scatter, also with q a [T, H, D] view of a wider fused row
    table = meta(int(w.max_seq_len) + 8, 64, dtype=torch.float32)
    positions = meta(w.total_q, dtype=torch.int64)
    B._rope_shapes(st.q, st.key, st.value, st.key_cache, st.value_cache, st.slot_mapping, positions, table)
    fused = meta(w.total_q, w.num_heads + 2 * w.num_kv_heads, w.head_dim)
    B._rope_shapes(fused[:, :w.num_heads], st.key, st.value, st.key_cache, st.value_cache, st.slot_mapping,
                   positions, table)


def test_empty_step_is_accepted():
    k = meta(0, 2, 64)
    cache = meta(4, 16, 2, 64)
    B._scatter_shapes(k, k, cache, cache, meta(0, dtype=torch.int64))
    B._attention_shapes(meta(0, 8, 64), cache, cache, meta(0, 3, dtype=torch.int32), meta(0, dtype=torch.int32),
                        meta(1, dtype=torch.int32), meta(0, 8, 64))


def test_mismatched_shapes_are_refused():
    w = W.tiny_decode(seed=0)
    st = meta_step(w)
    T, H, D = st.q.shape
    Bn = w.num_seqs
    att = dict(q=st.q, key_cache=st.key_cache, value_cache=st.value_cache, block_tables=st.block_tables,
               seq_lens=st.seq_lens, query_start_loc=st.query_start_loc, out=st.out)
    bad_attention = [
        ("out", meta(T - 1, H, D)),                                   # one token short
        ("out", meta(T, H, D // 2)),                                  # half a row
        ("value_cache", meta(*st.key_cache.shape[:-1], D // 2)),      # caches differ
        ("key_cache", meta(w.num_blocks, w.block_size, 1, D)[..., None]),  # five dimensions
        ("query_start_loc", meta(Bn, dtype=torch.int32)),             # B entries instead of B + 1
        ("block_tables", meta(Bn + 1, 4, dtype=torch.int32)),         # one row too many
        ("q", meta(T, H * D)),                                        # flattened rows
    ]
    for name, t in bad_attention:
        kw = dict(att, **{name: t})
        if name == "key_cache":
            kw["value_cache"] = t
        with pytest.raises(ValueError):
            B._attention_shapes(**kw)
    # head_dim of q and of the caches differ (caches consistent with each other)
    other = meta(w.num_blocks, w.block_size, w.num_kv_heads, 128)
    with pytest.raises(ValueError, match="head_dim"):
        B._attention_shapes(**dict(att, key_cache=other, value_cache=other))

    sc = dict(key=st.key, value=st.value, key_cache=st.key_cache, value_cache=st.value_cache,
              slot_mapping=st.slot_mapping)
    for name, t in [("value", meta(T + 1, w.num_kv_heads, D)), ("slot_mapping", meta(T - 1, dtype=torch.int64)),
                    ("key", meta(T, w.num_kv_heads + 1, D))]:
        kw = dict(sc, **{name: t})
        if name == "key":
            kw["value"] = t
        with pytest.raises(ValueError):
            B._scatter_shapes(**kw)

    table = meta(64, 64, dtype=torch.float32)
    pos = meta(T, dtype=torch.int64)
    with pytest.raises(ValueError):
        B._rope_shapes(st.q, st.key, st.value, st.key_cache, st.value_cache, st.slot_mapping,
                       meta(T + 2, dtype=torch.int64), table)
    with pytest.raises(ValueError):
        B._rope_shapes(meta(T, H, D + 8), st.key, st.value, st.key_cache, st.value_cache, st.slot_mapping, pos,
                       table)
    with pytest.raises(ValueError):
        B._rope_shapes(st.q, st.key, st.value, st.key_cache, st.value_cache, st.slot_mapping, pos,
                       meta(64 * 64, dtype=torch.float32))

    L = int(w.seq_lens.max())
    ok = meta(L, w.num_kv_heads, D)
    with pytest.raises(ValueError):
        B._gather_shapes(st.key_cache, st.value_cache, st.block_tables[0], L, meta(L - 1, w.num_kv_heads, D), ok)
    with pytest.raises(ValueError):
        B._gather_shapes(st.key_cache, st.value_cache, meta(0, dtype=torch.int32), L, ok, ok)  # no blocks


def test_binding_refuses_host_tensors_before_calling_the_library():
    w = W.tiny_decode(seed=0)
    st = meta_step(w)
    launches = B.pa_launch_count()
    with pytest.raises(TypeError):
        B.pa_attention_varlen(st.q, st.key_cache, st.value_cache, st.block_tables, st.seq_lens,
                              st.query_start_loc, w.max_query_len, w.max_seq_len, w.scale, st.out, st.workspace)
    with pytest.raises(TypeError):
        B.pa_reshape_and_cache(st.key, st.value, st.key_cache, st.value_cache, st.slot_mapping)
    assert B.pa_launch_count() == launches
