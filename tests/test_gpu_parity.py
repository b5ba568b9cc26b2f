"""CUDA path against the fp64 CPU oracle, through the C ABI (needs a GB300).

Tolerance for attention outputs (bf16 inputs, fp32 accumulation, bf16
output): |gpu - oracle| <= 2e-3 + 1e-2 * |oracle| elementwise. The cache
scatter and block-table gather must match bit for bit.
"""

import numpy as np
import pytest
import torch

from paged_kv_cache_55_gb300 import binding as B
from paged_kv_cache_55_gb300 import workloads as W
from paged_kv_cache_55_gb300.runner import DeviceStep, bf16_tensor, bf16_to_float64, bf16_to_numpy_bits

pytestmark = pytest.mark.gpu

ATOL, RTOL = 2e-3, 1e-2


def assert_attention_close(gpu: np.ndarray, ref: np.ndarray, what: str = ""):
    assert gpu.shape == ref.shape
    err = np.abs(gpu - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; "
                             f"first {idx.tolist()} gpu={gpu[bad][:5]} ref={ref[bad][:5]}")


def run_and_check(w: W.Workload, oracle, check_status=True):
    st = DeviceStep(w)
    st.run()
    torch.cuda.synchronize()
    if check_status:
        assert B.pa_debug_status() == 0
    kc, vc, ref = oracle.run_step(w)
    assert np.array_equal(bf16_to_numpy_bits(st.key_cache), kc), "key cache differs after reshape_and_cache"
    assert np.array_equal(bf16_to_numpy_bits(st.value_cache), vc), "value cache differs after reshape_and_cache"
    gpu = bf16_to_float64(st.out)
    assert np.isfinite(gpu).all(), "non-finite output (a masked or unowned slot leaked)"
    assert_attention_close(gpu, ref, w.name)
    return st, ref


SMALL_CASES = {
    # name: kwargs of make_workload
    "ragged_decode_g4_d128": dict(context_lens=[0, 6, 15, 16, 511, 512, 513, 1100, 1535, 2047, 40, 3],
                                  query_lens=[1] * 12, num_heads=32, num_kv_heads=8, head_dim=128),
    "decode_g8_d128_long": dict(context_lens=[4999, 700, 32], query_lens=[1] * 3,
                                num_heads=64, num_kv_heads=8, head_dim=128),
    # one very long request: few (request, KV head) pairs, so partitions of 1024 keys
    "single_long_request_g8": dict(context_lens=[99999], query_lens=[1], num_heads=64, num_kv_heads=8, head_dim=128),
    "decode_g1_d64": dict(context_lens=[100, 1, 900, 513], query_lens=[1] * 4,
                          num_heads=4, num_kv_heads=4, head_dim=64),
    "decode_g2_d64": dict(context_lens=[30, 1400, 7], query_lens=[1] * 3,
                          num_heads=8, num_kv_heads=4, head_dim=64),
    "decode_g4_d64": dict(context_lens=[77, 600], query_lens=[1, 1], num_heads=8, num_kv_heads=2, head_dim=64),
    "decode_g8_d64": dict(context_lens=[1030, 3], query_lens=[1, 1], num_heads=16, num_kv_heads=2, head_dim=64),
    "mixed_chunks_g4_d128": dict(context_lens=[0, 37, 600, 20, 1000, 5, 0],
                                 query_lens=[40, 2, 1, 129, 1, 7, 1],
                                 num_heads=32, num_kv_heads=8, head_dim=128),
    "mixed_chunks_g1_d128": dict(context_lens=[0, 300, 64], query_lens=[17, 1, 33],
                                 num_heads=4, num_kv_heads=4, head_dim=128),
    # head dims 80 and 96: rows padded to two 64-element atoms, zero-filled past head_dim
    "decode_g4_d80": dict(context_lens=[0, 700, 33, 1500], query_lens=[1, 1, 2, 1], num_heads=16, num_kv_heads=4,
                          head_dim=80),
    "decode_g8_d96": dict(context_lens=[1030, 3, 260], query_lens=[1, 1, 1], num_heads=16, num_kv_heads=2,
                          head_dim=96),
    "chunks_g4_d80": dict(context_lens=[0, 37, 600, 20], query_lens=[40, 2, 1, 300], num_heads=16, num_kv_heads=4,
                          head_dim=80),
    "chunks_g1_d96": dict(context_lens=[0, 1000, 5], query_lens=[300, 260, 129], num_heads=4, num_kv_heads=4,
                          head_dim=96),
    "chunks_g2_d96": dict(context_lens=[500, 0], query_lens=[77, 200], num_heads=8, num_kv_heads=4, head_dim=96,
                          q_scale=8.0),
    "mixed_chunks_g8_d64": dict(context_lens=[10, 800, 0], query_lens=[5, 1, 24],
                                num_heads=16, num_kv_heads=2, head_dim=64),
    # chunks that fill both 128-row halves of a tile, several tiles and a ragged tail
    "long_chunks_g1_d64": dict(context_lens=[0, 1000, 5], query_lens=[300, 260, 129],
                               num_heads=4, num_kv_heads=4, head_dim=64),
    "long_chunks_g2_d128": dict(context_lens=[130, 0], query_lens=[389, 1],
                                num_heads=8, num_kv_heads=4, head_dim=128),
    # sharp scores over several 128-key ranges: row maxima grow within ranges
    "sharp_long_chunks_g4_d128": dict(context_lens=[200, 0], query_lens=[300, 130], num_heads=8, num_kv_heads=2,
                                      head_dim=128, q_scale=8.0),
    # 8- and 32-token cache blocks (16-key tiles are two blocks or half a block)
    "block8_decode_g4_d128": dict(context_lens=[0, 6, 15, 16, 511, 1100, 40, 3], query_lens=[1] * 8, num_heads=32,
                                  num_kv_heads=8, head_dim=128, block_size=8),
    "block32_decode_g8_d64": dict(context_lens=[1030, 3, 31, 32, 33, 700], query_lens=[1] * 6, num_heads=16,
                                  num_kv_heads=2, head_dim=64, block_size=32),
    "block8_mixed_chunks_g4_d128": dict(context_lens=[0, 37, 600, 20, 5], query_lens=[40, 2, 1, 129, 7],
                                        num_heads=32, num_kv_heads=8, head_dim=128, block_size=8),
    "block32_mixed_chunks_g2_d128": dict(context_lens=[130, 0, 999], query_lens=[389, 1, 70], num_heads=8,
                                         num_kv_heads=4, head_dim=128, block_size=32),
    "block8_long_request_g8": dict(context_lens=[20000], query_lens=[1], num_heads=64, num_kv_heads=8,
                                   head_dim=128, block_size=8),
    "empty_requests": dict(context_lens=[10, 0, 700, 33], query_lens=[0, 1, 0, 3],
                           num_heads=8, num_kv_heads=2, head_dim=128),
    "sharp_scores": dict(context_lens=[300, 1800, 4], query_lens=[1, 1, 9], num_heads=32, num_kv_heads=8,
                         head_dim=128, q_scale=8.0),
    "seq_len_one": dict(context_lens=[0, 0, 0], query_lens=[1, 1, 1], num_heads=8, num_kv_heads=2, head_dim=64),
    # head_dim 256: decode (four warps per SM, 16 KB ring slots), split requests (merge of
    # 8 outputs per lane), and the one-half tile kernel (128-row tiles, two score buffers)
    "decode_g4_d256": dict(context_lens=[0, 700, 33, 1500, 2047], query_lens=[1] * 5, num_heads=16,
                           num_kv_heads=4, head_dim=256),
    "decode_g8_d256_long": dict(context_lens=[5000, 31, 0], query_lens=[1, 1, 1], num_heads=16, num_kv_heads=2,
                                head_dim=256),
    "chunks_g2_d256": dict(context_lens=[0, 300, 1000, 7], query_lens=[200, 1, 130, 3], num_heads=8,
                           num_kv_heads=4, head_dim=256),
    "chunks_g1_d256_sharp": dict(context_lens=[500, 0], query_lens=[140, 300], num_heads=4, num_kv_heads=4,
                                 head_dim=256, q_scale=8.0),
    "chunks_g8_d256": dict(context_lens=[10, 2000, 0], query_lens=[40, 1, 17], num_heads=16, num_kv_heads=2,
                           head_dim=256),
    "chunks_g4_d256": dict(context_lens=[0, 37, 600, 20, 1000], query_lens=[40, 2, 1, 129, 1], num_heads=16,
                           num_kv_heads=4, head_dim=256),
    "block8_chunks_g4_d256": dict(context_lens=[0, 37, 600, 20], query_lens=[40, 2, 1, 129], num_heads=8,
                                  num_kv_heads=2, head_dim=256, block_size=8),
    "block32_mixed_g2_d256": dict(context_lens=[130, 0, 999, 3000], query_lens=[389, 1, 70, 1], num_heads=8,
                                  num_kv_heads=4, head_dim=256, block_size=32),
    "seq_len_one_d256": dict(context_lens=[0, 0], query_lens=[1, 1], num_heads=4, num_kv_heads=2, head_dim=256),
}


def test_growing_key_norms_rescale_within_ranges(oracle):
    # Keys whose norm grows along the chunk make each row's running maximum
    # jump by more than 2^8 inside a 128-key range again and again, so the
    # probabilities already written for the range, O and the row sum are
    # rescaled mid-range (the prefill tile path; G = 4 and G = 1).
    for heads, kv_heads, d in ((8, 2, 128), (4, 4, 64), (8, 4, 256)):
        w = W.make_workload("growing_keys", context_lens=[0, 37], query_lens=[256, 200], num_heads=heads,
                            num_kv_heads=kv_heads, head_dim=d, seed=11, q_scale=2.0)
        k = W.bf16_bits_to_f32(w.key)
        q0 = np.asarray(w.query_start_loc)
        for b in range(w.num_seqs):
            n = int(q0[b + 1] - q0[b])
            k[q0[b]:q0[b + 1]] *= (1.0 + np.arange(n, dtype=np.float32) / 8.0)[:, None, None]
        w.key = W.f32_to_bf16_bits(k)
        run_and_check(w, oracle)


def test_tiny_decode(oracle):
    run_and_check(W.tiny_decode(seed=0), oracle)


@pytest.mark.parametrize("name", sorted(SMALL_CASES))
def test_small_cases(oracle, name):
    w = W.make_workload(name, seed=5, **SMALL_CASES[name])
    run_and_check(w, oracle)


FP16_CASES = ["block8_mixed_chunks_g4_d128", "block32_decode_g8_d64", "ragged_decode_g4_d128", "decode_g8_d64", "decode_g1_d64", "mixed_chunks_g4_d128",
              "mixed_chunks_g1_d128", "mixed_chunks_g8_d64", "long_chunks_g2_d128", "sharp_long_chunks_g4_d128",
              "empty_requests", "seq_len_one", "chunks_g2_d256", "decode_g8_d256_long", "block32_mixed_g2_d256"]


@pytest.mark.parametrize("name", FP16_CASES)
def test_small_cases_fp16(oracle, name):
    """The same cases with fp16 q, K/V and out (the oracle decodes IEEE binary16)."""
    w = W.make_workload(name, seed=6, dtype="fp16", **SMALL_CASES[name])
    assert w.dtype == "fp16"
    run_and_check(w, oracle)


def test_repeated_steps_on_reused_memory(oracle):
    """Fresh buffers each time (the caching allocator hands back the previous
    step's memory, stale plans included) and a torch kernel right before the
    step: the plan must be read only after it is written."""
    kw = SMALL_CASES["mixed_chunks_g4_d128"]
    w = W.make_workload("repeat", seed=5, **kw)
    kc, vc, ref = oracle.run_step(w)
    for trial in range(6):
        st = DeviceStep(w)
        st.out.fill_(float("nan") if trial % 2 else 0.0)
        st.run()
        torch.cuda.synchronize()
        assert B.pa_debug_status() == 0
        gpu = bf16_to_float64(st.out)
        assert np.isfinite(gpu).all(), f"trial {trial}: non-finite output"
        assert_attention_close(gpu, ref, f"trial {trial}")
        del st


def test_batch_larger_than_one_planning_block(oracle):
    """More than 1024 requests: the planner's chunked two-pass path."""
    rng = np.random.default_rng(77)
    B_ = 1500
    ctx = rng.integers(0, 700, size=B_)
    ql = np.where(rng.random(B_) < 0.05, rng.integers(2, 6, size=B_), 1)
    w = W.make_workload("many", context_lens=ctx, query_lens=ql, num_heads=8, num_kv_heads=2, head_dim=64, seed=78)
    run_and_check(w, oracle)


def test_shared_prefix_step(oracle):
    w = W.mixed_step(seed=2, n_prefill=3, chunk=96, n_decode=20, n_shared=8, shared_blocks=6)
    run_and_check(w, oracle)


@pytest.mark.parametrize("case", ["seq_len_one", "seq_len_one_d256"])
def test_seq_len_one_returns_v_row_exactly(case):
    w = W.make_workload("one", seed=9, **SMALL_CASES[case])
    st = DeviceStep(w)
    st.run()
    out = bf16_to_numpy_bits(st.out)
    G = w.num_heads // w.num_kv_heads
    for b in range(w.num_seqs):
        for h in range(w.num_heads):
            assert np.array_equal(out[b, h], w.value[b, h // G]), "seq_len 1 must return the new V row"


def test_block_permutation_gives_identical_bits():
    """Relabelling physical blocks (cache moved with the table) must not change one output bit."""
    base = W.make_workload("perm", seed=21, **SMALL_CASES["ragged_decode_g4_d128"])
    a = DeviceStep(base)
    a.run()
    rng = np.random.default_rng(4)
    perm = rng.permutation(base.num_blocks)  # old id -> new id
    w2 = W.make_workload("perm", seed=21, **SMALL_CASES["ragged_decode_g4_d128"])
    inv = np.empty_like(perm)
    inv[perm] = np.arange(perm.size)
    w2.key_cache = base.key_cache[inv]
    w2.value_cache = base.value_cache[inv]
    used = w2.block_tables >= 0
    w2.block_tables = np.where(used & (w2.block_tables < base.num_blocks),
                               perm[np.clip(w2.block_tables, 0, base.num_blocks - 1)], w2.block_tables).astype(np.int32)
    bs = base.block_size
    w2.slot_mapping = perm[base.slot_mapping // bs] * bs + base.slot_mapping % bs
    b = DeviceStep(w2)
    b.run()
    assert np.array_equal(bf16_to_numpy_bits(a.out), bf16_to_numpy_bits(b.out))


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_copy_blocks_bit_exact(oracle, dtype):
    """Copy-on-write block copy against the oracle, bit for bit; 3000 pairs over a
    GQA-shaped pool (and a small D = 64 pool), raw bits of either element type."""
    rng = np.random.default_rng(31)
    for nb, hkv, d, npairs in ((7000, 8, 128, 3000), (50, 2, 64, 17)):
        w = W.make_workload("copy", context_lens=[nb * 16 // 2], query_lens=[1], num_heads=hkv * 4,
                            num_kv_heads=hkv, head_dim=d, num_blocks=nb, seed=8, dtype=dtype)
        ids = rng.permutation(nb)
        m = np.stack([ids[:npairs], ids[npairs:2 * npairs]], axis=1).astype(np.int64)
        kc, vc = w.key_cache.copy(), w.value_cache.copy()
        oracle.copy_blocks(kc, vc, m)
        kt = bf16_tensor(w.key_cache, "cuda", dtype)
        vt = bf16_tensor(w.value_cache, "cuda", dtype)
        B.pa_copy_blocks(kt, vt, torch.from_numpy(m).cuda())
        torch.cuda.synchronize()
        assert B.pa_debug_status() == 0
        assert np.array_equal(bf16_to_numpy_bits(kt), kc) and np.array_equal(bf16_to_numpy_bits(vt), vc)


def test_copy_blocks_flags_and_skips_bad_ids():
    w = W.make_workload("copy", context_lens=[100], query_lens=[1], num_heads=8, num_kv_heads=2, head_dim=64,
                        num_blocks=12, seed=9)
    kt = bf16_tensor(w.key_cache, "cuda")
    vt = bf16_tensor(w.value_cache, "cuda")
    m = torch.tensor([[1, 2], [3, 12], [-1, 4], [5, 6]], dtype=torch.int64, device="cuda")
    B.pa_copy_blocks(kt, vt, m)
    flags = B.pa_debug_status()
    assert flags == B.FLAG_BLOCK_RANGE
    k = bf16_to_numpy_bits(kt)
    assert np.array_equal(k[2], w.key_cache[1]) and np.array_equal(k[6], w.key_cache[5])
    assert np.array_equal(k[4], w.key_cache[4]) and np.array_equal(k[11], w.key_cache[11])  # skipped pairs
    B.pa_copy_blocks(kt, vt, torch.zeros((0, 2), dtype=torch.int64, device="cuda"))  # nothing to do
    assert B.pa_debug_status() == 0


@pytest.mark.parametrize("bs", [8, 16, 32])
def test_gather_kv_bit_exact(bs):
    kw = dict(SMALL_CASES["ragged_decode_g4_d128"], block_size=bs)
    w = W.make_workload("gather", seed=3, **kw)
    st = DeviceStep(w)
    st.reshape_and_cache()
    kc = bf16_to_numpy_bits(st.key_cache)
    vc = bf16_to_numpy_bits(st.value_cache)
    for b in range(w.num_seqs):
        L = int(w.seq_lens[b])
        ko = torch.empty((L, w.num_kv_heads, w.head_dim), dtype=torch.bfloat16, device="cuda")
        vo = torch.empty_like(ko)
        B.pa_gather_kv(st.key_cache, st.value_cache, st.block_tables[b], L, ko, vo)
        j = np.arange(L)
        rows = w.block_tables[b, j // bs]
        assert np.array_equal(bf16_to_numpy_bits(ko), kc[rows, j % bs])
        assert np.array_equal(bf16_to_numpy_bits(vo), vc[rows, j % bs])
    assert B.pa_debug_status() == 0


def test_out_of_range_slot_is_flagged_and_skipped():
    w = W.tiny_decode(seed=1)
    st = DeviceStep(w)
    bad = st.slot_mapping.clone()
    bad[1] = w.num_blocks * w.block_size + 5
    bad[2] = -1
    B.pa_reshape_and_cache(st.key, st.value, st.key_cache, st.value_cache, bad)
    flags = B.pa_debug_status()
    assert flags & B.FLAG_SLOT_RANGE
    kc = bf16_to_numpy_bits(st.key_cache).reshape(-1, w.num_kv_heads, w.head_dim)
    for t in (0, 3):
        assert np.array_equal(kc[w.slot_mapping[t]], w.key[t])
    for t in (1, 2):
        assert np.array_equal(kc[w.slot_mapping[t]], w.key_cache.reshape(-1, w.num_kv_heads, w.head_dim)[w.slot_mapping[t]])
    assert B.pa_debug_status() == 0  # cleared by the previous read


def test_out_of_range_block_id_is_flagged():
    w = W.make_workload("badblock", seed=8, **SMALL_CASES["decode_g4_d64"])
    st = DeviceStep(w)
    st.reshape_and_cache()
    st.block_tables[1, 0] = w.num_blocks + 3
    st.attention()
    flags = B.pa_debug_status()
    assert flags & B.FLAG_BLOCK_RANGE
    out = bf16_to_float64(st.out)
    assert np.isfinite(out[0]).all()


def test_inconsistent_lengths_are_flagged():
    w = W.make_workload("badlen", seed=8, **SMALL_CASES["decode_g4_d64"])
    st = DeviceStep(w)
    st.reshape_and_cache()
    st.seq_lens[0] = w.max_seq_len + 1  # above the host bound
    st.attention()
    assert B.pa_debug_status() & B.FLAG_LENGTHS


def test_host_side_errors():
    w = W.tiny_decode(seed=0)
    st = DeviceStep(w)
    lib = B._lib()
    s = torch.cuda.current_stream().cuda_stream
    base = [st.q.data_ptr(), st.q.stride(0), st.key_cache.data_ptr(), st.value_cache.data_ptr(),
            st.block_tables.data_ptr(), st.block_tables.shape[1], st.seq_lens.data_ptr(),
            st.query_start_loc.data_ptr(), w.num_seqs, w.total_q, w.max_query_len, w.max_seq_len,
            w.num_heads, w.num_kv_heads, w.head_dim, 16, w.num_blocks, w.scale, st.out.data_ptr(),
            st.workspace.data_ptr(), st.workspace.numel(), 0, s]

    def call(**chg):
        a = list(base)
        names = ["q", "qs", "kc", "vc", "bt", "mb", "sl", "qsl", "B", "T", "mq", "ms", "H", "Hkv", "D", "bs",
                 "nb", "scale", "out", "ws", "wsb", "dtype", "stream"]
        for k, v in chg.items():
            a[names.index(k)] = v
        return lib.pa_attention_varlen(*a)

    assert call() == 0
    assert call(q=None) == -1
    assert call(D=112) == -3
    assert call(bs=64) == -3
    assert call(Hkv=3) == -2
    assert call(dtype=2) == -3  # 0 = bf16, 1 = fp16
    assert call(wsb=16) == -5
    assert call(out=st.out.data_ptr() + 2) == -4
    assert call(scale=float("nan")) == -2
    torch.cuda.synchronize()
    assert B.pa_debug_status() == 0


# --------------------------------------------------------------------------
# Full-size named workloads, in the launch configuration the benchmark times,
# compared with the oracle at every output element (the oracle evaluates the
# whole step on the host cores: a few seconds per decode workload, about ten
# for the mixed step's prefill chunks).
# --------------------------------------------------------------------------

NAMED = ["mha_decode", "gqa_decode", "long_decode", "mixed_step"]


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("name", NAMED)
def test_named_full_size(oracle, name, dtype):
    """Every output of the full-size workload against the oracle, and the whole
    cache bit for bit after the scatter (rows written and rows left alone)."""
    w = W.by_name(name, seed=0, dtype=dtype)
    run_and_check(w, oracle)


def test_gqa_decode_other_seeds(oracle):
    """The headline workload drawn from two more seeds (other lengths, blocks and values)."""
    for seed in (1, 2):
        run_and_check(W.by_name("gqa_decode", seed=seed), oracle)


def test_huge_scores_in_prefill_tiles(oracle):
    """Scores of order 1e10 (log2 domain) in the tensor-core tiles: the softmax exponent must
    stay bounded although the products are far beyond fp32's integer precision. (bf16 q of
    order 1e10: the softmax is one-hot, so fp32 accumulation error, which grows with |q.k|,
    cannot move a near tie; fp16 q is limited to 65504.)"""
    w = W.make_workload("huge_scores", context_lens=[900, 0, 2100], query_lens=[150, 300, 1],
                        num_heads=32, num_kv_heads=8, head_dim=128, q_scale=2.0e9, seed=21)
    run_and_check(w, oracle)


def test_large_fp16_scores_in_prefill_tiles(oracle):
    w = W.make_workload("large_scores_fp16", context_lens=[900, 0, 2100], query_lens=[150, 300, 1],
                        num_heads=32, num_kv_heads=8, head_dim=128, q_scale=300.0, seed=21, dtype="fp16")
    run_and_check(w, oracle)


@pytest.mark.parametrize("head_dim,block_size", [(128, 16), (128, 8), (128, 32), (96, 16), (64, 16)])
def test_bf16_values_beyond_fp16_in_prefill_tiles(oracle, head_dim, block_size):
    """bf16 V rows holding magnitudes that no fp16 value reaches (65536 up to 1e30): the
    tensor-core tiles keep those key ranges in bf16 (P as a hi + lo pair) and rewrite the
    other ranges of the same tiles as fp16; 65280, the largest bf16 value below 65504, stays
    on the fp16 path."""
    w = W.make_workload("big_v", context_lens=[700, 300, 0], query_lens=[200, 250, 130], num_heads=16,
                        num_kv_heads=4, head_dim=head_dim, block_size=block_size, seed=23)
    rng = np.random.default_rng(5)
    bs, D = w.block_size, w.head_dim
    vc = w.value_cache.reshape(-1, w.num_kv_heads, D)
    for pos in (260, 300, 301):  # request 0, its third range of 128 keys
        slot = int(w.block_tables[0, pos // bs]) * bs + pos % bs
        vc[slot, 1] = W.f32_to_bf16_bits((rng.standard_normal(D) * 1e5).astype(np.float32))
    slot = int(w.block_tables[0, 40 // bs]) * bs + 40 % bs  # its first range: 65280 fits fp16
    vc[slot, 3, :2] = W.f32_to_bf16_bits(np.array([65280.0, -65280.0], np.float32))
    row = int(w.query_start_loc[1]) + 7  # request 1, a new V row at position 307
    w.value[row, 2, :5] = W.f32_to_bf16_bits(np.array([7e4, -3e6, 1e30, 65280.0, -65536.0], np.float32))
    run_and_check(w, oracle)
