"""8-bit (E4M3) KV caches through the C ABI against the fp64 oracle (needs a GB300).

The quantising scatter and the byte copies must match the oracle bit for bit;
attention outputs must be within |gpu - oracle| <= 2e-3 + 1e-2 |oracle|,
where the oracle decodes every code exactly and multiplies by the cache scale.
"""

import numpy as np
import pytest
import torch

from paged_kv_cache_55_gb300 import binding as B
from paged_kv_cache_55_gb300 import workloads as W
from paged_kv_cache_55_gb300.runner import DeviceStep, bf16_to_float64

from test_gpu_parity import NAMED, assert_attention_close

pytestmark = pytest.mark.gpu

FP8 = W.FP8_E4M3


def run_fp8(w: W.Workload, oracle):
    st = DeviceStep(w)
    st.run()
    torch.cuda.synchronize()
    assert B.pa_debug_status() == 0
    kc, vc, ref = oracle.run_step(w)
    assert np.array_equal(st.key_cache.cpu().numpy(), kc), "8-bit key cache differs after the quantising scatter"
    assert np.array_equal(st.value_cache.cpu().numpy(), vc), "8-bit value cache differs after the quantising scatter"
    gpu = bf16_to_float64(st.out)
    assert np.isfinite(gpu).all(), "non-finite output (a masked or unowned slot leaked)"
    assert_attention_close(gpu, ref, w.name)
    return st, ref


CASES = {
    # name: (make_workload kwargs); query_len <= 8 / G (decode tokens and short drafts)
    "g4_d128_ragged": dict(context_lens=[0, 6, 15, 16, 511, 512, 513, 1100, 1535, 2047, 40, 3],
                           query_lens=[1] * 12, num_heads=32, num_kv_heads=8, head_dim=128),
    "g8_d128_long": dict(context_lens=[4999, 700, 32], query_lens=[1] * 3, num_heads=64, num_kv_heads=8,
                         head_dim=128),
    "g8_d128_one_long_request": dict(context_lens=[70000], query_lens=[1], num_heads=64, num_kv_heads=8,
                                     head_dim=128),
    "g1_d64": dict(context_lens=[100, 1, 900, 513], query_lens=[1] * 4, num_heads=4, num_kv_heads=4, head_dim=64),
    "g2_d64_drafts": dict(context_lens=[30, 1400, 7], query_lens=[4, 1, 3], num_heads=8, num_kv_heads=4,
                          head_dim=64),
    "g1_d128_drafts": dict(context_lens=[0, 300, 64, 2000], query_lens=[8, 1, 5, 7], num_heads=4, num_kv_heads=4,
                           head_dim=128),
    "g2_d128_drafts_empty": dict(context_lens=[50, 0, 777], query_lens=[4, 0, 2], num_heads=8, num_kv_heads=4,
                                 head_dim=128),
    "g4_d64": dict(context_lens=[77, 600], query_lens=[2, 1], num_heads=8, num_kv_heads=2, head_dim=64),
    "g8_d64": dict(context_lens=[1030, 3], query_lens=[1, 1], num_heads=16, num_kv_heads=2, head_dim=64),
    "g4_d128_sharp": dict(context_lens=[300, 2500, 17], query_lens=[1, 2, 1], num_heads=32, num_kv_heads=8,
                          head_dim=128, q_scale=8.0),
    # chunked-prefill chunks (tensor-core tiles over 8-bit caches) mixed with decode tokens
    "g4_d128_chunks": dict(context_lens=[0, 37, 600, 20, 1000, 5, 0], query_lens=[40, 2, 1, 129, 1, 7, 300],
                           num_heads=32, num_kv_heads=8, head_dim=128),
    "g1_d64_chunks": dict(context_lens=[0, 1000, 5], query_lens=[300, 260, 129], num_heads=4, num_kv_heads=4,
                          head_dim=64),
    "g4_d80_mixed": dict(context_lens=[0, 700, 33, 1500, 20], query_lens=[1, 1, 2, 1, 150], num_heads=16,
                         num_kv_heads=4, head_dim=80),
    "g2_d96_mixed": dict(context_lens=[1030, 3, 260, 0], query_lens=[1, 4, 1, 300], num_heads=8, num_kv_heads=4,
                         head_dim=96),
    "g8_d64_chunks": dict(context_lens=[10, 800, 0], query_lens=[5, 1, 24], num_heads=16, num_kv_heads=2,
                          head_dim=64),
    "g2_d128_sharp_chunks": dict(context_lens=[700, 3000], query_lens=[200, 77], num_heads=8, num_kv_heads=4,
                                 head_dim=128, q_scale=8.0),
    # head_dim 256: rows of two 128-code atoms (decode), units of half a row (tiles)
    "g4_d256_mixed": dict(context_lens=[0, 700, 33, 1500, 20], query_lens=[1, 1, 2, 1, 150], num_heads=16,
                          num_kv_heads=4, head_dim=256),
    "g1_d256_chunks": dict(context_lens=[0, 1000, 5000], query_lens=[300, 130, 1], num_heads=4, num_kv_heads=4,
                           head_dim=256),
}


@pytest.mark.parametrize("bs", [16, 8, 32])
@pytest.mark.parametrize("name", sorted(CASES))
def test_fp8_cases(oracle, name, bs):
    for dtype in ("bf16", "fp16"):
        w = W.make_workload(f"fp8_{name}_bs{bs}_{dtype}", seed=7, block_size=bs, dtype=dtype, kv_dtype=FP8,
                            **CASES[name])
        run_fp8(w, oracle)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("head_dim", [64, 80, 96, 128, 256])
def test_fp8_every_code_round_trips_exactly(dtype, head_dim):
    """seq_len 1: the output is the token's own V row. With v_scale = 2^-4 and V made of
    code values times 2^-4 (exact in bf16 and fp16), the scatter stores those codes and the
    output must be the V row bit for bit: every finite code, subnormals and signed zero
    included, widens exactly and lands at its own d."""
    Hkv, D = 2, head_dim
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    T = -(-codes.size // (Hkv * D)) + 1
    rng = np.random.default_rng(5)
    pick = np.concatenate([codes, rng.choice(codes, size=T * Hkv * D - codes.size)])
    vals = torch.from_numpy(pick).view(torch.float8_e4m3fn).to(torch.float32).numpy() * np.float32(2.0 ** -4)
    w = W.make_workload("fp8_codes", context_lens=[0] * T, query_lens=[1] * T, num_heads=Hkv * 4, num_kv_heads=Hkv,
                        head_dim=D, dtype=dtype, kv_dtype=FP8, k_scale=0.1, v_scale=2.0 ** -4, seed=3)
    w.value = W.f32_to_bits(vals.reshape(T, Hkv, D), dtype)
    st = DeviceStep(w)
    st.run()
    torch.cuda.synchronize()
    assert B.pa_debug_status() == 0
    got = bf16_to_float64(st.out).reshape(T, Hkv, 4, D)
    want = np.repeat(W.bits_to_f32(w.value, dtype)[:, :, None, :], 4, axis=2).astype(np.float64)
    # values, not bits: the fp32 accumulator turns the -0 code's product into +0
    assert np.array_equal(got, want), "seq_len 1 over an 8-bit cache must return the V row exactly"


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("name", NAMED)
def test_fp8_named_full_size(oracle, name, dtype):
    """Full-size workloads over 8-bit caches: the whole quantised cache bit for bit
    and every attention output against the oracle."""
    w = W.by_name(name, seed=0, kv_dtype=FP8, dtype=dtype)
    run_fp8(w, oracle)


@pytest.mark.parametrize("bs", [8, 16, 32])
def test_fp8_copy_blocks_and_gather_bit_exact(oracle, bs):
    w = W.make_workload("fp8_copy", context_lens=[200, 35, 600], query_lens=[1, 1, 1], num_heads=8,
                        num_kv_heads=2, head_dim=128, block_size=bs, kv_dtype=FP8, seed=4)
    st = DeviceStep(w)
    rng = np.random.default_rng(2)
    ids = rng.permutation(w.num_blocks)
    mapping = np.stack([ids[:6], ids[6:12]], axis=1).astype(np.int64)
    B.pa_copy_blocks(st.key_cache, st.value_cache, torch.from_numpy(mapping).cuda())
    kref, vref = w.key_cache.copy(), w.value_cache.copy()
    oracle.copy_blocks(kref, vref, mapping)
    torch.cuda.synchronize()
    assert B.pa_debug_status() == 0
    assert np.array_equal(st.key_cache.cpu().numpy(), kref) and np.array_equal(st.value_cache.cpu().numpy(), vref)
    # block-table gather of request 2 (bytes)
    L = int(w.seq_lens[2])
    ko = torch.empty((L, 2, 128), dtype=torch.uint8, device="cuda")
    vo = torch.empty_like(ko)
    B.pa_gather_kv(st.key_cache, st.value_cache, st.block_tables[2].contiguous(), L, ko, vo)
    torch.cuda.synchronize()
    j = np.arange(L)
    slots = w.block_tables[2, j // bs].astype(np.int64) * bs + j % bs
    assert np.array_equal(ko.cpu().numpy(), kref.reshape(-1, 2, 128)[slots])
    assert np.array_equal(vo.cpu().numpy(), vref.reshape(-1, 2, 128)[slots])


def test_fp8_host_errors():
    w = W.make_workload("fp8_err", context_lens=[10], query_lens=[1], num_heads=8, num_kv_heads=2, head_dim=128,
                        kv_dtype=FP8, seed=1)
    st = DeviceStep(w)
    for ks, vs in ((0.0, 1.0), (1.0, -1.0), (float("inf"), 1.0), (1.0, float("nan"))):
        with pytest.raises(B.PagedAttnError) as e:
            B.pa_attention_varlen_fp8(st.q, st.key_cache, st.value_cache, st.block_tables, st.seq_lens,
                                      st.query_start_loc, 1, 11, w.scale, ks, vs, st.out, st.workspace)
        assert e.value.status == -2
        with pytest.raises(B.PagedAttnError) as e:
            B.pa_reshape_and_cache_fp8(st.key, st.value, st.key_cache, st.value_cache, st.slot_mapping, ks, vs)
        assert e.value.status == -2
    torch.cuda.synchronize()
    assert B.pa_debug_status() == 0


@pytest.mark.parametrize("q_scale", [3.0e4, 2.0e9])
def test_fp8_bf16_queries_beyond_fp16_range(oracle, q_scale):
    """Over 8-bit caches the tensor cores take fp16 operands: bf16 q rows whose largest |q|
    reaches 2^15 (here up to ~1e5 and ~1e10) are scaled by a power of two first, so they must
    still match the oracle (the softmax is then nearly one-hot); decode tokens and a chunk."""
    w = W.make_workload(f"fp8_bigq_{q_scale:g}", context_lens=[40, 900, 3, 2100], query_lens=[1, 2, 1, 150],
                        num_heads=32, num_kv_heads=8, head_dim=128, kv_dtype=FP8, q_scale=q_scale, seed=12)
    run_fp8(w, oracle)
