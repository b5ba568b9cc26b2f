"""pa_attention_varlen_static: the attention entry point for callers that cannot allocate.

Some callers cannot call cudaMalloc: a plugin inside a host framework that
owns every device allocation, or a serving process whose device memory is all
reserved up front by its own pool.
For them the library offers a variant that takes no workspace and uses a
scratch array compiled into the library instead. This test calls it through
the C ABI, twice in a row (the second call reuses whatever the first left in
the array), and checks both outputs against the regular entry point's output
within the attention tolerance of the other GPU tests. It also checks that a
problem too big for the array is refused before anything is launched.

Kept in its own file, collected last, so a failure here cannot hide others.
"""

import ctypes

import numpy as np
import pytest
import torch

from paged_kv_cache_55_gb300 import binding as B
from paged_kv_cache_55_gb300 import workloads as W
from paged_kv_cache_55_gb300.runner import DeviceStep, bf16_to_float64, bf16_to_numpy_bits

pytestmark = pytest.mark.gpu

ATOL, RTOL = 2e-3, 1e-2


def _static_call(st: DeviceStep, out: torch.Tensor, dtype: int = B.PA_BF16) -> int:
    w = st.w
    lib = B._lib()
    return lib.pa_attention_varlen_static(
        st.q.data_ptr(), st.q.stride(0), st.key_cache.data_ptr(), st.value_cache.data_ptr(),
        st.block_tables.data_ptr(), st.block_tables.shape[1], st.seq_lens.data_ptr(), st.query_start_loc.data_ptr(),
        w.num_seqs, w.total_q, st.max_query_len, st.max_seq_len, w.num_heads, w.num_kv_heads, w.head_dim,
        w.block_size, w.num_blocks, ctypes.c_float(w.scale), out.data_ptr(), dtype,
        torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_static_workspace_matches_regular_entry_point_twice(dtype):
    # decode requests long enough to be split into partitions, plus causal prefill chunks
    w = W.make_workload("no_alloc", context_lens=[3000, 17, 900, 0, 1500, 64, 2600, 5],
                        query_lens=[1, 1, 1, 33, 1, 12, 1, 1], num_heads=32, num_kv_heads=8, head_dim=128, seed=13,
                        dtype=dtype)
    st = DeviceStep(w)
    need = B.pa_attention_workspace_size(w.num_seqs, w.total_q, st.max_query_len, st.max_seq_len, w.num_heads,
                                         w.num_kv_heads, w.head_dim)
    assert 0 < need <= B.PA_STATIC_WORKSPACE_BYTES
    st.run()  # regular entry point, caller-provided workspace
    torch.cuda.synchronize()
    ref = bf16_to_float64(st.out)
    ref_bits = bf16_to_numpy_bits(st.out)
    for _ in range(2):
        out = torch.full_like(st.out, float("nan"))
        assert _static_call(st, out, B.PA_FP16 if dtype == "fp16" else B.PA_BF16) == 0
        torch.cuda.synchronize()
        assert B.pa_debug_status() == 0
        got = bf16_to_float64(out)
        assert np.isfinite(got).all()
        assert (np.abs(got - ref) <= ATOL + RTOL * np.abs(ref)).all()
        assert np.array_equal(bf16_to_numpy_bits(out), ref_bits)


def test_static_workspace_refuses_problems_that_do_not_fit():
    w = W.tiny_decode(seed=0)
    st = DeviceStep(w)
    launches = B.pa_launch_count()
    lib = B._lib()
    big_seq = 1 << 25  # a 32M-token bound needs more partials than the array holds, at any partition size
    assert B.pa_attention_workspace_size(w.num_seqs, w.total_q, st.max_query_len, big_seq, w.num_heads,
                                         w.num_kv_heads, w.head_dim) > B.PA_STATIC_WORKSPACE_BYTES
    rc = lib.pa_attention_varlen_static(
        st.q.data_ptr(), st.q.stride(0), st.key_cache.data_ptr(), st.value_cache.data_ptr(),
        st.block_tables.data_ptr(), st.block_tables.shape[1], st.seq_lens.data_ptr(), st.query_start_loc.data_ptr(),
        w.num_seqs, w.total_q, st.max_query_len, big_seq, w.num_heads, w.num_kv_heads, w.head_dim,
        w.block_size, w.num_blocks, ctypes.c_float(w.scale), st.out.data_ptr(), B.PA_BF16,
        torch.cuda.current_stream().cuda_stream)
    assert rc == -5  # PA_ERR_WORKSPACE
    assert B.pa_launch_count() == launches

