"""Seeded random problems over every supported combination, against the oracle
(needs a GB300): group size, head dim, block size, element type, ragged
lengths (empty requests, decode tokens, short drafts, prefill chunks), sharp
scores. Each case is small enough for the full fp64 oracle."""

import numpy as np
import pytest

from paged_kv_cache_55_gb300 import workloads as W

from test_gpu_fp8 import run_fp8
from test_gpu_parity import run_and_check

pytestmark = pytest.mark.gpu


def random_case(seed: int) -> W.Workload:
    rng = np.random.default_rng(1000 + seed)
    G = int(rng.choice([1, 2, 4, 8]))
    Hkv = int(rng.choice([1, 2, 4]))
    D = int(rng.choice([64, 80, 96, 128, 256]))
    bs = int(rng.choice([8, 16, 32]))
    dtype = str(rng.choice(["bf16", "fp16"]))
    B = int(rng.integers(1, 13))
    ctx = np.rint(np.exp(rng.uniform(0, np.log(3000), size=B))).astype(int) - 1
    kind = rng.choice(["empty", "decode", "draft", "chunk"], size=B, p=[0.1, 0.5, 0.15, 0.25])
    ql = np.where(kind == "empty", 0, np.where(kind == "decode", 1, np.where(
        kind == "draft", rng.integers(2, 10, size=B), rng.integers(10, 300, size=B))))
    q_scale = float(rng.choice([1.0, 4.0]))
    kv = W.FP8_E4M3 if seed % 3 == 2 else ""  # every third case over 8-bit caches
    name = f"fuzz{seed}_g{G}_hkv{Hkv}_d{D}_bs{bs}_{dtype}_q{q_scale:g}{'_fp8' if kv else ''}"
    return W.make_workload(name, context_lens=ctx, query_lens=ql, num_heads=Hkv * G, num_kv_heads=Hkv,
                           head_dim=D, block_size=bs, seed=seed, dtype=dtype, q_scale=q_scale, kv_dtype=kv)


@pytest.mark.parametrize("seed", range(24))
def test_random_problem_matches_oracle(oracle, seed):
    w = random_case(seed)
    if w.kv_fp8:
        run_fp8(w, oracle)
    else:
        run_and_check(w, oracle)
