"""Seeded synthetic inputs for one paged-attention step.

This module builds host arrays only. It holds none of the attention arithmetic:
no scores, no softmax, no gather. Both the CPU oracle and the CUDA library read
what it makes, so neither side can influence the other's inputs.

What a step's inputs are follows the vLLM inference notes
("AI Infra入门干货总结：大模型是如何高效推理的", §Paged Attention and §Continuous
Batching):

* the per-layer KV cache is ``[num_blocks, block_size, num_kv_heads, head_dim]``
  for K and for V (the layer/K-V axes of the 6-D layout are split off);
* ``block_tables[b, i]`` names the physical block that holds logical block ``i``
  of request ``b``;
* ``slot_mapping[t]`` names the flat slot ``block * block_size + offset`` where
  new token ``t`` writes its K/V row;
* each request contributes ``query_len = num_tokens - num_computed_tokens``
  query tokens; ``seq_len`` counts every KV token including this step's.

The generator has to place each request's history into the pool, so it uses
the slot convention above to find where a history row lives. That convention
is the *input contract* (it defines what a valid cache state is); the oracle
and the kernels each implement the reverse mapping on their own.

Element data is bf16, carried as ``uint16`` bit patterns. Unowned slots hold
the bf16 NaN ``0x7FC0`` so that a kernel which reads them leaks NaN into its
output. Block-table entries past a request's last block hold junk.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np

BF16_NAN = np.uint16(0x7FC0)
FP16_NAN = np.uint16(0x7E00)
DTYPES = ("bf16", "fp16")
NAN_BITS = {"bf16": BF16_NAN, "fp16": FP16_NAN}
TABLE_JUNK = np.int32(-2147483648)


def blocks_needed(num_tokens: int, block_size: int) -> int:
    """Pages a request of ``num_tokens`` occupies: ceil(num_tokens / block_size).

    The deployment article's page-allocation diagram (page 4, §2.2) gives the
    worked values: 512 estimated tokens take 4 pages of 128 tokens, 256 take 2,
    and growing past 512 takes one more page.
    """
    if num_tokens < 0 or block_size <= 0:
        raise ValueError("num_tokens must be >= 0 and block_size > 0")
    return (num_tokens + block_size - 1) // block_size


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest even), as uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> 16) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> 16).astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_fp16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to IEEE fp16 (round to nearest even), as uint16 bits."""
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def fp16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    """Widen fp16 bit patterns to float32 (exact)."""
    return np.asarray(h, dtype=np.uint16).view(np.float16).astype(np.float32)


def f32_to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    return f32_to_fp16_bits(x) if dtype == "fp16" else f32_to_bf16_bits(x)


def bits_to_f32(h: np.ndarray, dtype: str) -> np.ndarray:
    return fp16_bits_to_f32(h) if dtype == "fp16" else bf16_bits_to_f32(h)


def rope_cos_sin_cache(max_position: int, rotary_dim: int, base: float = 10000.0) -> np.ndarray:
    """The precomputed rotary table (float32 [max_position, rotary_dim]): row p holds
    cos(p * theta_i) for i < rotary_dim / 2, then sin(p * theta_i), with RoFormer's
    frequencies theta_i = base^(-2 i / rotary_dim). Input data for the rotary step."""
    i = np.arange(rotary_dim // 2, dtype=np.float64)
    theta = base ** (-2.0 * i / rotary_dim)
    ang = np.arange(max_position, dtype=np.float64)[:, None] * theta[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)


FP8_E4M3 = "fp8_e4m3"
FP8_NAN = np.uint8(0x7F)  # E4M3 S.1111.111


def fp8_codes(rng: np.random.Generator, shape, magnitude: float = 16.0) -> np.ndarray:
    """Seeded E4M3 codes (uint8) for cache history: random sign and 3-bit
    fraction, and the exponent field of ``magnitude * |z|`` for z ~ N(0, 1)
    (clipped to the format's exponents 0..15; the NaN pattern becomes the
    largest finite code). Decoded, the values follow ``magnitude * N(0, 1)``
    to within a factor of two, like N(0, 1) data stored with a cache scale of
    1 / magnitude."""
    n = int(np.prod(shape))
    sign = rng.integers(0, 2, size=n, dtype=np.uint8)
    z = np.abs(rng.standard_normal(n)) * magnitude
    e = np.clip(np.floor(np.log2(np.maximum(z, 1e-30))) + 7, 0, 15).astype(np.uint8)
    f = rng.integers(0, 8, size=n, dtype=np.uint8)
    codes = (sign << 7) | (e << 3) | f
    codes[(codes & 0x7F) == 0x7F] -= 1
    return codes.reshape(shape)


def _normal_elems(rng: np.random.Generator, shape, scale: float = 1.0, dtype: str = "bf16") -> np.ndarray:
    """Seeded N(0, scale^2) values rounded to the element type, as uint16 bits
    (the same draws for either type)."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    step = 1 << 24
    for s in range(0, n, step):
        e = min(n, s + step)
        x = rng.standard_normal(e - s, dtype=np.float32)
        if scale != 1.0:
            x *= np.float32(scale)
        out[s:e] = f32_to_bits(x, dtype)
    return out.reshape(shape)


@dataclasses.dataclass
class Workload:
    """One step of paged attention: the cache before the step plus the step's inputs."""

    name: str
    seed: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    scale: float
    q: np.ndarray               # uint16 [T, H, D]
    key: np.ndarray             # uint16 [T, Hkv, D]  new K rows of this step
    value: np.ndarray           # uint16 [T, Hkv, D]  new V rows of this step
    slot_mapping: np.ndarray    # int64  [T]
    key_cache: np.ndarray       # uint16 [num_blocks, bs, Hkv, D]  state before the step
    value_cache: np.ndarray     # uint16 [num_blocks, bs, Hkv, D]
    block_tables: np.ndarray    # int32  [B, max_blocks_per_seq]
    seq_lens: np.ndarray        # int32  [B]
    query_start_loc: np.ndarray  # int32 [B + 1]
    shared_blocks: Optional[np.ndarray] = None  # physical ids shared by several requests
    dtype: str = "bf16"          # element type of q, key, value (and 16-bit caches): "bf16" or "fp16"
    meta: dict = dataclasses.field(default_factory=dict)
    kv_dtype: str = ""           # cache type: "" (= dtype) or "fp8_e4m3" (uint8 codes)
    k_scale: float = 1.0         # 8-bit caches: K value = code * k_scale
    v_scale: float = 1.0

    @property
    def kv_fp8(self) -> bool:
        return self.kv_dtype == FP8_E4M3

    @property
    def num_seqs(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def total_q(self) -> int:
        return int(self.query_start_loc[-1])

    @property
    def query_lens(self) -> np.ndarray:
        return np.diff(self.query_start_loc).astype(np.int32)

    @property
    def max_query_len(self) -> int:
        ql = self.query_lens
        return int(ql.max()) if ql.size else 0

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max()) if self.seq_lens.size else 0

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    def kv_tokens_logical(self) -> int:
        """KV tokens the step reads, counted once per request (shared blocks repeat)."""
        return int(self.seq_lens.astype(np.int64).sum())

    def kv_tokens_unique(self) -> int:
        """KV tokens in distinct physical blocks the step reads (shared prefix once)."""
        bs = self.block_size
        seen = {}
        for b in range(self.num_seqs):
            L = int(self.seq_lens[b])
            nb = blocks_needed(L, bs)
            for i in range(nb):
                blk = int(self.block_tables[b, i])
                used = min(bs, L - i * bs)
                seen[blk] = max(seen.get(blk, 0), used)
        return int(sum(seen.values()))


def make_workload(
    name: str,
    *,
    context_lens: Sequence[int],
    query_lens: Sequence[int],
    num_heads: int,
    num_kv_heads: int,
    head_dim: int,
    block_size: int = 16,
    num_blocks: Optional[int] = None,
    slack: float = 0.10,
    seed: int = 0,
    q_scale: float = 1.0,
    shared_prefix_requests: Sequence[int] = (),
    shared_prefix_blocks: int = 0,
    extra_table_cols: int = 2,
    scale: Optional[float] = None,
    dtype: str = "bf16",
    kv_dtype: str = "",
    k_scale: float = 0.0625 * 1.1,
    v_scale: float = 0.0625 * 0.7,
) -> Workload:
    """Build one step: request ``b`` has ``context_lens[b]`` cached tokens and
    ``query_lens[b]`` new tokens, so ``seq_len = context + query``.

    Physical blocks are drawn from a seeded shuffled pool of ``num_blocks``
    (default: blocks needed + ``slack``). Requests listed in
    ``shared_prefix_requests`` map their first ``shared_prefix_blocks`` logical
    blocks to the same physical blocks (a copy-on-write shared prefix); their
    contexts must fill those blocks so that new tokens land in private blocks.
    Elements are bf16 or fp16 (``dtype``); unowned cache slots hold that
    type's NaN. With ``kv_dtype="fp8_e4m3"`` the caches hold 8-bit codes
    (history drawn by ``fp8_codes``, unowned slots the E4M3 NaN) read with the
    float scales ``k_scale`` and ``v_scale``; the new K/V rows stay 16-bit.
    """
    if dtype not in DTYPES:
        raise ValueError(f"dtype must be one of {DTYPES}")
    if kv_dtype not in ("", dtype, FP8_E4M3):
        raise ValueError("kv_dtype must be empty, equal to dtype, or fp8_e4m3")
    fp8 = kv_dtype == FP8_E4M3
    rng = np.random.default_rng(seed)
    ctx = np.asarray(context_lens, dtype=np.int64)
    ql = np.asarray(query_lens, dtype=np.int64)
    if ctx.shape != ql.shape:
        raise ValueError("context_lens and query_lens differ in length")
    if (ctx < 0).any() or (ql < 0).any():
        raise ValueError("lengths must be non-negative")
    if num_heads % num_kv_heads:
        raise ValueError("num_heads must be a multiple of num_kv_heads")
    B = int(ctx.shape[0])
    L = ctx + ql
    bs = block_size
    H, Hkv, D = num_heads, num_kv_heads, head_dim
    shared = sorted(set(int(b) for b in shared_prefix_requests))
    S = int(shared_prefix_blocks) if shared else 0
    for b in shared:
        if ctx[b] < S * bs:
            raise ValueError("a shared-prefix request must have its context cover the shared blocks")

    per_req_blocks = [blocks_needed(int(x), bs) for x in L]
    private_need = sum(n - (S if b in shared else 0) for b, n in enumerate(per_req_blocks))
    need = private_need + S
    if num_blocks is None:
        num_blocks = max(need, int(math.ceil(need * (1.0 + slack))))
    if num_blocks < need:
        raise ValueError(f"pool of {num_blocks} blocks cannot hold {need}")
    pool = rng.permutation(num_blocks).astype(np.int32)
    shared_ids = pool[:S].copy()
    cursor = S

    max_blocks = max([1] + per_req_blocks) + extra_table_cols
    tables = np.full((B, max_blocks), TABLE_JUNK, dtype=np.int32)
    # junk beyond each request's blocks: a mix of INT32_MIN and random ids
    junk = rng.integers(-(2**31), 2**31 - 1, size=tables.shape, dtype=np.int64).astype(np.int32)
    tables[:, 1::2] = junk[:, 1::2]
    for b in range(B):
        n = per_req_blocks[b]
        first = 0
        if b in shared:
            tables[b, :S] = shared_ids
            first = S
        take = n - first
        tables[b, first:n] = pool[cursor:cursor + take]
        cursor += take

    if fp8:
        kc = np.full((num_blocks, bs, Hkv, D), FP8_NAN, dtype=np.uint8)
        vc = np.full((num_blocks, bs, Hkv, D), FP8_NAN, dtype=np.uint8)
    else:
        kc = np.full((num_blocks, bs, Hkv, D), NAN_BITS[dtype], dtype=np.uint16)
        vc = np.full((num_blocks, bs, Hkv, D), NAN_BITS[dtype], dtype=np.uint16)
    kflat = kc.reshape(num_blocks * bs, Hkv, D)
    vflat = vc.reshape(num_blocks * bs, Hkv, D)

    def history(n):
        return fp8_codes(rng, (n, Hkv, D)) if fp8 else _normal_elems(rng, (n, Hkv, D), dtype=dtype)

    # History rows (positions < context). Shared-prefix rows are written once.
    prefix_written = False
    for b in range(B):
        c = int(ctx[b])
        start = 0
        if b in shared:
            if not prefix_written:
                pos = np.arange(S * bs)
                slots = tables[b, pos // bs].astype(np.int64) * bs + pos % bs
                kflat[slots] = history(pos.size)
                vflat[slots] = history(pos.size)
                prefix_written = True
            start = S * bs
        if c > start:
            pos = np.arange(start, c)
            slots = tables[b, pos // bs].astype(np.int64) * bs + pos % bs
            kflat[slots] = history(pos.size)
            vflat[slots] = history(pos.size)

    # This step's tokens: query rows and the new K/V rows with their slots.
    T = int(ql.sum())
    qsl = np.zeros(B + 1, dtype=np.int32)
    qsl[1:] = np.cumsum(ql)
    q = _normal_elems(rng, (T, H, D), scale=q_scale, dtype=dtype)
    key = _normal_elems(rng, (T, Hkv, D), dtype=dtype)
    value = _normal_elems(rng, (T, Hkv, D), dtype=dtype)
    slot_mapping = np.empty(T, dtype=np.int64)
    for b in range(B):
        pos = np.arange(int(ctx[b]), int(L[b]))
        slot_mapping[qsl[b]:qsl[b + 1]] = tables[b, pos // bs].astype(np.int64) * bs + pos % bs

    return Workload(
        name=name, seed=seed, num_heads=H, num_kv_heads=Hkv, head_dim=D,
        block_size=bs, num_blocks=int(num_blocks),
        scale=float(np.float32(1.0 / math.sqrt(D))) if scale is None else float(np.float32(scale)),
        q=q, key=key, value=value, slot_mapping=slot_mapping,
        key_cache=kc, value_cache=vc, block_tables=tables,
        seq_lens=L.astype(np.int32), query_start_loc=qsl,
        shared_blocks=shared_ids if S else None, dtype=dtype,
        meta={"context_lens": ctx.astype(np.int32)},
        kv_dtype=FP8_E4M3 if fp8 else "",
        k_scale=float(np.float32(k_scale)) if fp8 else 1.0,
        v_scale=float(np.float32(v_scale)) if fp8 else 1.0,
    )


# --------------------------------------------------------------------------
# The five named workloads (sizes from the paged-attention step being built:
# 7B/8B-class head counts, 16-token blocks, variable lengths).
# --------------------------------------------------------------------------

def tiny_decode(seed: int = 0, dtype: str = "bf16", kv_dtype: str = "") -> Workload:
    """4 requests with seq_lens {1, 7, 16, 33}, one new token each; H=4, Hkv=1,
    D=64, 32 physical blocks in a seeded random order."""
    L = np.array([1, 7, 16, 33])
    return make_workload("tiny_decode", context_lens=L - 1, query_lens=[1] * 4,
                         num_heads=4, num_kv_heads=1, head_dim=64, num_blocks=32, seed=seed, dtype=dtype,
                         kv_dtype=kv_dtype)


def mha_decode(seed: int = 0, batch: int = 64, dtype: str = "bf16", block_size: int = 16,
               kv_dtype: str = "") -> Workload:
    """MHA 7B-like decode layer: H=Hkv=32, D=128, seq_lens ~ U[128, 2048]."""
    rng = np.random.default_rng(seed + 1000)
    L = rng.integers(128, 2048, size=batch, endpoint=True)
    return make_workload("mha_decode", context_lens=L - 1, query_lens=[1] * batch,
                         num_heads=32, num_kv_heads=32, head_dim=128, seed=seed, dtype=dtype, block_size=block_size,
                         kv_dtype=kv_dtype)


def gqa_seq_lens(seed: int, batch: int) -> np.ndarray:
    """Lognormal sequence lengths, median 1024, sigma 1.0, clipped to [16, 8192]."""
    rng = np.random.default_rng(seed + 2000)
    x = np.exp(rng.normal(math.log(1024.0), 1.0, size=batch))
    return np.clip(np.rint(x), 16, 8192).astype(np.int64)


def gqa_decode(seed: int = 0, batch: int = 256, dtype: str = "bf16", block_size: int = 16,
               kv_dtype: str = "") -> Workload:
    """GQA 8B-like decode layer: batch 256, H=32, Hkv=8, D=128, lognormal lengths."""
    L = gqa_seq_lens(seed, batch)
    w = make_workload("gqa_decode", context_lens=L - 1, query_lens=[1] * batch,
                      num_heads=32, num_kv_heads=8, head_dim=128, seed=seed, dtype=dtype, block_size=block_size,
                      kv_dtype=kv_dtype)
    w.meta["lognormal_sigma"] = 1.0
    return w


def long_decode(seed: int = 0, batch: int = 8, seq_len: int = 32768, dtype: str = "bf16",
                block_size: int = 16, kv_dtype: str = "") -> Workload:
    """Long-context decode: 8 requests of 32768 tokens, H=64, Hkv=8, D=128."""
    return make_workload("long_decode", context_lens=[seq_len - 1] * batch, query_lens=[1] * batch,
                         num_heads=64, num_kv_heads=8, head_dim=128, seed=seed, dtype=dtype,
                         block_size=block_size, kv_dtype=kv_dtype)


def mixed_step(seed: int = 0, n_prefill: int = 16, chunk: int = 512, n_decode: int = 240,
               n_shared: int = 64, shared_blocks: int = 64, batch: Optional[int] = None,
               dtype: str = "bf16", block_size: int = 16, kv_dtype: str = "") -> Workload:
    """Continuous-batching step: 16 prefill chunks of 512 query tokens (prior
    context U[0, 4096]) plus 240 decode requests (context U[256, 4096]); the
    first 64 physical blocks of 64 decode requests are one shared prefix.
    Requests appear in a seeded random order. `batch` scales the step down
    (batch / 16 prefill chunks, the rest decode, a quarter of those sharing)."""
    if batch is not None:
        n_prefill = max(1, batch // 16)
        n_decode = batch - n_prefill
        n_shared = n_decode // 4
    rng = np.random.default_rng(seed + 3000)
    pre_ctx = rng.integers(0, 4096, size=n_prefill, endpoint=True)
    dec_ctx = rng.integers(256, 4096, size=n_decode, endpoint=True)
    lo = shared_blocks * block_size + 1
    dec_ctx[:n_shared] = rng.integers(lo, 4096, size=n_shared, endpoint=True)
    ctx = np.concatenate([pre_ctx, dec_ctx])
    ql = np.concatenate([np.full(n_prefill, chunk), np.ones(n_decode, dtype=np.int64)])
    is_shared = np.zeros(ctx.size, dtype=bool)
    is_shared[n_prefill:n_prefill + n_shared] = True
    order = rng.permutation(ctx.size)
    ctx, ql, is_shared = ctx[order], ql[order], is_shared[order]
    w = make_workload("mixed_step", context_lens=ctx, query_lens=ql,
                      num_heads=32, num_kv_heads=8, head_dim=128, seed=seed,
                      shared_prefix_requests=np.nonzero(is_shared)[0].tolist(),
                      shared_prefix_blocks=shared_blocks, dtype=dtype, block_size=block_size,
                      kv_dtype=kv_dtype)
    return w


NAMED = {
    "tiny_decode": tiny_decode,
    "mha_decode": mha_decode,
    "gqa_decode": gqa_decode,
    "long_decode": long_decode,
    "mixed_step": mixed_step,
}


def by_name(name: str, seed: int = 0, **kw) -> Workload:
    if name not in NAMED:
        raise KeyError(f"unknown workload {name!r}; known: {sorted(NAMED)}")
    return NAMED[name](seed=seed, **kw)
