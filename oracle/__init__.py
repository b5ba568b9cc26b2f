"""ctypes wrapper around the fp64 CPU oracle (``oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg use it. The CUDA library never imports it.

``build()`` compiles ``liboracle.so`` next to the source with the system C
compiler; ``Oracle`` loads a built library (the tests also load deliberately
broken copies to show that the pins catch planted mistakes).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "oracle.c")
LIBRARY = os.path.join(HERE, "liboracle.so")

ERRORS = {
    0: "ok",
    -1: "bad argument",
    -2: "slot out of range",
    -3: "duplicate slot or destination block",
    -4: "block id out of range",
    -5: "inconsistent lengths",
    -6: "out of memory",
}


# element types of q, the caches and out (the oracle's ORACLE_BF16 / ORACLE_FP16)
DTYPES = {"bf16": 0, "fp16": 1}


class OracleError(RuntimeError):
    pass


def compile_oracle(source: str = SOURCE, output: str = LIBRARY) -> str:
    """Compile the oracle into a shared library. Contraction of a*b+c into a
    fused multiply-add is switched off so both host architectures round alike."""
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
           source, "-o", output, "-lm"]
    subprocess.run(cmd, check=True)
    return output


def build(force: bool = False) -> str:
    if force or not os.path.exists(LIBRARY) or os.path.getmtime(LIBRARY) < os.path.getmtime(SOURCE):
        compile_oracle()
    return LIBRARY


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


class Oracle:
    def __init__(self, lib_path: Optional[str] = None):
        if lib_path is None:
            lib_path = build()
        self.lib = ctypes.CDLL(lib_path)
        L = self.lib
        L.oracle_reshape_and_cache.argtypes = [_P, _P, _P, _P, _P, _I64, _I32, _I32, _I32, _I64]
        L.oracle_reshape_and_cache.restype = ctypes.c_int
        common = [_P, _P, _P, _P, _I32, _P, _P, _I32, _I32, _I32, _I32, _I32, _I64, ctypes.c_float, _I32]
        L.oracle_attention_varlen.argtypes = common + [_P, _I32]
        L.oracle_attention_varlen.restype = ctypes.c_int
        L.oracle_attention_sampled.argtypes = common + [_I64, _P, _P, _P]
        L.oracle_attention_sampled.restype = ctypes.c_int
        L.oracle_attention_weights.argtypes = common + [_I64, _I32, _P]
        L.oracle_attention_weights.restype = ctypes.c_int
        L.oracle_copy_blocks.argtypes = [_P, _P, _P, _I64, _I64, _I64]
        L.oracle_copy_blocks.restype = ctypes.c_int
        L.oracle_round_elements.argtypes = [_P, _I64, _I32, _P]
        L.oracle_round_elements.restype = ctypes.c_int
        L.oracle_rope_reshape_and_cache.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _I32, _I32, _I32, _I64, _I32,
                                                    _I32, _I32, _I32, _I64, _I32]
        L.oracle_rope_reshape_and_cache.restype = ctypes.c_int
        L.oracle_decode_elements.argtypes = [_P, _I64, _I32, _P]
        L.oracle_decode_elements.restype = ctypes.c_int

    @staticmethod
    def _check(rc: int, what: str) -> None:
        if rc < 0:
            raise OracleError(f"{what}: {ERRORS.get(rc, rc)}")

    def reshape_and_cache(self, key, value, key_cache, value_cache, slot_mapping, block_size):
        """Scatter in place into ``key_cache`` / ``value_cache`` (uint16 arrays)."""
        key = np.ascontiguousarray(key, dtype=np.uint16)
        value = np.ascontiguousarray(value, dtype=np.uint16)
        slot_mapping = np.ascontiguousarray(slot_mapping, dtype=np.int64)
        assert key_cache.flags.c_contiguous and value_cache.flags.c_contiguous
        assert key_cache.dtype == np.uint16 and value_cache.dtype == np.uint16
        nb, bs, hkv, d = key_cache.shape
        assert bs == block_size
        rc = self.lib.oracle_reshape_and_cache(_ptr(key), _ptr(value), _ptr(key_cache), _ptr(value_cache),
                                               _ptr(slot_mapping), int(slot_mapping.shape[0]),
                                               hkv, d, bs, nb)
        self._check(rc, "reshape_and_cache")

    def copy_blocks(self, key_cache, value_cache, block_mapping) -> None:
        """Copy-on-write block copy in place on ``key_cache`` / ``value_cache`` (uint16
        [num_blocks, bs, Hkv, D]); ``block_mapping`` int64 [n, 2] = (source, destination)."""
        assert key_cache.flags.c_contiguous and value_cache.flags.c_contiguous
        assert key_cache.dtype == np.uint16 and value_cache.dtype == np.uint16
        m = np.ascontiguousarray(block_mapping, dtype=np.int64).reshape(-1, 2)
        nb = key_cache.shape[0]
        block_elems = int(np.prod(key_cache.shape[1:]))
        rc = self.lib.oracle_copy_blocks(_ptr(key_cache), _ptr(value_cache), _ptr(m), int(m.shape[0]),
                                         block_elems, nb)
        self._check(rc, "copy_blocks")

    def round_elements(self, x, dtype: str = "bf16") -> np.ndarray:
        """The oracle's round-to-nearest-even of float64 values to 16-bit element bits."""
        x = np.ascontiguousarray(x, dtype=np.float64)
        out = np.zeros(x.shape, dtype=np.uint16)
        rc = self.lib.oracle_round_elements(_ptr(x), int(x.size), DTYPES[dtype], _ptr(out))
        self._check(rc, "round_elements")
        return out

    def rope_reshape_and_cache(self, q, key, value, key_cache, value_cache, slot_mapping, positions,
                               cos_sin_cache, is_neox: bool, block_size: int, dtype: str = "bf16"):
        """Rotate ``q`` in place (uint16 [T, H, D]); write the rotated key and the value rows
        into the caches in place. cos_sin_cache: float32 [max_position, rotary_dim]."""
        assert q.flags.c_contiguous and q.dtype == np.uint16
        assert key_cache.flags.c_contiguous and value_cache.flags.c_contiguous
        key = np.ascontiguousarray(key, dtype=np.uint16)
        value = np.ascontiguousarray(value, dtype=np.uint16)
        slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
        pos = np.ascontiguousarray(positions, dtype=np.int64)
        cs = np.ascontiguousarray(cos_sin_cache, dtype=np.float32)
        T, H, D = q.shape
        nb, bs, hkv, d = key_cache.shape
        assert bs == block_size and d == D
        rc = self.lib.oracle_rope_reshape_and_cache(
            _ptr(q), _ptr(key), _ptr(value), _ptr(key_cache), _ptr(value_cache), _ptr(slots), _ptr(pos), _ptr(cs),
            int(cs.shape[0]), int(cs.shape[1]), int(bool(is_neox)), T, H, hkv, D, bs, nb, DTYPES[dtype])
        self._check(rc, "rope_reshape_and_cache")

    def decode_elements(self, bits, dtype: str = "bf16") -> np.ndarray:
        """The oracle's widening of 16-bit element bit patterns to float64."""
        bits = np.ascontiguousarray(bits, dtype=np.uint16)
        out = np.zeros(bits.shape, dtype=np.float64)
        rc = self.lib.oracle_decode_elements(_ptr(bits), int(bits.size), DTYPES[dtype], _ptr(out))
        self._check(rc, "decode_elements")
        return out

    def _common(self, q, key_cache, value_cache, block_tables, seq_lens, query_start_loc,
                num_heads, scale, dtype):
        q = np.ascontiguousarray(q, dtype=np.uint16)
        kc = np.ascontiguousarray(key_cache, dtype=np.uint16)
        vc = np.ascontiguousarray(value_cache, dtype=np.uint16)
        bt = np.ascontiguousarray(block_tables, dtype=np.int32)
        sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
        qsl = np.ascontiguousarray(query_start_loc, dtype=np.int32)
        nb, bs, hkv, d = kc.shape
        keep = (q, kc, vc, bt, sl, qsl)
        args = [_ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), int(bt.shape[1]), _ptr(sl), _ptr(qsl),
                int(sl.shape[0]), int(num_heads), hkv, d, bs, nb, float(scale), DTYPES[dtype]]
        return keep, args, d

    def attention(self, q, key_cache, value_cache, block_tables, seq_lens, query_start_loc,
                  num_heads, scale, num_threads: int = 0, dtype: str = "bf16") -> np.ndarray:
        """fp64 output [total_q, num_heads, head_dim]; elements decode as ``dtype``."""
        keep, args, d = self._common(q, key_cache, value_cache, block_tables, seq_lens,
                                     query_start_loc, num_heads, scale, dtype)
        total_q = int(keep[5][-1])
        out = np.zeros((total_q, num_heads, d), dtype=np.float64)
        if num_threads <= 0:
            num_threads = os.cpu_count() or 1
        rc = self.lib.oracle_attention_varlen(*args, _ptr(out), int(num_threads))
        self._check(rc, "attention")
        return out

    def attention_sampled(self, q, key_cache, value_cache, block_tables, seq_lens, query_start_loc,
                          num_heads, scale, tokens, heads, dtype: str = "bf16") -> np.ndarray:
        """fp64 output [n_samples, head_dim] for the given (token, head) pairs."""
        keep, args, d = self._common(q, key_cache, value_cache, block_tables, seq_lens,
                                     query_start_loc, num_heads, scale, dtype)
        tokens = np.ascontiguousarray(tokens, dtype=np.int64)
        heads = np.ascontiguousarray(heads, dtype=np.int32)
        out = np.zeros((tokens.shape[0], d), dtype=np.float64)
        rc = self.lib.oracle_attention_sampled(*args, int(tokens.shape[0]), _ptr(tokens), _ptr(heads),
                                               _ptr(out))
        self._check(rc, "attention_sampled")
        return out

    def attention_weights(self, q, key_cache, value_cache, block_tables, seq_lens, query_start_loc,
                          num_heads, scale, token, head, dtype: str = "bf16") -> np.ndarray:
        """Softmax weights of one (token, head) pair over its visible keys."""
        keep, args, d = self._common(q, key_cache, value_cache, block_tables, seq_lens,
                                     query_start_loc, num_heads, scale, dtype)
        w = np.zeros(int(keep[4].max()) + 1, dtype=np.float64)
        n = self.lib.oracle_attention_weights(*args, int(token), int(head), _ptr(w))
        self._check(n, "attention_weights")
        return w[:n].copy()

    # convenience: a whole Workload (from paged_kv_cache_55_gb300.workloads)
    def run_step(self, w, num_threads: int = 0):
        """Apply the step to host copies: returns (key_cache, value_cache, out)."""
        kc = w.key_cache.copy()
        vc = w.value_cache.copy()
        self.reshape_and_cache(w.key, w.value, kc, vc, w.slot_mapping, w.block_size)
        out = self.attention(w.q, kc, vc, w.block_tables, w.seq_lens, w.query_start_loc,
                             w.num_heads, w.scale, num_threads=num_threads, dtype=w.dtype)
        return kc, vc, out


_default: Optional[Oracle] = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default
