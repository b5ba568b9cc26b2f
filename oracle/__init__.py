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
# 8-bit cache codes (ORACLE_FP8_E4M3): caches of uint8, one float scale per cache
FP8_E4M3 = "fp8_e4m3"
KV_CODES = {"bf16": 0, "fp16": 1, FP8_E4M3: 2}


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
        common = [_P, _P, _P, _P, _I32, _P, _P, _I32, _I32, _I32, _I32, _I32, _I64, ctypes.c_float, _I32,
                  _I32, ctypes.c_float, ctypes.c_float]
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
        L.oracle_fp8_decode.argtypes = [_P, _I64, _P]
        L.oracle_fp8_decode.restype = ctypes.c_int
        L.oracle_fp8_round.argtypes = [_P, _I64, _P]
        L.oracle_fp8_round.restype = ctypes.c_int
        L.oracle_fp8_quantize.argtypes = [_P, _I64, _I32, ctypes.c_float, _P]
        L.oracle_fp8_quantize.restype = ctypes.c_int
        L.oracle_reshape_and_cache_fp8.argtypes = [_P, _P, _P, _P, _P, _I64, _I32, _I32, _I32, _I64, _I32,
                                                   ctypes.c_float, ctypes.c_float]
        L.oracle_reshape_and_cache_fp8.restype = ctypes.c_int
        L.oracle_rope_reshape_and_cache_fp8.argtypes = L.oracle_rope_reshape_and_cache.argtypes + [ctypes.c_float,
                                                                                                   ctypes.c_float]
        L.oracle_rope_reshape_and_cache_fp8.restype = ctypes.c_int

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
        """Copy-on-write block copy in place on ``key_cache`` / ``value_cache`` (uint16, or
        uint8 codes, [num_blocks, bs, Hkv, D]); ``block_mapping`` int64 [n, 2] = (source, destination)."""
        assert key_cache.flags.c_contiguous and value_cache.flags.c_contiguous
        assert key_cache.dtype == value_cache.dtype and key_cache.dtype in (np.uint16, np.uint8)
        m = np.ascontiguousarray(block_mapping, dtype=np.int64).reshape(-1, 2)
        nb = key_cache.shape[0]
        block_elems = int(np.prod(key_cache.shape[1:]))
        if key_cache.dtype == np.uint8:  # 8-bit codes: the same raw copy, two codes per 16-bit unit
            assert block_elems % 2 == 0
            block_elems //= 2
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

    def rope_reshape_and_cache_fp8(self, q, key, value, key_cache, value_cache, slot_mapping, positions,
                                   cos_sin_cache, is_neox: bool, block_size: int, k_scale: float, v_scale: float,
                                   dtype: str = "bf16"):
        """As rope_reshape_and_cache into 8-bit caches (uint8): the rotated key and the value rows
        are stored as E4M3 codes of x / k_scale and x / v_scale."""
        assert q.flags.c_contiguous and q.dtype == np.uint16
        assert key_cache.flags.c_contiguous and value_cache.flags.c_contiguous
        assert key_cache.dtype == np.uint8 and value_cache.dtype == np.uint8
        key = np.ascontiguousarray(key, dtype=np.uint16)
        value = np.ascontiguousarray(value, dtype=np.uint16)
        slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
        pos = np.ascontiguousarray(positions, dtype=np.int64)
        cs = np.ascontiguousarray(cos_sin_cache, dtype=np.float32)
        T, H, D = q.shape
        nb, bs, hkv, d = key_cache.shape
        assert bs == block_size and d == D
        rc = self.lib.oracle_rope_reshape_and_cache_fp8(
            _ptr(q), _ptr(key), _ptr(value), _ptr(key_cache), _ptr(value_cache), _ptr(slots), _ptr(pos), _ptr(cs),
            int(cs.shape[0]), int(cs.shape[1]), int(bool(is_neox)), T, H, hkv, D, bs, nb, DTYPES[dtype],
            float(k_scale), float(v_scale))
        self._check(rc, "rope_reshape_and_cache_fp8")

    def decode_elements(self, bits, dtype: str = "bf16") -> np.ndarray:
        """The oracle's widening of 16-bit element bit patterns to float64."""
        bits = np.ascontiguousarray(bits, dtype=np.uint16)
        out = np.zeros(bits.shape, dtype=np.float64)
        rc = self.lib.oracle_decode_elements(_ptr(bits), int(bits.size), DTYPES[dtype], _ptr(out))
        self._check(rc, "decode_elements")
        return out

    def fp8_decode(self, codes) -> np.ndarray:
        """The oracle's E4M3 decoding of 8-bit codes to float64."""
        codes = np.ascontiguousarray(codes, dtype=np.uint8)
        out = np.zeros(codes.shape, dtype=np.float64)
        self._check(self.lib.oracle_fp8_decode(_ptr(codes), int(codes.size), _ptr(out)), "fp8_decode")
        return out

    def fp8_round(self, x) -> np.ndarray:
        """The oracle's rounding of float64 values to E4M3 codes (ties to even, saturating)."""
        x = np.ascontiguousarray(x, dtype=np.float64)
        out = np.zeros(x.shape, dtype=np.uint8)
        self._check(self.lib.oracle_fp8_round(_ptr(x), int(x.size), _ptr(out)), "fp8_round")
        return out

    def fp8_quantize(self, bits, scale: float, dtype: str = "bf16") -> np.ndarray:
        """Codes of 16-bit elements: E4M3(binary32(x / scale))."""
        bits = np.ascontiguousarray(bits, dtype=np.uint16)
        out = np.zeros(bits.shape, dtype=np.uint8)
        rc = self.lib.oracle_fp8_quantize(_ptr(bits), int(bits.size), DTYPES[dtype], float(scale), _ptr(out))
        self._check(rc, "fp8_quantize")
        return out

    def reshape_and_cache_fp8(self, key, value, key_cache, value_cache, slot_mapping, block_size,
                              k_scale: float, v_scale: float, dtype: str = "bf16"):
        """Quantising scatter in place into 8-bit ``key_cache`` / ``value_cache`` (uint8 arrays)."""
        key = np.ascontiguousarray(key, dtype=np.uint16)
        value = np.ascontiguousarray(value, dtype=np.uint16)
        slot_mapping = np.ascontiguousarray(slot_mapping, dtype=np.int64)
        assert key_cache.flags.c_contiguous and value_cache.flags.c_contiguous
        assert key_cache.dtype == np.uint8 and value_cache.dtype == np.uint8
        nb, bs, hkv, d = key_cache.shape
        assert bs == block_size
        rc = self.lib.oracle_reshape_and_cache_fp8(_ptr(key), _ptr(value), _ptr(key_cache), _ptr(value_cache),
                                                   _ptr(slot_mapping), int(slot_mapping.shape[0]), hkv, d, bs, nb,
                                                   DTYPES[dtype], float(k_scale), float(v_scale))
        self._check(rc, "reshape_and_cache_fp8")

    def _common(self, q, key_cache, value_cache, block_tables, seq_lens, query_start_loc,
                num_heads, scale, dtype, k_scale=1.0, v_scale=1.0):
        q = np.ascontiguousarray(q, dtype=np.uint16)
        # 8-bit caches hold E4M3 codes; 16-bit caches hold elements of q's type
        kv_fp8 = np.asarray(key_cache).dtype == np.uint8
        cache_t = np.uint8 if kv_fp8 else np.uint16
        kc = np.ascontiguousarray(key_cache, dtype=cache_t)
        vc = np.ascontiguousarray(value_cache, dtype=cache_t)
        bt = np.ascontiguousarray(block_tables, dtype=np.int32)
        sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
        qsl = np.ascontiguousarray(query_start_loc, dtype=np.int32)
        nb, bs, hkv, d = kc.shape
        keep = (q, kc, vc, bt, sl, qsl)
        args = [_ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), int(bt.shape[1]), _ptr(sl), _ptr(qsl),
                int(sl.shape[0]), int(num_heads), hkv, d, bs, nb, float(scale), DTYPES[dtype],
                KV_CODES[FP8_E4M3] if kv_fp8 else DTYPES[dtype], float(k_scale), float(v_scale)]
        return keep, args, d

    def attention(self, q, key_cache, value_cache, block_tables, seq_lens, query_start_loc,
                  num_heads, scale, num_threads: int = 0, dtype: str = "bf16",
                  k_scale: float = 1.0, v_scale: float = 1.0) -> np.ndarray:
        """fp64 output [total_q, num_heads, head_dim]; elements decode as ``dtype``; uint8
        caches hold E4M3 codes whose values are code * k_scale (K) and code * v_scale (V)."""
        keep, args, d = self._common(q, key_cache, value_cache, block_tables, seq_lens,
                                     query_start_loc, num_heads, scale, dtype, k_scale, v_scale)
        total_q = int(keep[5][-1])
        out = np.zeros((total_q, num_heads, d), dtype=np.float64)
        if num_threads <= 0:
            num_threads = os.cpu_count() or 1
        rc = self.lib.oracle_attention_varlen(*args, _ptr(out), int(num_threads))
        self._check(rc, "attention")
        return out

    def attention_sampled(self, q, key_cache, value_cache, block_tables, seq_lens, query_start_loc,
                          num_heads, scale, tokens, heads, dtype: str = "bf16",
                          k_scale: float = 1.0, v_scale: float = 1.0) -> np.ndarray:
        """fp64 output [n_samples, head_dim] for the given (token, head) pairs."""
        keep, args, d = self._common(q, key_cache, value_cache, block_tables, seq_lens,
                                     query_start_loc, num_heads, scale, dtype, k_scale, v_scale)
        tokens = np.ascontiguousarray(tokens, dtype=np.int64)
        heads = np.ascontiguousarray(heads, dtype=np.int32)
        out = np.zeros((tokens.shape[0], d), dtype=np.float64)
        rc = self.lib.oracle_attention_sampled(*args, int(tokens.shape[0]), _ptr(tokens), _ptr(heads),
                                               _ptr(out))
        self._check(rc, "attention_sampled")
        return out

    def attention_weights(self, q, key_cache, value_cache, block_tables, seq_lens, query_start_loc,
                          num_heads, scale, token, head, dtype: str = "bf16",
                          k_scale: float = 1.0, v_scale: float = 1.0) -> np.ndarray:
        """Softmax weights of one (token, head) pair over its visible keys."""
        keep, args, d = self._common(q, key_cache, value_cache, block_tables, seq_lens,
                                     query_start_loc, num_heads, scale, dtype, k_scale, v_scale)
        w = np.zeros(int(keep[4].max()) + 1, dtype=np.float64)
        n = self.lib.oracle_attention_weights(*args, int(token), int(head), _ptr(w))
        self._check(n, "attention_weights")
        return w[:n].copy()

    # convenience: a whole Workload (from paged_kv_cache_55_gb300.workloads)
    def run_step(self, w, num_threads: int = 0):
        """Apply the step to host copies: returns (key_cache, value_cache, out)."""
        kc = w.key_cache.copy()
        vc = w.value_cache.copy()
        if getattr(w, "kv_dtype", w.dtype) == FP8_E4M3:
            self.reshape_and_cache_fp8(w.key, w.value, kc, vc, w.slot_mapping, w.block_size,
                                       w.k_scale, w.v_scale, dtype=w.dtype)
            out = self.attention(w.q, kc, vc, w.block_tables, w.seq_lens, w.query_start_loc, w.num_heads,
                                 w.scale, num_threads=num_threads, dtype=w.dtype, k_scale=w.k_scale,
                                 v_scale=w.v_scale)
            return kc, vc, out
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
