"""Thin ctypes binding of libpagedattn.so with the C ABI's names.

Argument marshalling only: torch tensors become device pointers, shapes become
sizes, the current torch stream becomes the ``stream`` argument. Every step of
the computation runs in the library's CUDA kernels; there is no fallback. If
the library has not been built, importing the functions raises.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIBRARY = os.path.join(HERE, "libpagedattn.so")

PA_BF16, PA_FP16, PA_FP8_E4M3 = 0, 1, 2
_ELEM_CODES = {torch.bfloat16: PA_BF16, torch.float16: PA_FP16}
# 8-bit caches are uint8 tensors of E4M3 codes
_CACHE_CODES = {torch.bfloat16: PA_BF16, torch.float16: PA_FP16, torch.uint8: PA_FP8_E4M3}
STATUS = {
    0: "PA_OK", -1: "PA_ERR_NULL", -2: "PA_ERR_DIMS", -3: "PA_ERR_UNSUPPORTED", -4: "PA_ERR_ALIGN",
    -5: "PA_ERR_WORKSPACE", -6: "PA_ERR_LAUNCH", -7: "PA_ERR_DEVICE_BOUNDS", -8: "PA_ERR_CUDA",
}
FLAG_SLOT_RANGE, FLAG_BLOCK_RANGE, FLAG_LENGTHS, FLAG_QUERY_LOC, FLAG_TIMEOUT = 1, 2, 4, 8, 16
FLAG_POSITION_RANGE = 32


class PagedAttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)} ({_lib().pa_status_string(status).decode()})")


_LIB: Optional[ctypes.CDLL] = None

_P, _I32, _I64, _SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t

SIGNATURES = {
    "pa_reshape_and_cache": ([_P, _P, _I64, _I64, _P, _P, _P, _I32, _I32, _I32, _I32, _I64, _I32, _P], ctypes.c_int),
    "pa_attention_workspace_size": ([_I32, _I32, _I32, _I32, _I32, _I32, _I32, _I32], _SZ),
    "pa_attention_plan_info": ([_I32, _I32, _I32, _I32, _P, _P], ctypes.c_int),
    "pa_attention_varlen": ([_P, _I64, _P, _P, _P, _I32, _P, _P, _I32, _I32, _I32, _I32, _I32, _I32, _I32,
                             _I32, _I64, ctypes.c_float, _P, _P, _SZ, _I32, _P], ctypes.c_int),
    "pa_gather_kv": ([_P, _P, _P, _I32, _I32, _I32, _I32, _I64, _P, _P, _I32, _P], ctypes.c_int),
    "pa_status_string": ([_I32], ctypes.c_char_p),
    "pa_debug_status": ([_P, _P], ctypes.c_int),
    "pa_launch_count": ([], ctypes.c_uint64),
    "pa_last_cuda_error": ([], ctypes.c_char_p),
    "pa_copy_blocks": ([_P, _P, _P, _I32, _I32, _I32, _I32, _I64, _I32, _P], ctypes.c_int32),
    "pa_rope_reshape_and_cache": ([_P, _I64, _P, _P, _I64, _I64, _P, _P, _P, _P, _P, _I32, _I32, _I32, _I32, _I32,
                                   _I32, _I32, _I32, _I64, _I32, _P], ctypes.c_int32),
    "pa_attention_set_timing_events": ([_P, _P], ctypes.c_int),
    "pa_attention_set_tile_timing_events": ([_P, _P], ctypes.c_int),
    "pa_attention_varlen_static": ([_P, _I64, _P, _P, _P, _I32, _P, _P, _I32, _I32, _I32, _I32, _I32, _I32,
                                    _I32, _I32, _I64, ctypes.c_float, _P, _I32, _P], ctypes.c_int),
    "pa_rope_reshape_and_cache_fp8": ([_P, _I64, _P, _P, _I64, _I64, _P, _P, _P, _P, _P, _I32, _I32, _I32, _I32,
                                       _I32, _I32, _I32, _I32, _I64, ctypes.c_float, ctypes.c_float, _I32, _P],
                                      ctypes.c_int32),
    "pa_reshape_and_cache_fp8": ([_P, _P, _I64, _I64, _P, _P, _P, _I32, _I32, _I32, _I32, _I64, ctypes.c_float,
                                  ctypes.c_float, _I32, _P], ctypes.c_int),
    "pa_attention_varlen_fp8": ([_P, _I64, _P, _P, _P, _I32, _P, _P, _I32, _I32, _I32, _I32, _I32, _I32, _I32,
                                 _I32, _I64, ctypes.c_float, ctypes.c_float, ctypes.c_float, _P, _P, _SZ, _I32, _P],
                                ctypes.c_int),
}

# Size of the library's built-in scratch array used by pa_attention_varlen_static.
PA_STATIC_WORKSPACE_BYTES = 32 << 20


def load_library(path: str = LIBRARY) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -m paged_kv_cache_55_gb300.build` "
                           "(the CUDA path has no fallback)")
    lib = ctypes.CDLL(path)
    for name, (args, res) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


def _lib() -> ctypes.CDLL:
    global _LIB
    if _LIB is None:
        _LIB = load_library()
    return _LIB


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(status: int, what: str) -> None:
    if status != 0:
        if status in (-6, -8):  # PA_ERR_LAUNCH, PA_ERR_CUDA: name the CUDA error behind it
            what = f"{what} [{pa_last_cuda_error()}]"
        raise PagedAttnError(status, what)


def _need(t: torch.Tensor, name: str, dtype: torch.dtype) -> None:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


def _elem_code(*named) -> int:
    """The C dtype of element tensors that must share one 16-bit float type (bf16 or fp16)."""
    first = named[0][0]
    if not isinstance(first, torch.Tensor) or first.dtype not in _ELEM_CODES:
        raise TypeError(f"{named[0][1]} must be a bfloat16 or float16 CUDA tensor")
    for t, n in named:
        _need(t, n, first.dtype)
    return _ELEM_CODES[first.dtype]


def _cache_code(*named) -> int:
    """The C dtype of cache tensors that share one type: bf16, fp16, or uint8 (E4M3 codes)."""
    first = named[0][0]
    if not isinstance(first, torch.Tensor) or first.dtype not in _CACHE_CODES:
        raise TypeError(f"{named[0][1]} must be a bfloat16, float16 or uint8 CUDA tensor")
    for t, n in named:
        _need(t, n, first.dtype)
    return _CACHE_CODES[first.dtype]


# Shape checks. The C ABI receives plain pointers, so a tensor of the wrong
# size would be read or written past its end on the device; these checks use
# only .shape and run before any library call.
def _dims(t: torch.Tensor, n: int, name: str) -> None:
    if t.dim() != n:
        raise ValueError(f"{name} must have {n} dimensions, got shape {tuple(t.shape)}")


def _cache_pair_shapes(key_cache: torch.Tensor, value_cache: torch.Tensor) -> None:
    _dims(key_cache, 4, "key_cache")
    if value_cache.shape != key_cache.shape:
        raise ValueError(f"value_cache {tuple(value_cache.shape)} must have key_cache's shape "
                         f"{tuple(key_cache.shape)} [num_blocks, block_size, num_kv_heads, head_dim]")


def _scatter_shapes(key: torch.Tensor, value: torch.Tensor, key_cache: torch.Tensor, value_cache: torch.Tensor,
                    slot_mapping: torch.Tensor) -> None:
    """key/value [T, Hkv, D], caches [NB, bs, Hkv, D], slot_mapping [T]."""
    _dims(key, 3, "key")
    if value.shape != key.shape:
        raise ValueError(f"value {tuple(value.shape)} must have key's shape {tuple(key.shape)}")
    _cache_pair_shapes(key_cache, value_cache)
    if tuple(key_cache.shape[2:]) != tuple(key.shape[1:]):
        raise ValueError(f"cache rows {tuple(key_cache.shape[2:])} must be key's [Hkv, D] {tuple(key.shape[1:])}")
    _dims(slot_mapping, 1, "slot_mapping")
    if slot_mapping.shape[0] != key.shape[0]:
        raise ValueError(f"slot_mapping has {slot_mapping.shape[0]} entries for {key.shape[0]} tokens")


def _attention_shapes(q: torch.Tensor, key_cache: torch.Tensor, value_cache: torch.Tensor,
                      block_tables: torch.Tensor, seq_lens: torch.Tensor, query_start_loc: torch.Tensor,
                      out: torch.Tensor) -> None:
    """q and out [T, H, D], caches [NB, bs, Hkv, D], block_tables [B, M], seq_lens [B], query_start_loc [B+1]."""
    _dims(q, 3, "q")
    if out.shape != q.shape:
        raise ValueError(f"out {tuple(out.shape)} must have q's shape {tuple(q.shape)}")
    _cache_pair_shapes(key_cache, value_cache)
    if key_cache.shape[3] != q.shape[2]:
        raise ValueError(f"head_dim of the caches ({key_cache.shape[3]}) and of q ({q.shape[2]}) differ")
    _dims(seq_lens, 1, "seq_lens")
    _dims(block_tables, 2, "block_tables")
    _dims(query_start_loc, 1, "query_start_loc")
    b = seq_lens.shape[0]
    if block_tables.shape[0] != b or query_start_loc.shape[0] != b + 1:
        raise ValueError(f"{b} requests need block_tables [{b}, M] and query_start_loc [{b + 1}], got "
                         f"{tuple(block_tables.shape)} and {tuple(query_start_loc.shape)}")


def _rope_shapes(q: torch.Tensor, key: torch.Tensor, value: torch.Tensor, key_cache: torch.Tensor,
                 value_cache: torch.Tensor, slot_mapping: torch.Tensor, positions: torch.Tensor,
                 cos_sin_cache: torch.Tensor) -> None:
    """q [T, H, D], key/value [T, Hkv, D], caches [NB, bs, Hkv, D], slot_mapping and positions [T],
    cos_sin_cache [max_position, rotary_dim]."""
    _scatter_shapes(key, value, key_cache, value_cache, slot_mapping)
    _dims(q, 3, "q")
    if q.shape[0] != key.shape[0] or q.shape[2] != key.shape[2]:
        raise ValueError(f"q {tuple(q.shape)} must be [T, H, D] for key {tuple(key.shape)}")
    _dims(positions, 1, "positions")
    if positions.shape[0] != q.shape[0]:
        raise ValueError(f"positions has {positions.shape[0]} entries for {q.shape[0]} tokens")
    _dims(cos_sin_cache, 2, "cos_sin_cache")


def _gather_shapes(key_cache: torch.Tensor, value_cache: torch.Tensor, block_table_row: torch.Tensor, seq_len: int,
                   key_out: torch.Tensor, value_out: torch.Tensor) -> None:
    """caches [NB, bs, Hkv, D], block_table_row [>= ceil(seq_len / bs)], outputs [seq_len, Hkv, D]."""
    _cache_pair_shapes(key_cache, value_cache)
    _dims(block_table_row, 1, "block_table_row")
    bs = key_cache.shape[1]
    if block_table_row.shape[0] * bs < seq_len:
        raise ValueError(f"block_table_row has {block_table_row.shape[0]} blocks of {bs} for {seq_len} tokens")
    want = (seq_len, key_cache.shape[2], key_cache.shape[3])
    if tuple(key_out.shape) != want or tuple(value_out.shape) != want:
        raise ValueError(f"key_out and value_out must be {want}, got {tuple(key_out.shape)} and "
                         f"{tuple(value_out.shape)}")


def _index_tensors(*named) -> None:
    for t, n in named:
        _need(t, n, torch.int32)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")


def _workspace(workspace: torch.Tensor) -> None:
    if not isinstance(workspace, torch.Tensor) or not workspace.is_cuda or not workspace.is_contiguous():
        raise TypeError("workspace must be a contiguous CUDA tensor")


def pa_reshape_and_cache(key: torch.Tensor, value: torch.Tensor, key_cache: torch.Tensor,
                         value_cache: torch.Tensor, slot_mapping: torch.Tensor, stream=None) -> None:
    """key/value [T, Hkv, D] (token stride free), caches [NB, bs, Hkv, D], all bf16 or all fp16;
    slots int64 [T]."""
    dt = _elem_code((key, "key"), (value, "value"), (key_cache, "key_cache"), (value_cache, "value_cache"))
    _need(slot_mapping, "slot_mapping", torch.int64)
    _scatter_shapes(key, value, key_cache, value_cache, slot_mapping)
    T, hkv, d = key.shape
    if key.stride(2) != 1 or key.stride(1) != d or value.stride(2) != 1 or value.stride(1) != d:
        raise ValueError("each token row of key/value must be [Hkv, D] contiguous")
    if not (key_cache.is_contiguous() and value_cache.is_contiguous() and slot_mapping.is_contiguous()):
        raise ValueError("caches and slot_mapping must be contiguous")
    nb, bs = key_cache.shape[0], key_cache.shape[1]
    _check(_lib().pa_reshape_and_cache(key.data_ptr(), value.data_ptr(), key.stride(0), value.stride(0),
                                       key_cache.data_ptr(), value_cache.data_ptr(), slot_mapping.data_ptr(),
                                       T, hkv, d, bs, nb, dt, _stream(stream)), "pa_reshape_and_cache")


def pa_reshape_and_cache_fp8(key: torch.Tensor, value: torch.Tensor, key_cache: torch.Tensor,
                             value_cache: torch.Tensor, slot_mapping: torch.Tensor, k_scale: float, v_scale: float,
                             stream=None) -> None:
    """Quantising scatter: key/value [T, Hkv, D] bf16 or fp16 (token stride free), caches uint8
    [NB, bs, Hkv, D] of E4M3 codes (code = E4M3(x / scale)); slots int64 [T]."""
    dt = _elem_code((key, "key"), (value, "value"))
    _need(key_cache, "key_cache", torch.uint8)
    _need(value_cache, "value_cache", torch.uint8)
    _need(slot_mapping, "slot_mapping", torch.int64)
    _scatter_shapes(key, value, key_cache, value_cache, slot_mapping)
    T, hkv, d = key.shape
    if key.stride(2) != 1 or key.stride(1) != d or value.stride(2) != 1 or value.stride(1) != d:
        raise ValueError("each token row of key/value must be [Hkv, D] contiguous")
    if not (key_cache.is_contiguous() and value_cache.is_contiguous() and slot_mapping.is_contiguous()):
        raise ValueError("caches and slot_mapping must be contiguous")
    nb, bs = key_cache.shape[0], key_cache.shape[1]
    _check(_lib().pa_reshape_and_cache_fp8(key.data_ptr(), value.data_ptr(), key.stride(0), value.stride(0),
                                           key_cache.data_ptr(), value_cache.data_ptr(), slot_mapping.data_ptr(),
                                           T, hkv, d, bs, nb, float(k_scale), float(v_scale), dt,
                                           _stream(stream)), "pa_reshape_and_cache_fp8")


def pa_attention_workspace_size(num_seqs: int, total_q_tokens: int, max_query_len: int, max_seq_len: int,
                                num_heads: int, num_kv_heads: int, head_dim: int, block_size: int = 16) -> int:
    n = _lib().pa_attention_workspace_size(num_seqs, total_q_tokens, max_query_len, max_seq_len, num_heads,
                                           num_kv_heads, head_dim, block_size)
    if n == 0 and num_seqs > 0:
        raise ValueError("invalid sizes for pa_attention_workspace_size")
    return int(n)


def pa_attention_plan_info(num_seqs: int, max_seq_len: int, num_heads: int, num_kv_heads: int):
    pt, mp = ctypes.c_int32(0), ctypes.c_int32(0)
    _check(_lib().pa_attention_plan_info(num_seqs, max_seq_len, num_heads, num_kv_heads,
                                         ctypes.addressof(pt), ctypes.addressof(mp)), "pa_attention_plan_info")
    return int(pt.value), int(mp.value)


def pa_attention_varlen(q: torch.Tensor, key_cache: torch.Tensor, value_cache: torch.Tensor,
                        block_tables: torch.Tensor, seq_lens: torch.Tensor, query_start_loc: torch.Tensor,
                        max_query_len: int, max_seq_len: int, scale: float, out: torch.Tensor,
                        workspace: torch.Tensor, stream=None) -> None:
    """q [T, H, D], caches [NB, bs, Hkv, D], out [T, H, D] contiguous (all bf16 or all fp16),
    block_tables [B, M] int32, seq_lens [B] int32, query_start_loc [B+1] int32, workspace uint8 (device)."""
    dt = _elem_code((q, "q"), (out, "out"), (key_cache, "key_cache"), (value_cache, "value_cache"))
    _index_tensors((block_tables, "block_tables"), (seq_lens, "seq_lens"), (query_start_loc, "query_start_loc"))
    _attention_shapes(q, key_cache, value_cache, block_tables, seq_lens, query_start_loc, out)
    _workspace(workspace)
    if not out.is_contiguous() or not key_cache.is_contiguous() or not value_cache.is_contiguous():
        raise ValueError("out and the caches must be contiguous")
    T, H, D = q.shape
    if q.stride(2) != 1 or q.stride(1) != D:
        raise ValueError("each token row of q must be [H, D] contiguous")
    nb, bs, hkv, _ = key_cache.shape
    B = seq_lens.shape[0]
    _check(_lib().pa_attention_varlen(q.data_ptr(), q.stride(0), key_cache.data_ptr(), value_cache.data_ptr(),
                                      block_tables.data_ptr(), block_tables.shape[1], seq_lens.data_ptr(),
                                      query_start_loc.data_ptr(), B, T, max_query_len, max_seq_len, H, hkv, D, bs,
                                      nb, float(scale), out.data_ptr(), workspace.data_ptr(),
                                      workspace.numel() * workspace.element_size(), dt, _stream(stream)),
           "pa_attention_varlen")


def pa_attention_varlen_fp8(q: torch.Tensor, key_cache: torch.Tensor, value_cache: torch.Tensor,
                            block_tables: torch.Tensor, seq_lens: torch.Tensor, query_start_loc: torch.Tensor,
                            max_query_len: int, max_seq_len: int, scale: float, k_scale: float, v_scale: float,
                            out: torch.Tensor, workspace: torch.Tensor, stream=None) -> None:
    """pa_attention_varlen over 8-bit caches: caches uint8 [NB, bs, Hkv, D] of E4M3 codes whose values
    are code * k_scale and code * v_scale; q and out bf16 or fp16."""
    dt = _elem_code((q, "q"), (out, "out"))
    _need(key_cache, "key_cache", torch.uint8)
    _need(value_cache, "value_cache", torch.uint8)
    _index_tensors((block_tables, "block_tables"), (seq_lens, "seq_lens"), (query_start_loc, "query_start_loc"))
    _attention_shapes(q, key_cache, value_cache, block_tables, seq_lens, query_start_loc, out)
    _workspace(workspace)
    if not out.is_contiguous() or not key_cache.is_contiguous() or not value_cache.is_contiguous():
        raise ValueError("out and the caches must be contiguous")
    T, H, D = q.shape
    if q.stride(2) != 1 or q.stride(1) != D:
        raise ValueError("each token row of q must be [H, D] contiguous")
    nb, bs, hkv, _ = key_cache.shape
    B = seq_lens.shape[0]
    _check(_lib().pa_attention_varlen_fp8(q.data_ptr(), q.stride(0), key_cache.data_ptr(), value_cache.data_ptr(),
                                          block_tables.data_ptr(), block_tables.shape[1], seq_lens.data_ptr(),
                                          query_start_loc.data_ptr(), B, T, max_query_len, max_seq_len, H, hkv, D,
                                          bs, nb, float(scale), float(k_scale), float(v_scale), out.data_ptr(),
                                          workspace.data_ptr(), workspace.numel() * workspace.element_size(), dt,
                                          _stream(stream)), "pa_attention_varlen_fp8")


def pa_attention_varlen_static(q: torch.Tensor, key_cache: torch.Tensor, value_cache: torch.Tensor,
                               block_tables: torch.Tensor, seq_lens: torch.Tensor, query_start_loc: torch.Tensor,
                               max_query_len: int, max_seq_len: int, scale: float, out: torch.Tensor,
                               stream=None) -> None:
    """pa_attention_varlen without a workspace argument, for callers that cannot allocate: the
    library's built-in scratch array (PA_STATIC_WORKSPACE_BYTES) is used instead. Calls on one device
    share that array, so calls on different streams must not overlap."""
    dt = _elem_code((q, "q"), (out, "out"), (key_cache, "key_cache"), (value_cache, "value_cache"))
    _index_tensors((block_tables, "block_tables"), (seq_lens, "seq_lens"), (query_start_loc, "query_start_loc"))
    _attention_shapes(q, key_cache, value_cache, block_tables, seq_lens, query_start_loc, out)
    if not out.is_contiguous() or not key_cache.is_contiguous() or not value_cache.is_contiguous():
        raise ValueError("out and the caches must be contiguous")
    T, H, D = q.shape
    if q.stride(2) != 1 or q.stride(1) != D:
        raise ValueError("each token row of q must be [H, D] contiguous")
    nb, bs, hkv, _ = key_cache.shape
    B = seq_lens.shape[0]
    _check(_lib().pa_attention_varlen_static(q.data_ptr(), q.stride(0), key_cache.data_ptr(),
                                             value_cache.data_ptr(), block_tables.data_ptr(), block_tables.shape[1],
                                             seq_lens.data_ptr(), query_start_loc.data_ptr(), B, T, max_query_len,
                                             max_seq_len, H, hkv, D, bs, nb, float(scale), out.data_ptr(), dt,
                                             _stream(stream)), "pa_attention_varlen_static")


def pa_rope_reshape_and_cache(q: torch.Tensor, key: torch.Tensor, value: torch.Tensor, key_cache: torch.Tensor,
                              value_cache: torch.Tensor, slot_mapping: torch.Tensor, positions: torch.Tensor,
                              cos_sin_cache: torch.Tensor, is_neox: bool = True, stream=None) -> None:
    """Rotate q in place and write the rotated key and the value rows into the caches.
    q [T, H, D], key/value [T, Hkv, D] (token strides free), caches [NB, bs, Hkv, D] (one 16-bit type);
    slot_mapping and positions int64 [T]; cos_sin_cache float32 [max_position, rotary_dim]."""
    dt = _elem_code((q, "q"), (key, "key"), (value, "value"), (key_cache, "key_cache"), (value_cache, "value_cache"))
    _need(slot_mapping, "slot_mapping", torch.int64)
    _need(positions, "positions", torch.int64)
    _need(cos_sin_cache, "cos_sin_cache", torch.float32)
    _rope_shapes(q, key, value, key_cache, value_cache, slot_mapping, positions, cos_sin_cache)
    T, H, D = q.shape
    _, hkv, d = key.shape
    for t, n in ((q, "q"), (key, "key"), (value, "value")):
        if t.stride(2) != 1 or t.stride(1) != D:
            raise ValueError(f"each token row of {n} must be [heads, D] contiguous")
    if not (key_cache.is_contiguous() and value_cache.is_contiguous() and cos_sin_cache.is_contiguous()
            and slot_mapping.is_contiguous() and positions.is_contiguous()):
        raise ValueError("caches, cos_sin_cache, slot_mapping and positions must be contiguous")
    nb, bs = key_cache.shape[0], key_cache.shape[1]
    max_pos, rot = cos_sin_cache.shape
    _check(_lib().pa_rope_reshape_and_cache(q.data_ptr(), q.stride(0), key.data_ptr(), value.data_ptr(),
                                            key.stride(0), value.stride(0), key_cache.data_ptr(),
                                            value_cache.data_ptr(), slot_mapping.data_ptr(), positions.data_ptr(),
                                            cos_sin_cache.data_ptr(), max_pos, rot, int(bool(is_neox)), T, H, hkv, D,
                                            bs, nb, dt, _stream(stream)), "pa_rope_reshape_and_cache")


def pa_rope_reshape_and_cache_fp8(q: torch.Tensor, key: torch.Tensor, value: torch.Tensor,
                                  key_cache: torch.Tensor, value_cache: torch.Tensor, slot_mapping: torch.Tensor,
                                  positions: torch.Tensor, cos_sin_cache: torch.Tensor, k_scale: float,
                                  v_scale: float, is_neox: bool = True, stream=None) -> None:
    """pa_rope_reshape_and_cache into 8-bit caches (uint8 [NB, bs, Hkv, D] of E4M3 codes): the rotated
    key and the value rows are stored as codes of x / k_scale and x / v_scale."""
    dt = _elem_code((q, "q"), (key, "key"), (value, "value"))
    _need(key_cache, "key_cache", torch.uint8)
    _need(value_cache, "value_cache", torch.uint8)
    _need(slot_mapping, "slot_mapping", torch.int64)
    _need(positions, "positions", torch.int64)
    _need(cos_sin_cache, "cos_sin_cache", torch.float32)
    _rope_shapes(q, key, value, key_cache, value_cache, slot_mapping, positions, cos_sin_cache)
    T, H, D = q.shape
    _, hkv, d = key.shape
    for t, n in ((q, "q"), (key, "key"), (value, "value")):
        if t.stride(2) != 1 or t.stride(1) != D:
            raise ValueError(f"each token row of {n} must be [heads, D] contiguous")
    if not (key_cache.is_contiguous() and value_cache.is_contiguous() and cos_sin_cache.is_contiguous()
            and slot_mapping.is_contiguous() and positions.is_contiguous()):
        raise ValueError("caches, cos_sin_cache, slot_mapping and positions must be contiguous")
    nb, bs = key_cache.shape[0], key_cache.shape[1]
    max_pos, rot = cos_sin_cache.shape
    _check(_lib().pa_rope_reshape_and_cache_fp8(q.data_ptr(), q.stride(0), key.data_ptr(), value.data_ptr(),
                                                key.stride(0), value.stride(0), key_cache.data_ptr(),
                                                value_cache.data_ptr(), slot_mapping.data_ptr(), positions.data_ptr(),
                                                cos_sin_cache.data_ptr(), max_pos, rot, int(bool(is_neox)), T, H,
                                                hkv, D, bs, nb, float(k_scale), float(v_scale), dt, _stream(stream)),
           "pa_rope_reshape_and_cache_fp8")


def pa_copy_blocks(key_cache: torch.Tensor, value_cache: torch.Tensor, block_mapping: torch.Tensor,
                   stream=None) -> None:
    """Copy-on-write block copy: block_mapping int64 [n, 2] (source, destination) on the device;
    caches bf16, fp16 or uint8 (8-bit codes)."""
    dt = _cache_code((key_cache, "key_cache"), (value_cache, "value_cache"))
    _need(block_mapping, "block_mapping", torch.int64)
    if not (key_cache.is_contiguous() and value_cache.is_contiguous() and block_mapping.is_contiguous()):
        raise ValueError("caches and block_mapping must be contiguous")
    if block_mapping.dim() != 2 or block_mapping.shape[1] != 2:
        raise ValueError("block_mapping must be [n, 2]")
    _cache_pair_shapes(key_cache, value_cache)
    nb, bs, hkv, d = key_cache.shape
    _check(_lib().pa_copy_blocks(key_cache.data_ptr(), value_cache.data_ptr(), block_mapping.data_ptr(),
                                 block_mapping.shape[0], hkv, d, bs, nb, dt, _stream(stream)), "pa_copy_blocks")


def pa_gather_kv(key_cache: torch.Tensor, value_cache: torch.Tensor, block_table_row: torch.Tensor,
                 seq_len: int, key_out: torch.Tensor, value_out: torch.Tensor, stream=None) -> None:
    dt = _cache_code((key_cache, "key_cache"), (value_cache, "value_cache"), (key_out, "key_out"),
                     (value_out, "value_out"))
    _need(block_table_row, "block_table_row", torch.int32)
    _gather_shapes(key_cache, value_cache, block_table_row, seq_len, key_out, value_out)
    if not all(t.is_contiguous() for t in (key_cache, value_cache, block_table_row, key_out, value_out)):
        raise ValueError("caches, block_table_row and the outputs must be contiguous")
    nb, bs, hkv, d = key_cache.shape
    _check(_lib().pa_gather_kv(key_cache.data_ptr(), value_cache.data_ptr(), block_table_row.data_ptr(), seq_len,
                               hkv, d, bs, nb, key_out.data_ptr(), value_out.data_ptr(), dt,
                               _stream(stream)), "pa_gather_kv")


def pa_debug_status(stream=None) -> int:
    """Synchronise the stream and return (then clear) the device status flags."""
    flags = ctypes.c_uint32(0)
    st = _lib().pa_debug_status(_stream(stream), ctypes.addressof(flags))
    if st not in (0, -7):
        raise PagedAttnError(st, "pa_debug_status")
    return int(flags.value)


def pa_launch_count() -> int:
    return int(_lib().pa_launch_count())


def pa_last_cuda_error() -> str:
    return _lib().pa_last_cuda_error().decode()


def pa_attention_set_timing_events(start: Optional[torch.cuda.Event], stop: Optional[torch.cuda.Event]) -> None:
    s = start.cuda_event if start is not None else None
    e = stop.cuda_event if stop is not None else None
    _check(_lib().pa_attention_set_timing_events(s, e), "pa_attention_set_timing_events")


def pa_attention_set_tile_timing_events(start: Optional[torch.cuda.Event],
                                        stop: Optional[torch.cuda.Event]) -> None:
    s = start.cuda_event if start is not None else None
    e = stop.cuda_event if stop is not None else None
    _check(_lib().pa_attention_set_tile_timing_events(s, e), "pa_attention_set_tile_timing_events")


def pa_status_string(status: int) -> str:
    return _lib().pa_status_string(status).decode()
