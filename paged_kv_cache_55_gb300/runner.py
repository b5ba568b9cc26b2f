"""Device buffers for one paged-attention step and the two library calls on them.

``DeviceStep`` uploads a ``workloads.Workload`` (cache state plus the step's
inputs) to the GPU once and then runs the step: ``pa_reshape_and_cache``
followed by ``pa_attention_varlen`` on the same stream. It only allocates and
marshals; the computation is the library's.
"""

from __future__ import annotations

import numpy as np
import torch

from . import binding as B
from .workloads import Workload


TORCH_DTYPES = {"bf16": torch.bfloat16, "fp16": torch.float16}


def bf16_tensor(a: np.ndarray, device, dtype: str = "bf16") -> torch.Tensor:
    """uint16 bit patterns of the element type -> a bf16 / fp16 tensor on `device` (bits preserved)."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(TORCH_DTYPES[dtype])


def bf16_to_numpy_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_to_float64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


class DeviceStep:
    def __init__(self, w: Workload, device: str = "cuda", rope=None):
        """``rope``: optional (cos_sin_cache float32 [P, rotary_dim], positions int64 [T], is_neox):
        the step then rotates q and K with pa_rope_reshape_and_cache instead of pa_reshape_and_cache."""
        self.w = w
        self.device = torch.device(device)
        dev = self.device
        self.q = bf16_tensor(w.q, dev, w.dtype)
        self.key = bf16_tensor(w.key, dev, w.dtype)
        self.value = bf16_tensor(w.value, dev, w.dtype)
        self.slot_mapping = torch.from_numpy(w.slot_mapping).to(dev)
        self.kv_fp8 = w.kv_fp8
        if self.kv_fp8:  # 8-bit caches: uint8 E4M3 codes
            self.key_cache0 = torch.from_numpy(np.ascontiguousarray(w.key_cache)).to(dev)
            self.value_cache0 = torch.from_numpy(np.ascontiguousarray(w.value_cache)).to(dev)
        else:
            self.key_cache0 = bf16_tensor(w.key_cache, dev, w.dtype)
            self.value_cache0 = bf16_tensor(w.value_cache, dev, w.dtype)
        self.key_cache = self.key_cache0.clone()
        self.value_cache = self.value_cache0.clone()
        self.block_tables = torch.from_numpy(w.block_tables).to(dev)
        self.seq_lens = torch.from_numpy(w.seq_lens).to(dev)
        self.query_start_loc = torch.from_numpy(w.query_start_loc).to(dev)
        self.out = torch.empty((w.total_q, w.num_heads, w.head_dim), dtype=TORCH_DTYPES[w.dtype], device=dev)
        self.max_query_len = w.max_query_len
        self.max_seq_len = w.max_seq_len
        nbytes = B.pa_attention_workspace_size(w.num_seqs, w.total_q, self.max_query_len, self.max_seq_len,
                                               w.num_heads, w.num_kv_heads, w.head_dim, w.block_size)
        self.workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
        self.rope = None
        if rope is not None:
            table, positions, is_neox = rope
            self.rope = (torch.from_numpy(np.ascontiguousarray(table, dtype=np.float32)).to(dev),
                         torch.from_numpy(np.ascontiguousarray(positions, dtype=np.int64)).to(dev), bool(is_neox))

    def reset_cache(self) -> None:
        """Restore the cache to its state before the step."""
        self.key_cache.copy_(self.key_cache0)
        self.value_cache.copy_(self.value_cache0)

    def reshape_and_cache(self, stream=None) -> None:
        if self.rope is not None:
            table, positions, is_neox = self.rope
            if self.kv_fp8:
                B.pa_rope_reshape_and_cache_fp8(self.q, self.key, self.value, self.key_cache, self.value_cache,
                                                self.slot_mapping, positions, table, self.w.k_scale, self.w.v_scale,
                                                is_neox=is_neox, stream=stream)
            else:
                B.pa_rope_reshape_and_cache(self.q, self.key, self.value, self.key_cache, self.value_cache,
                                            self.slot_mapping, positions, table, is_neox=is_neox, stream=stream)
            return
        if self.kv_fp8:
            B.pa_reshape_and_cache_fp8(self.key, self.value, self.key_cache, self.value_cache, self.slot_mapping,
                                       self.w.k_scale, self.w.v_scale, stream=stream)
            return
        B.pa_reshape_and_cache(self.key, self.value, self.key_cache, self.value_cache, self.slot_mapping,
                               stream=stream)

    def attention(self, stream=None) -> None:
        if self.kv_fp8:
            B.pa_attention_varlen_fp8(self.q, self.key_cache, self.value_cache, self.block_tables, self.seq_lens,
                                      self.query_start_loc, self.max_query_len, self.max_seq_len, self.w.scale,
                                      self.w.k_scale, self.w.v_scale, self.out, self.workspace, stream=stream)
            return
        B.pa_attention_varlen(self.q, self.key_cache, self.value_cache, self.block_tables, self.seq_lens,
                              self.query_start_loc, self.max_query_len, self.max_seq_len, self.w.scale,
                              self.out, self.workspace, stream=stream)

    def run(self, stream=None) -> None:
        self.reshape_and_cache(stream)
        self.attention(stream)
