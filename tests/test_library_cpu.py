"""The C-ABI library builds, loads and exports what include/pagedattn.h declares (no GPU)."""

import os
import re
import subprocess

import pytest

from paged_kv_cache_55_gb300 import binding as B
from paged_kv_cache_55_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return B.load_library()


def declared_functions():
    names = []
    inc = os.path.join(ROOT, "include")
    for f in sorted(os.listdir(inc)):
        if f.endswith(".h"):
            text = open(os.path.join(inc, f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^[A-Za-z_][\w\s\*]*?\b(pa_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("pa_reshape_and_cache", "pa_attention_varlen", "pa_attention_workspace_size"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIBRARY], capture_output=True, text=True, check=True).stdout
    exported = set(line.split()[-1] for line in out.splitlines() if line.strip())
    for name in declared_functions():
        assert name in exported, f"{name} declared in include/ but not exported"
        assert hasattr(lib, name)
    assert set(B.SIGNATURES) <= set(declared_functions())


def test_status_strings(lib):
    for code in range(0, -9, -1):
        s = lib.pa_status_string(code).decode()
        assert s and s != "unknown status"
    assert lib.pa_status_string(5).decode() == "unknown status"


def test_workspace_sizes_are_host_arithmetic(lib):
    # GQA decode at batch 256 with lengths up to 8192: partials for every split
    n = lib.pa_attention_workspace_size(256, 256, 1, 8192, 32, 8, 128, 16)
    assert n > 256 * 8 * 16 * 8 * 128 * 4
    assert lib.pa_attention_workspace_size(4, 4, 1, 33, 4, 1, 64, 16) > 0
    # unsupported or inconsistent sizes give 0
    assert lib.pa_attention_workspace_size(4, 4, 1, 33, 4, 1, 112, 16) == 0  # head dims 64, 80, 96, 128, 256
    assert lib.pa_attention_workspace_size(4, 4, 1, 33, 4, 1, 256, 16) > 0
    assert lib.pa_attention_workspace_size(4, 4, 1, 33, 4, 1, 192, 16) == 0
    assert lib.pa_attention_workspace_size(4, 4, 1, 33, 4, 1, 96, 16) > 0
    assert lib.pa_attention_workspace_size(4, 4, 1, 33, 4, 1, 80, 16) > 0
    assert lib.pa_attention_workspace_size(4, 4, 1, 33, 4, 3, 64, 16) == 0
    assert lib.pa_attention_workspace_size(4, 4, 1, 33, 4, 1, 64, 64) == 0  # block sizes 8, 16, 32 only
    assert lib.pa_attention_workspace_size(4, 4, 1, 33, 4, 1, 64, 32) > 0
    assert lib.pa_attention_workspace_size(4, 4, 40, 33, 4, 1, 64, 16) == 0
    pt, mp = B.pa_attention_plan_info(8, 32768, 64, 8)
    assert pt % 16 == 0 and mp == -(-32768 // pt)
    # one size serves both cache types: 8-bit caches run 12 decode warps per SM and split 8 x 32768
    # keys into 1536-key partitions (22 per request) where 16-bit caches use 2048 (16)
    assert pt == 2048
    n = lib.pa_attention_workspace_size(8, 8, 1, 32768, 64, 8, 128, 16)
    partials_8bit = 8 * 8 * 22 * 8 * (128 + 1) * 4
    assert n >= partials_8bit


def test_validation_rejects_before_any_cuda_call(lib):
    # dtype and size errors return before the library touches the device
    args = [None, 0, None, None, None, 0, None, None, 1, 1, 1, 1, 4, 1, 64, 16, 1, 1.0, None, None, 0]
    assert lib.pa_attention_varlen(*args, 2, None) == -3       # dtype (0 = bf16, 1 = fp16)
    assert lib.pa_attention_varlen(*args, 1, None) != -3       # fp16 passes the dtype check
    assert lib.pa_reshape_and_cache(None, None, 0, 0, None, None, None, 0, 1, 64, 16, 1, 1, None) == 0
    assert lib.pa_reshape_and_cache(None, None, 0, 0, None, None, None, 1, 1, 64, 16, 1, 7, None) == -3
    assert lib.pa_reshape_and_cache(None, None, 0, 0, None, None, None, -1, 1, 64, 16, 1, 0, None) == -2
    assert lib.pa_reshape_and_cache(None, None, 0, 0, None, None, None, 0, 1, 64, 16, 1, 0, None) == 0
    assert lib.pa_attention_set_timing_events(None, None) == 0
    assert lib.pa_launch_count() == 0
    assert lib.pa_last_cuda_error() == b"cudaSuccess"
    assert lib.pa_copy_blocks(None, None, None, 3, 8, 128, 16, 10, 3, None) == -3   # dtype
    assert lib.pa_copy_blocks(None, None, None, 3, 8, 128, 16, 10, 2, None) == -1   # 8-bit caches pass the checks
    assert lib.pa_copy_blocks(None, None, None, 3, 8, 8, 16, 10, 2, None) == -4     # 8 codes: half a vector
    assert lib.pa_copy_blocks(None, None, None, -1, 8, 128, 16, 10, 0, None) == -2  # negative count
    assert lib.pa_copy_blocks(None, None, None, 3, 8, 100, 16, 10, 0, None) == -4   # rows not 16-byte vectors
    assert lib.pa_copy_blocks(None, None, None, 0, 8, 128, 16, 10, 1, None) == 0    # nothing to do
    assert lib.pa_copy_blocks(None, None, None, 3, 8, 128, 16, 10, 0, None) == -1   # null pointers


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError, match="no fallback"):
        B.load_library(str(tmp_path / "libpagedattn.so"))


def test_product_code_never_touches_the_oracle():
    pkg = os.path.join(ROOT, "paged_kv_cache_55_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, flags=re.M), f
                assert "liboracle" not in text and "oracle.c" not in text, f


def test_fp8_validation_rejects_before_any_cuda_call(lib):
    # pa_reshape_and_cache_fp8: element type, scales, shapes
    r = lib.pa_reshape_and_cache_fp8
    assert r(None, None, 0, 0, None, None, None, 0, 1, 64, 16, 1, 1.0, 1.0, 0, None) == 0
    assert r(None, None, 0, 0, None, None, None, 1, 1, 64, 16, 1, 1.0, 1.0, 2, None) == -3   # 8-bit inputs
    assert r(None, None, 0, 0, None, None, None, 1, 1, 64, 16, 1, 0.0, 1.0, 0, None) == -2   # zero scale
    assert r(None, None, 0, 0, None, None, None, 1, 1, 64, 16, 1, 1.0, float("inf"), 0, None) == -2
    assert r(None, None, 0, 0, None, None, None, 1, 1, 112, 16, 1, 1.0, 1.0, 0, None) == -3  # head_dim
    assert r(None, None, 0, 0, None, None, None, 1, 1, 80, 16, 1, 1.0, 1.0, 0, None) == -1   # 80: null pointers
    assert r(None, None, 0, 0, None, None, None, 1, 1, 64, 16, 1, 1.0, 1.0, 1, None) == -1   # fp16: null pointers
    # pa_attention_varlen_fp8: scales and element type
    a = lib.pa_attention_varlen_fp8
    base = [None, 0, None, None, None, 1, None, None, 1, 1, 1, 1, 8, 2, 64, 16, 1, 1.0]
    assert a(*base, 1.0, 1.0, None, None, 0, 0, None) == -1                 # passes to the null check
    assert a(*base, -1.0, 1.0, None, None, 0, 0, None) == -2
    assert a(*base, 1.0, float("nan"), None, None, 0, 0, None) == -2
    assert a(*base, 1.0, 1.0, None, None, 0, 2, None) == -3                 # q must be bf16 or fp16
    long_q = [None, 0, None, None, None, 1, None, None, 1, 8, 8, 8, 8, 2, 64, 16, 1, 1.0]
    assert a(*long_q, 1.0, 1.0, None, None, 0, 0, None) == -1               # chunks pass to the null check
    assert lib.pa_gather_kv(None, None, None, 4, 2, 64, 16, 10, None, None, 2, None) == -1
    assert lib.pa_launch_count() == 0


def test_row_sizes_beyond_int32_are_refused_before_any_cuda_call(lib):
    # num_kv_heads * head_dim elements (or bytes) per token row is an int32 inside the kernels
    huge = 1 << 25  # x 128 elements = 2^32
    assert lib.pa_reshape_and_cache(1, 1, 1 << 33, 1 << 33, 1, 1, 1, 1, huge, 128, 16, 1, 0, None) == -3
    assert lib.pa_reshape_and_cache(1, 1, 1 << 33, 1 << 33, 1, 1, 1, 1, 1 << 20, 128, 16, 1, 0, None) != -3
    assert lib.pa_reshape_and_cache_fp8(1, 1, 1 << 33, 1 << 33, 1, 1, 1, 1, huge, 128, 16, 1, 1.0, 1.0, 0,
                                        None) == -3
    assert lib.pa_gather_kv(16, 16, 4, 4, huge // 2, 128, 16, 10, 16, 16, 0, None) == -3
    # rotary scatter: q, K and V rows of one token in 16-byte chunks
    r = lib.pa_rope_reshape_and_cache
    assert r(16, 1 << 40, 16, 16, 1 << 40, 1 << 40, 16, 16, 8, 8, 16, 4096, 128, 1, 1, 1 << 28, 8, 128, 16, 10, 0,
             None) == -3
    assert lib.pa_launch_count() == 0


def test_static_workspace_size_matches_the_header():
    """The binding's copy of PA_STATIC_WORKSPACE_BYTES is the header's value."""
    text = open(os.path.join(ROOT, "include", "pagedattn.h")).read()
    m = re.search(r"#define\s+PA_STATIC_WORKSPACE_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", text)
    assert m, "PA_STATIC_WORKSPACE_BYTES is not a (N u << S) literal any more: update this test"
    assert B.PA_STATIC_WORKSPACE_BYTES == int(m.group(1)) << int(m.group(2))


def test_partition_sizes_follow_the_batch(lib):
    """The split-KV plan's partition size: 512 tokens once the (request, KV head) pairs
    give every decode warp two or more (batch 256 x 8 KV heads on 1216 warps: 512, the
    measured best); otherwise the longest request's keys spread over the warps, rounded
    up to a multiple of 512 and kept within [512, 2048]."""
    pt, mp = B.pa_attention_plan_info(256, 8192, 32, 8)
    assert (pt, mp) == (512, 16)
    pt, mp = B.pa_attention_plan_info(64, 2048, 32, 32)  # MHA batch 64: 2048 pairs
    assert (pt, mp) == (512, 4)
    # few pairs: 4 requests x 8 KV heads x 4096 keys over 1216 warps -> 108 -> 512
    assert B.pa_attention_plan_info(4, 4096, 32, 8)[0] == 512
    # 16 x 8 pairs of 16384 keys -> 1725 per warp -> 2048
    assert B.pa_attention_plan_info(16, 16384, 32, 8) == (2048, 8)
    # 10 x 8 pairs of 8192 keys -> 539 per warp -> 1024
    assert B.pa_attention_plan_info(10, 8192, 32, 8) == (1024, 8)
    # an empty batch still plans one partition of the minimum size
    assert B.pa_attention_plan_info(0, 0, 32, 8)[0] == 512


def test_kernel_hash_ignores_comments_only(tmp_path):
    """bench.py keys the committed ncu counters to a hash of the timed kernel's code
    with `//` comments removed: that is sound only while no string literal in those
    sources contains `//`, and the hash must move with any change to the code (checked
    on copies of the sources)."""
    import shutil
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    for rel in bench.KERNEL_SOURCES:
        text = open(os.path.join(bench.ROOT, rel), encoding="utf-8").read()
        code = "\n".join(line.split("//", 1)[0] for line in text.splitlines())
        assert "/*" not in code, rel
        for lit in re.findall(r'"(?:[^"\\\n]|\\.)*"', code):
            assert "//" not in lit, (rel, lit)
        dst = tmp_path / rel
        dst.parent.mkdir(parents=True, exist_ok=True)
        shutil.copyfile(os.path.join(bench.ROOT, rel), dst)
    h0 = bench.kernel_source_hash()
    assert bench.kernel_source_hash(str(tmp_path)) == h0
    copy = tmp_path / bench.KERNEL_SOURCES[0]
    original = copy.read_text(encoding="utf-8")
    copy.write_text(original.replace("\n", "  // a comment\n", 3) + "\n// another\n\n", encoding="utf-8")
    assert bench.kernel_source_hash(str(tmp_path)) == h0
    copy.write_text(original + "\nstatic int unused_marker_for_the_hash_test = 0;\n", encoding="utf-8")
    assert bench.kernel_source_hash(str(tmp_path)) != h0
