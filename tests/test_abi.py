"""The C ABI library builds, loads without a GPU and exports every symbol the
header declares; host-side validation rejects bad arguments before touching
the device.  CPU only."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pagedkv.h")


@pytest.fixture(scope="module")
def pk():
    from paged_kv_cache_10_gb300 import build, pagedkv
    build.build()
    return pagedkv


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(pk):
    syms = declared_symbols()
    assert "pkv_paged_attention_decode" in syms and "pkv_paged_kv_append" in syms and "pkv_copy_blocks" in syms
    lib = ctypes.CDLL(pk.LIB_PATH)
    missing = [s for s in syms if not hasattr(lib, s)]
    assert not missing
    assert sorted(pk.EXPORTED) == sorted(s for s in syms if s in pk.EXPORTED)
    assert set(syms) <= set(pk.EXPORTED)


def test_status_strings_and_version(pk):
    assert pk.status_string(0) == "ok"
    assert "workspace" in pk.status_string(5)
    assert pk.status_string(99) == "unknown status"
    assert re.match(r"^\d+\.\d+\.\d+$", pk.version())


def test_workspace_size_arithmetic(pk):
    # one partition: no workspace
    assert pk.decode_workspace_bytes(64, 32, 128, 512, 512) == 0
    # S*Hq*NP rows of m and l (256-byte aligned regions) plus D floats each
    S, Hq, D, L, P = 8, 64, 128, 32768, 512
    rows = S * Hq * (L // P)
    ml = -(-rows * 4 // 256) * 256
    assert pk.decode_workspace_bytes(S, Hq, D, L, P) == 2 * ml + rows * D * 4
    # auto sizes for its smallest partition (256 tokens), covering any choice it makes
    assert pk.decode_workspace_bytes(S, Hq, D, L, 0) == pk.decode_workspace_bytes(S, Hq, D, L, 256)
    assert pk.decode_workspace_bytes(S, Hq, D, L, 100) == 0  # not a multiple of the block size


def test_validation_rejects_before_any_launch(pk):
    L = pk.lib()
    d = pk.CacheDesc(num_blocks=8, num_kv_heads=2, head_size=128, kv_dtype="bf16").c()
    fake = 1 << 20  # never dereferenced: every call below fails validation first
    # head_size 96 is unsupported
    d96 = pk.CacheDesc(num_blocks=8, num_kv_heads=2, head_size=96, kv_dtype="bf16").c()
    assert L.pkv_paged_attention_decode(fake, 1, 2, 4, fake, fake, ctypes.byref(d96), fake, 4, fake, 64,
                                        0.1, fake, None, 0, 0, None) == pk.ERR_UNSUPPORTED
    # group of 3 query heads per KV head is unsupported; 5 heads over 2 is invalid
    assert L.pkv_paged_attention_decode(fake, 1, 2, 6, fake, fake, ctypes.byref(d), fake, 4, fake, 64,
                                        0.1, fake, None, 0, 0, None) == pk.ERR_UNSUPPORTED
    assert L.pkv_paged_attention_decode(fake, 1, 2, 5, fake, fake, ctypes.byref(d), fake, 4, fake, 64,
                                        0.1, fake, None, 0, 0, None) == pk.ERR_INVALID
    # q dtype must match a 16-bit pool
    assert L.pkv_paged_attention_decode(fake, 0, 2, 4, fake, fake, ctypes.byref(d), fake, 4, fake, 64,
                                        0.1, fake, None, 0, 0, None) == pk.ERR_UNSUPPORTED
    # max_seq_len beyond the table, partition not a multiple of 16, misaligned pointer
    assert L.pkv_paged_attention_decode(fake, 1, 2, 4, fake, fake, ctypes.byref(d), fake, 4, fake, 65,
                                        0.1, fake, None, 0, 0, None) == pk.ERR_INVALID
    assert L.pkv_paged_attention_decode(fake, 1, 2, 4, fake, fake, ctypes.byref(d), fake, 4, fake, 64,
                                        0.1, fake, None, 0, 24, None) == pk.ERR_INVALID
    assert L.pkv_paged_attention_decode(fake + 2, 1, 2, 4, fake, fake, ctypes.byref(d), fake, 4, fake, 64,
                                        0.1, fake, None, 0, 0, None) == pk.ERR_INVALID
    # workspace required for a split launch
    assert L.pkv_paged_attention_decode(fake, 1, 2, 4, fake, fake, ctypes.byref(d), fake, 4, fake, 64,
                                        0.1, fake, None, 0, 16, None) == pk.ERR_WORKSPACE
    # null descriptor, negative sizes
    assert L.pkv_paged_attention_decode(fake, 1, 2, 4, fake, fake, None, fake, 4, fake, 64,
                                        0.1, fake, None, 0, 0, None) == pk.ERR_INVALID
    assert L.pkv_paged_kv_append(fake, fake, 1, -1, fake, fake, fake, ctypes.byref(d), None) == pk.ERR_INVALID
    # append: bf16 input into an f16 pool is unsupported; misaligned slot_mapping invalid
    d16 = pk.CacheDesc(num_blocks=8, num_kv_heads=2, head_size=128, kv_dtype="f16").c()
    assert L.pkv_paged_kv_append(fake, fake, 1, 4, fake, fake, fake, ctypes.byref(d16), None) == pk.ERR_UNSUPPORTED
    assert L.pkv_paged_kv_append(fake, fake, 1, 4, fake + 4, fake, fake, ctypes.byref(d), None) == pk.ERR_INVALID
    # fp8 pool needs positive scales
    d8 = pk.CacheDesc(num_blocks=8, num_kv_heads=2, head_size=128, kv_dtype="e4m3", k_scale=0.0).c()
    assert L.pkv_copy_blocks(fake, fake, ctypes.byref(d8), fake, 1, None) == pk.ERR_INVALID
    # empty work is a no-op that needs no device
    assert L.pkv_copy_blocks(fake, fake, ctypes.byref(d), None, 0, None) == pk.OK
    assert L.pkv_paged_kv_append(None, None, 1, 0, None, None, None, ctypes.byref(d), None) == pk.OK


def test_prefill_validation_rejects_before_any_launch(pk):
    L = pk.lib()
    d = pk.CacheDesc(num_blocks=8, num_kv_heads=2, head_size=128, kv_dtype="bf16").c()
    d96 = pk.CacheDesc(num_blocks=8, num_kv_heads=2, head_size=96, kv_dtype="bf16").c()
    fake = 1 << 20  # never dereferenced

    def call(desc=d, q_dtype=1, work=None, nwork=0, scale=0.1, Hq=8, ws=None, ws_bytes=0):
        return L.pkv_paged_attention_prefill(fake, q_dtype, 64, Hq, 2, fake, 32, fake, fake, ctypes.byref(desc), fake,
                                             4, fake, work, nwork, scale, fake, ws, ws_bytes, None)

    assert call(nwork=-1) == pk.ERR_INVALID            # negative work-list length
    assert call(work=None, nwork=3) == pk.ERR_INVALID  # a length without a list
    assert call(work=fake, nwork=0) == pk.OK           # an empty list: nothing to run
    assert call(desc=d96) == pk.ERR_UNSUPPORTED        # head_size 96
    assert call(q_dtype=0) == pk.ERR_UNSUPPORTED       # f16 q over a bf16 pool
    assert call(scale=0.0) == pk.ERR_INVALID           # the row maximum needs scale > 0
    assert call(Hq=6) == pk.ERR_UNSUPPORTED            # 3 query heads per KV head
    assert call(Hq=5) == pk.ERR_INVALID                # heads not a multiple
    # fp8 pools: a 16-bit q, positive finite scales, a large enough aligned workspace
    d8 = pk.CacheDesc(num_blocks=8, num_kv_heads=2, head_size=128, kv_dtype="e4m3", k_scale=0.5, v_scale=0.25).c()
    need = L.pkv_prefill_workspace_bytes(pk.FP8_E4M3, 2, 2, 128, 4)
    assert need > 0
    assert call(desc=d8) == pk.ERR_WORKSPACE                           # no workspace
    assert call(desc=d8, ws=fake, ws_bytes=need - 1) == pk.ERR_WORKSPACE
    assert call(desc=d8, ws=fake + 4, ws_bytes=need + 4) == pk.ERR_INVALID  # not 16-byte aligned
    assert call(desc=d8, q_dtype=2, ws=fake, ws_bytes=need) == pk.ERR_UNSUPPORTED  # fp8 q
    for ks, vs in [(0.0, 1.0), (1.0, -1.0), (float("inf"), 1.0), (float("nan"), 1.0)]:
        bad = pk.CacheDesc(num_blocks=8, num_kv_heads=2, head_size=128, kv_dtype="e4m3", k_scale=ks, v_scale=vs).c()
        assert call(desc=bad, ws=fake, ws_bytes=need) == pk.ERR_INVALID


def test_cascade_validation_rejects_before_any_launch(pk):
    L = pk.lib()
    d = pk.CacheDesc(num_blocks=8, num_kv_heads=2, head_size=128, kv_dtype="bf16").c()
    d96 = pk.CacheDesc(num_blocks=8, num_kv_heads=2, head_size=96, kv_dtype="bf16").c()
    d8 = pk.CacheDesc(num_blocks=8, num_kv_heads=2, head_size=128, kv_dtype="e4m3", k_scale=0.0).c()
    fake = 1 << 20  # never dereferenced: every call below fails validation first

    def call(desc=d, q_dtype=1, S=2, Hq=8, mgb=2, part=16, ws=None, ws_bytes=0, q=fake):
        return L.pkv_paged_attention_decode_cascade(q, q_dtype, S, Hq, fake, fake, ctypes.byref(desc), fake, 4,
                                                    fake, 64, fake, fake, fake, fake, 1, 2, mgb, 0.1, fake, ws,
                                                    ws_bytes, part, None)

    assert call(S=0) == pk.OK                           # an empty batch needs no device
    assert call(S=65535) == pk.ERR_UNSUPPORTED          # the decode grid's join layer needs one more z index
    assert call(desc=d96) == pk.ERR_UNSUPPORTED         # head_size 96
    assert call(q_dtype=0) == pk.ERR_UNSUPPORTED        # f16 q over a bf16 pool
    assert call(Hq=6) == pk.ERR_UNSUPPORTED             # 3 query heads per KV head
    assert call(Hq=5) == pk.ERR_INVALID                 # heads not a multiple
    assert call(desc=d8) == pk.ERR_INVALID              # fp8 pool without a positive k_scale
    assert call(mgb=5) == pk.ERR_INVALID                # shared prefix longer than the block table
    assert call(part=24) == pk.ERR_INVALID              # partition not a multiple of the block size
    assert call(q=fake + 2) == pk.ERR_INVALID           # q not 16-byte aligned
    assert call() == pk.ERR_WORKSPACE                   # no workspace for the partials
    need = L.pkv_decode_cascade_workspace_bytes(2, 8, 128, 64, 16, 2)
    assert need > 0
    assert call(ws=fake, ws_bytes=need - 1) == pk.ERR_WORKSPACE


def test_prefill_workspace_bytes(pk):
    """0 for 16-bit pools (read in place); for fp8 pools a 4-byte table entry
    per (sequence, block) and two 16-bit copies of S * MB blocks, each part
    rounded up to 256 bytes."""
    L = pk.lib()
    for code in (pk.F16, pk.BF16):
        assert L.pkv_prefill_workspace_bytes(code, 8, 8, 128, 256) == 0
    up = lambda x: -(-x // 256) * 256
    for S, Hkv, D, MB in [(2, 2, 128, 4), (8, 8, 128, 256), (3, 1, 64, 7), (0, 4, 128, 10)]:
        copy = S * MB * Hkv * 16 * D * 2
        assert L.pkv_prefill_workspace_bytes(pk.FP8_E4M3, S, Hkv, D, MB) == up(S * MB * 4) + 2 * up(copy)
    assert L.pkv_prefill_workspace_bytes(pk.FP8_E4M3, -1, 2, 128, 4) == 0
    assert L.pkv_prefill_workspace_bytes(pk.FP8_E4M3, 2, 0, 128, 4) == 0


def test_header_declares_every_exported_function_in_c(pk, tmp_path):
    """include/pagedkv.h compiles as C99 and C++17 without warnings and
    declares every function the binding loads (a stray comment would hide
    a declaration from C callers while the library still builds)."""
    import shutil
    import subprocess
    if not shutil.which("gcc") or not shutil.which("g++"):
        pytest.skip("no host compiler")
    refs = "\n".join(f"    (void)&{s};" for s in sorted(pk.EXPORTED))
    src = tmp_path / "use_header.c"
    src.write_text(f'#include "pagedkv.h"\nint main(void) {{\n{refs}\n    return 0;\n}}\n')
    inc = os.path.dirname(HEADER)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", inc, "-fsyntax-only", str(src)], check=True)
    subprocess.run(["g++", "-std=c++17", "-Wall", "-Werror", "-I", inc, "-fsyntax-only", "-x", "c++", str(src)],
                   check=True)
