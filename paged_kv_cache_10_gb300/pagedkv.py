"""ctypes binding of ``libpagedkv.so`` (argument marshalling only).

Every computation runs in the library's CUDA kernels or its C++ allocator;
this module converts torch tensors to pointers, picks the stream and turns
status codes into exceptions.  It never falls back to another
implementation: if the library is missing it raises.

Names follow the C ABI in ``include/pagedkv.h`` without the ``pkv_`` prefix.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpagedkv.so")

OK, ERR_INVALID, ERR_UNSUPPORTED, ERR_OOM, ERR_CUDA, ERR_WORKSPACE, ERR_NOT_FOUND = range(7)
F16, BF16, FP8_E4M3 = 0, 1, 2
DTYPE_CODE = {"f16": F16, "bf16": BF16, "e4m3": FP8_E4M3}
DEVERR_BLOCK_ID, DEVERR_SEQ_LEN, DEVERR_SLOT, DEVERR_COPY_PAIR, DEVERR_TIMEOUT = 1, 2, 4, 8, 16

EXPORTED = [
    "pkv_paged_kv_append", "pkv_copy_blocks", "pkv_decode_workspace_bytes",
    "pkv_paged_attention_decode", "pkv_paged_attention_decode_noalloc", "pkv_decode_auto_partition", "pkv_get_device_error",
    "pkv_status_string", "pkv_version", "pkv_set_decode_path", "pkv_get_decode_path", "pkv_alloc_create", "pkv_alloc_destroy",
    "pkv_alloc_seq_new", "pkv_alloc_fork", "pkv_alloc_append_slot", "pkv_alloc_seq_extend",
    "pkv_alloc_free", "pkv_alloc_append_batch", "pkv_alloc_export", "pkv_alloc_block_table",
    "pkv_alloc_seq_len", "pkv_alloc_refcount", "pkv_alloc_num_free", "pkv_alloc_num_seqs",
    "pkv_alloc_fail_after", "pkv_paged_attention_decode_cascade", "pkv_decode_cascade_workspace_bytes",
    "pkv_alloc_prefix_groups", "pkv_swap_blocks", "pkv_alloc_swap_out", "pkv_alloc_swap_in",
    "pkv_paged_attention_prefill", "pkv_alloc_append_tokens", "pkv_block_hash", "pkv_prefix_block_hashes",
    "pkv_alloc_lookup", "pkv_alloc_seq_new_prefix", "pkv_alloc_commit", "pkv_alloc_num_cached",
    "pkv_alloc_block_hash_of", "pkv_alloc_reset_prefix_cache", "pkv_paged_attention_decode_append",
    "pkv_prefill_plan", "pkv_decode_plan", "pkv_prefill_workspace_bytes", "pkv_check_wait_timeout",
    "pkv_decode_cascade_staging_bytes",
]


class PagedKVError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


class OutOfBlocks(PagedKVError):
    pass


class _CacheDesc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_size", ctypes.c_int32),
                ("kv_dtype", ctypes.c_int32), ("k_scale", ctypes.c_float), ("v_scale", ctypes.c_float)]


@dataclass
class CacheDesc:
    num_blocks: int
    num_kv_heads: int
    head_size: int
    kv_dtype: str = "bf16"
    k_scale: float = 1.0
    v_scale: float = 1.0
    block_size: int = 16

    def c(self) -> _CacheDesc:
        return _CacheDesc(self.num_blocks, self.block_size, self.num_kv_heads, self.head_size,
                          DTYPE_CODE[self.kv_dtype], self.k_scale, self.v_scale)


_lib = None


def lib():
    """Loads the library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with paged_kv_cache_10_gb300.build.build()")
    L = ctypes.CDLL(LIB_PATH)
    P, i32, i64, u32p = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.POINTER(ctypes.c_uint32)
    D = ctypes.POINTER(_CacheDesc)
    sig = {
        "pkv_paged_kv_append": (i32, [P, P, i32, i32, P, P, P, D, P]),
        "pkv_copy_blocks": (i32, [P, P, D, P, i32, P]),
        "pkv_decode_workspace_bytes": (ctypes.c_size_t, [i32, i32, i32, i32, i32]),
        "pkv_paged_attention_decode": (i32, [P, i32, i32, i32, P, P, D, P, i32, P, i32, ctypes.c_float,
                                             P, P, ctypes.c_size_t, i32, P]),
        "pkv_paged_attention_decode_noalloc": (i32, [P, i32, i32, i32, P, P, D, P, i32, P, i32, ctypes.c_float,
                                                     P, i32, P]),
        "pkv_decode_auto_partition": (i32, [i32, i32, i32, i32, i32, i32]),
        "pkv_get_device_error": (i32, [u32p, P]),
        "pkv_check_wait_timeout": (i32, [i32, P]),
        "pkv_set_decode_path": (i32, [i32]),
        "pkv_get_decode_path": (i32, []),
        "pkv_status_string": (ctypes.c_char_p, [i32]),
        "pkv_version": (ctypes.c_char_p, []),
        "pkv_alloc_create": (P, [i32, i32, P]),
        "pkv_alloc_destroy": (None, [P]),
        "pkv_alloc_seq_new": (i32, [P, i64, i32]),
        "pkv_alloc_fork": (i32, [P, i64, i64]),
        "pkv_alloc_append_slot": (i32, [P, i64, P, P, P]),
        "pkv_alloc_seq_extend": (i32, [P, i64, i32]),
        "pkv_alloc_free": (i32, [P, i64]),
        "pkv_alloc_append_batch": (i32, [P, P, i32, P, P, i32, P]),
        "pkv_alloc_export": (i32, [P, P, i32, P, i32, P]),
        "pkv_alloc_block_table": (i32, [P, i64, P, i32, P]),
        "pkv_alloc_seq_len": (i32, [P, i64, P]),
        "pkv_alloc_refcount": (i32, [P, i32]),
        "pkv_alloc_num_free": (i32, [P]),
        "pkv_alloc_num_seqs": (i32, [P]),
        "pkv_alloc_fail_after": (None, [P, i64]),
        "pkv_paged_attention_decode_cascade": (i32, [P, i32, i32, i32, P, P, D, P, i32, P, i32, P, P, P, P, i32, i32,
                                                     i32, ctypes.c_float, P, P, ctypes.c_size_t, i32, P]),
        "pkv_decode_cascade_workspace_bytes": (ctypes.c_size_t, [i32, i32, i32, i32, i32, i32]),
        "pkv_decode_cascade_staging_bytes": (ctypes.c_size_t, [i32, i32, i32, i32, i32, i32, i32]),
        "pkv_alloc_prefix_groups": (i32, [P, P, i32, i32, P, P, P, P, P, P, P]),
        "pkv_swap_blocks": (i32, [P, P, D, P, P, i32, P, i32, i32, P]),
        "pkv_alloc_swap_out": (i32, [P, P, i64, P, i32, P]),
        "pkv_alloc_swap_in": (i32, [P, P, i64, P, i32, P]),
        "pkv_alloc_append_tokens": (i32, [P, P, P, i32, P, i64, P, i32, P]),
        "pkv_paged_attention_decode_append": (i32, [P, P, i32, P, P, P, i32, i32, i32, P, P, D, P, i32, P, i32,
                                                    ctypes.c_float, P, P, ctypes.c_size_t, i32, P, i32, P]),
        "pkv_decode_plan": (i32, [P, i32, i32, i32, i32, P, i32, P]),
        "pkv_block_hash": (ctypes.c_uint64, [ctypes.c_uint64, P, i32, P, i32]),
        "pkv_prefix_block_hashes": (i32, [P, i64, i32, P, i32, P, P, i64, P]),
        "pkv_alloc_lookup": (i32, [P, P, i32]),
        "pkv_alloc_seq_new_prefix": (i32, [P, i64, P, i32, i32, P]),
        "pkv_alloc_commit": (i32, [P, i64, P, i32, P]),
        "pkv_alloc_num_cached": (i32, [P]),
        "pkv_alloc_block_hash_of": (i64, [P, i32, P]),
        "pkv_alloc_reset_prefix_cache": (None, [P]),
        "pkv_paged_attention_prefill": (i32, [P, i32, i32, i32, i32, P, i32, P, P, D, P, i32, P, P, i32,
                                              ctypes.c_float, P, P, ctypes.c_size_t, P]),
        "pkv_prefill_workspace_bytes": (ctypes.c_size_t, [i32, i32, i32, i32, i32]),
        "pkv_prefill_plan": (i32, [P, P, i32, i32, i32, i32, P, i32, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def status_string(status: int) -> str:
    return lib().pkv_status_string(int(status)).decode()


def version() -> str:
    return lib().pkv_version().decode()


def _check(status: int, what: str) -> None:
    if status == ERR_OOM:
        raise OutOfBlocks(status, what)
    if status != OK:
        raise PagedKVError(status, what)


def _dev_ptr(t: torch.Tensor, name: str) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


_TORCH_CODE = {torch.float16: F16, torch.bfloat16: BF16}


def _dtype_code(t: torch.Tensor, declared: str | None) -> int:
    if declared is not None:
        return DTYPE_CODE[declared]
    if t.dtype not in _TORCH_CODE:
        raise TypeError(f"cannot infer element type from {t.dtype}; pass it explicitly")
    return _TORCH_CODE[t.dtype]


# ------------------------------------------------------------------- GPU ops
def paged_kv_append(k, v, slot_mapping, k_cache, v_cache, desc: CacheDesc, in_dtype: str | None = None,
                    stream=None) -> None:
    """k, v: [T, Hkv, D]; slot_mapping: int64 [T] (device)."""
    T = int(slot_mapping.shape[0])
    if slot_mapping.dtype != torch.int64:
        raise TypeError("slot_mapping must be int64")
    st = lib().pkv_paged_kv_append(_dev_ptr(k, "k"), _dev_ptr(v, "v"), _dtype_code(k, in_dtype), T,
                                   _dev_ptr(slot_mapping, "slot_mapping"), _dev_ptr(k_cache, "k_cache"),
                                   _dev_ptr(v_cache, "v_cache"), ctypes.byref(desc.c()), _stream(stream))
    _check(st, "paged_kv_append")


def copy_blocks(k_cache, v_cache, desc: CacheDesc, pairs, num_pairs: int | None = None, stream=None) -> None:
    """pairs: int32 [n, 2] (device) of (src, dst)."""
    n = int(pairs.shape[0]) if num_pairs is None else int(num_pairs)
    if pairs.dtype != torch.int32:
        raise TypeError("pairs must be int32")
    st = lib().pkv_copy_blocks(_dev_ptr(k_cache, "k_cache"), _dev_ptr(v_cache, "v_cache"), ctypes.byref(desc.c()),
                               _dev_ptr(pairs, "pairs") if n > 0 else None, n, _stream(stream))
    _check(st, "copy_blocks")


def decode_workspace_bytes(num_seqs: int, num_q_heads: int, head_size: int, max_seq_len: int,
                           partition_tokens: int = 0) -> int:
    return int(lib().pkv_decode_workspace_bytes(num_seqs, num_q_heads, head_size, max_seq_len, partition_tokens))


def decode_auto_partition(num_seqs, num_q_heads, num_kv_heads, head_size, max_seq_len, planned: bool = False) -> int:
    r = int(lib().pkv_decode_auto_partition(num_seqs, num_q_heads, num_kv_heads, head_size, max_seq_len,
                                            1 if planned else 0))
    if r < 0:
        _check(-r, "decode_auto_partition")
    return r


def paged_attention_decode(q, k_cache, v_cache, desc: CacheDesc, block_tables, seq_lens, max_seq_len: int,
                           scale: float, out, workspace=None, partition_tokens: int = 0,
                           q_dtype: str | None = None, stream=None) -> None:
    """q, out: [S, Hq, D]; block_tables: int32 [S, MB]; seq_lens: int32 [S] (device)."""
    S, Hq = int(q.shape[0]), int(q.shape[1])
    if block_tables.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise TypeError("block_tables and seq_lens must be int32")
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = _dev_ptr(workspace, "workspace"), workspace.numel() * workspace.element_size()
    st = lib().pkv_paged_attention_decode(_dev_ptr(q, "q"), _dtype_code(q, q_dtype), S, Hq,
                                          _dev_ptr(k_cache, "k_cache"), _dev_ptr(v_cache, "v_cache"),
                                          ctypes.byref(desc.c()), _dev_ptr(block_tables, "block_tables"),
                                          int(block_tables.shape[1]), _dev_ptr(seq_lens, "seq_lens"),
                                          int(max_seq_len), float(scale), _dev_ptr(out, "out"), ws_ptr, ws_bytes,
                                          int(partition_tokens), _stream(stream))
    _check(st, "paged_attention_decode")


PATH_AUTO, PATH_CUDA_CORES, PATH_TENSOR_CORES = 0, 1, 2


def set_decode_path(path: int) -> None:
    _check(lib().pkv_set_decode_path(int(path)), "set_decode_path")


def get_decode_path() -> int:
    return int(lib().pkv_get_decode_path())


class decode_path:
    """Context manager selecting the decode kernel (see pkv_set_decode_path)."""

    def __init__(self, path: int):
        self.path = path

    def __enter__(self):
        self.prev = get_decode_path()
        set_decode_path(self.path)
        return self

    def __exit__(self, *exc):
        set_decode_path(self.prev)
        return False


def paged_attention_decode_noalloc(q, k_cache, v_cache, desc: CacheDesc, block_tables, seq_lens,
                                   max_seq_len: int, scale: float, out, partition_tokens: int = 0,
                                   q_dtype: str | None = None, stream=None) -> None:
    """Decode attention for callers that cannot supply a workspace: the
    library's built-in 32 MiB scratch array is used instead (see the C
    declaration for its limits and sharing rules)."""
    S, Hq = int(q.shape[0]), int(q.shape[1])
    if block_tables.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise TypeError("block_tables and seq_lens must be int32")
    st = lib().pkv_paged_attention_decode_noalloc(_dev_ptr(q, "q"), _dtype_code(q, q_dtype), S, Hq,
                                                  _dev_ptr(k_cache, "k_cache"), _dev_ptr(v_cache, "v_cache"),
                                                  ctypes.byref(desc.c()), _dev_ptr(block_tables, "block_tables"),
                                                  int(block_tables.shape[1]), _dev_ptr(seq_lens, "seq_lens"),
                                                  int(max_seq_len), float(scale), _dev_ptr(out, "out"),
                                                  int(partition_tokens), _stream(stream))
    _check(st, "paged_attention_decode_noalloc")


def decode_cascade_workspace_bytes(num_seqs: int, num_q_heads: int, head_size: int, max_seq_len: int,
                                   partition_tokens: int, max_group_blocks: int) -> int:
    return int(lib().pkv_decode_cascade_workspace_bytes(num_seqs, num_q_heads, head_size, max_seq_len,
                                                        partition_tokens, max_group_blocks))


def decode_cascade_staging_bytes(kv_dtype: str, num_seqs: int, max_blocks_per_seq: int, num_groups: int,
                                 max_group_blocks: int, num_kv_heads: int, head_size: int) -> int:
    return int(lib().pkv_decode_cascade_staging_bytes(DTYPE_CODE[kv_dtype], num_seqs, max_blocks_per_seq, num_groups,
                                                      max_group_blocks, num_kv_heads, head_size))


def decode_cascade_total_workspace_bytes(kv_dtype: str, num_seqs: int, num_q_heads: int, num_kv_heads: int,
                                         head_size: int, max_seq_len: int, max_blocks_per_seq: int,
                                         partition_tokens: int, num_groups: int, max_group_blocks: int) -> int:
    """Whole workspace of a cascade decode call: the partials, then (fp8 pools)
    the groups' 16-bit prefix copy at the next 256-byte boundary."""
    part = decode_cascade_workspace_bytes(num_seqs, num_q_heads, head_size, max_seq_len, partition_tokens,
                                          max_group_blocks)
    stage = decode_cascade_staging_bytes(kv_dtype, num_seqs, max_blocks_per_seq, num_groups, max_group_blocks,
                                         num_kv_heads, head_size)
    return (-(-part // 256) * 256 + stage) if stage else part


@dataclass
class PrefixGroups:
    """Output of Allocator.prefix_groups (host numpy arrays)."""
    seq_group: np.ndarray      # int32 [n]
    group_blocks: np.ndarray   # int32 [num_groups]
    group_offsets: np.ndarray  # int32 [num_groups + 1]
    group_members: np.ndarray  # int32 [members]
    max_members: int
    max_blocks: int

    @property
    def num_groups(self) -> int:
        return int(self.group_blocks.shape[0])


def paged_attention_decode_append(k_new, v_new, slot_mapping, q, k_cache, v_cache, desc: CacheDesc, block_tables,
                                  seq_lens, max_seq_len: int, scale: float, out, workspace=None,
                                  partition_tokens: int = 0, q_dtype: str | None = None, in_dtype: str | None = None,
                                  cow_src=None, stream=None, work_units=None) -> None:
    """Copy-on-write copies into the appending rows' last blocks (cow_src
    int32 [S], -1 for none), append (one token per batch row, slot_mapping
    int64 [S]) and decode, in one launch."""
    S, Hq = int(q.shape[0]), int(q.shape[1])
    if slot_mapping.dtype != torch.int64 or int(slot_mapping.shape[0]) != S:
        raise ValueError("slot_mapping must be int64 with one entry per batch row")
    if cow_src is not None and (cow_src.dtype != torch.int32 or int(cow_src.shape[0]) != S):
        raise ValueError("cow_src must be int32 with one entry per batch row")
    ws_ptr = _dev_ptr(workspace, "workspace") if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib().pkv_paged_attention_decode_append(
        _dev_ptr(k_new, "k_new"), _dev_ptr(v_new, "v_new"), _dtype_code(k_new, in_dtype),
        _dev_ptr(slot_mapping, "slot_mapping"), _dev_ptr(cow_src, "cow_src") if cow_src is not None else None,
        _dev_ptr(q, "q"), _dtype_code(q, q_dtype), S, Hq,
        _dev_ptr(k_cache, "k_cache"), _dev_ptr(v_cache, "v_cache"), ctypes.byref(desc.c()),
        _dev_ptr(block_tables, "block_tables"), int(block_tables.shape[1]), _dev_ptr(seq_lens, "seq_lens"),
        int(max_seq_len), float(scale), _dev_ptr(out, "out"), ws_ptr, ws_bytes, int(partition_tokens),
        _dev_ptr(work_units, "work_units") if work_units is not None and work_units.numel() else None,
        int(work_units.numel()) if work_units is not None else 0, _stream(stream))
    _check(st, "paged_attention_decode_append")


def decode_plan(seq_lens, num_kv_heads: int, max_seq_len: int, partition_tokens: int = 0) -> np.ndarray:
    """Host work plan for paged_attention_decode_append: every (sequence,
    partition) unit, longest first (int32)."""
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    S = int(sl.size)
    n = ctypes.c_int32(0)
    st = lib().pkv_decode_plan(_np_ptr(sl) if S else None, S, int(num_kv_heads), int(max_seq_len),
                               int(partition_tokens), None, 0, ctypes.byref(n))
    if st not in (0, 5):
        _check(st, "decode_plan")
    out = np.zeros(max(int(n.value), 1), dtype=np.int32)
    st = lib().pkv_decode_plan(_np_ptr(sl) if S else None, S, int(num_kv_heads), int(max_seq_len),
                               int(partition_tokens), _np_ptr(out), int(out.size), ctypes.byref(n))
    _check(st, "decode_plan")
    return out[: int(n.value)]


def paged_attention_decode_cascade(q, k_cache, v_cache, desc: CacheDesc, block_tables, seq_lens, max_seq_len: int,
                                   scale: float, out, seq_group, group_blocks, group_offsets, group_members,
                                   max_group_members: int, max_group_blocks: int, workspace,
                                   partition_tokens: int = 0, q_dtype: str | None = None, stream=None) -> None:
    """Shared-prefix decode; the group arrays are int32 device tensors."""
    S, Hq = int(q.shape[0]), int(q.shape[1])
    ng = int(group_blocks.shape[0])
    ptr = lambda t, n: _dev_ptr(t, n) if t.numel() > 0 else None
    st = lib().pkv_paged_attention_decode_cascade(
        _dev_ptr(q, "q"), _dtype_code(q, q_dtype), S, Hq, _dev_ptr(k_cache, "k_cache"), _dev_ptr(v_cache, "v_cache"),
        ctypes.byref(desc.c()), _dev_ptr(block_tables, "block_tables"), int(block_tables.shape[1]),
        _dev_ptr(seq_lens, "seq_lens"), int(max_seq_len), _dev_ptr(seq_group, "seq_group"),
        ptr(group_blocks, "group_blocks"), ptr(group_offsets, "group_offsets"), ptr(group_members, "group_members"),
        ng, int(max_group_members), int(max_group_blocks), float(scale), _dev_ptr(out, "out"),
        _dev_ptr(workspace, "workspace"), workspace.numel() * workspace.element_size(), int(partition_tokens),
        _stream(stream))
    _check(st, "paged_attention_decode_cascade")


def paged_attention_prefill(q, k_cache, v_cache, desc: CacheDesc, query_start, max_query_len: int, block_tables,
                            seq_lens, scale: float, out, q_dtype: str | None = None, stream=None,
                            work_units=None, workspace=None) -> None:
    """Causal paged prefill: q, out [T, Hq, D]; query_start int32 [S + 1],
    block_tables int32 [S, MB], seq_lens int32 [S] (device tensors);
    work_units: optional device int32 CTA order from prefill_plan;
    workspace: device buffer of prefill_workspace_bytes(...) bytes (fp8 pools)."""
    T, Hq = int(q.shape[0]), int(q.shape[1])
    S = int(seq_lens.shape[0])
    if int(query_start.shape[0]) != S + 1:
        raise ValueError("query_start must have num_seqs + 1 entries")
    nw = 0 if work_units is None else int(work_units.numel())
    wp = _dev_ptr(work_units, "work_units") if nw else None
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = _dev_ptr(workspace, "workspace"), workspace.numel() * workspace.element_size()
    st = lib().pkv_paged_attention_prefill(
        _dev_ptr(q, "q"), _dtype_code(q, q_dtype), T, Hq, S, _dev_ptr(query_start, "query_start"), int(max_query_len),
        _dev_ptr(k_cache, "k_cache"), _dev_ptr(v_cache, "v_cache"), ctypes.byref(desc.c()),
        _dev_ptr(block_tables, "block_tables"), int(block_tables.shape[1]), _dev_ptr(seq_lens, "seq_lens"),
        wp, nw, float(scale), _dev_ptr(out, "out"), ws_ptr, ws_bytes, _stream(stream))
    _check(st, "paged_attention_prefill")


def prefill_workspace_bytes(kv_dtype: str, num_seqs: int, num_kv_heads: int, head_size: int,
                            max_blocks_per_seq: int) -> int:
    return int(lib().pkv_prefill_workspace_bytes(DTYPE_CODE[kv_dtype], num_seqs, num_kv_heads, head_size,
                                                 max_blocks_per_seq))


def prefill_plan(query_start, seq_lens, num_q_heads: int, num_kv_heads: int, max_query_len: int) -> np.ndarray:
    """Host work plan for paged_attention_prefill (host arrays in, int32
    units out, longest causal key range first)."""
    qs = np.ascontiguousarray(query_start, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    S = int(sl.size)
    if qs.size != S + 1:
        raise ValueError("query_start must have num_seqs + 1 entries")
    n = ctypes.c_int32(0)
    st = lib().pkv_prefill_plan(_np_ptr(qs), _np_ptr(sl) if S else None, S, int(num_q_heads), int(num_kv_heads),
                                int(max_query_len), None, 0, ctypes.byref(n))
    if st not in (0, 5):  # OK or WORKSPACE (count only)
        _check(st, "prefill_plan")
    out = np.zeros(max(int(n.value), 1), dtype=np.int32)
    st = lib().pkv_prefill_plan(_np_ptr(qs), _np_ptr(sl) if S else None, S, int(num_q_heads), int(num_kv_heads),
                                int(max_query_len), _np_ptr(out), int(out.size), ctypes.byref(n))
    _check(st, "prefill_plan")
    return out[: int(n.value)]


def block_hash(parent: int, tokens, extras=()) -> int:
    t = np.ascontiguousarray(tokens, dtype=np.int32)
    e = np.ascontiguousarray(extras, dtype=np.uint64)
    return int(lib().pkv_block_hash(int(parent), _np_ptr(t) if t.size else None, int(t.size),
                                    _np_ptr(e) if e.size else None, int(e.size)))


def prefix_block_hashes(tokens, block_size: int = 16, extras=(), salt: int | None = None) -> np.ndarray:
    """Cascaded hashes of the full blocks of a token sequence (uint64)."""
    t = np.ascontiguousarray(tokens, dtype=np.int32)
    e = np.ascontiguousarray(extras, dtype=np.uint64)
    nb = t.size // block_size
    out = np.empty(max(nb, 1), np.uint64)
    n = ctypes.c_int64(0)
    sv = ctypes.c_uint64(int(salt)) if salt is not None else None
    _check(lib().pkv_prefix_block_hashes(_np_ptr(t) if t.size else None, int(t.size), int(block_size),
                                         _np_ptr(e) if e.size else None, int(e.size),
                                         ctypes.byref(sv) if sv is not None else None, _np_ptr(out), nb,
                                         ctypes.byref(n)), "prefix_block_hashes")
    return out[: n.value].copy()


SWAP_OUT, SWAP_IN = 0, 1


def swap_blocks(k_cache, v_cache, desc: CacheDesc, k_host, v_host, pairs, direction: int, stream=None) -> None:
    """k_host, v_host: pinned CPU tensors [NH, Hkv, 16, D] (torch pin_memory
    memory is mapped); pairs: int32 device [n, 2] of (device block, host block)."""
    for t, n in ((k_host, "k_host"), (v_host, "v_host")):
        if t.is_cuda or not t.is_pinned() or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous pinned CPU tensor")
    n = int(pairs.shape[0])
    st = lib().pkv_swap_blocks(_dev_ptr(k_cache, "k_cache"), _dev_ptr(v_cache, "v_cache"), ctypes.byref(desc.c()),
                               k_host.data_ptr(), v_host.data_ptr(), int(k_host.shape[0]),
                               _dev_ptr(pairs, "pairs") if n else None, n, int(direction), _stream(stream))
    _check(st, "swap_blocks")


def get_device_error(stream=None) -> int:
    flags = ctypes.c_uint32(0)
    _check(lib().pkv_get_device_error(ctypes.byref(flags), _stream(stream)), "get_device_error")
    return int(flags.value)


def check_wait_timeout(which: int, stream=None) -> None:
    """Enqueues the library's check of its bounded waits: one CTA waits on a
    barrier nothing arrives at (which 0: the decode copy-pipeline wait, 1:
    the prefill tensor-core pipeline wait) until the wait gives up and sets
    DEVERR_TIMEOUT."""
    _check(lib().pkv_check_wait_timeout(int(which), _stream(stream)), "check_wait_timeout")


# ------------------------------------------------------------ host allocator
def _np_ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


class Allocator:
    """Host block allocator (C++): free list, reference counts, fork / append
    with copy-on-write / free."""

    def __init__(self, num_blocks: int, block_size: int = 16, free_order=None):
        self._order = None
        ptr = None
        if free_order is not None:
            self._order = np.ascontiguousarray(free_order, dtype=np.int32)
            ptr = _np_ptr(self._order)
        self._h = lib().pkv_alloc_create(int(num_blocks), int(block_size), ptr)
        if not self._h:
            raise PagedKVError(ERR_INVALID, "alloc_create")
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)

    def close(self):
        if self._h:
            lib().pkv_alloc_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def seq_new(self, seq: int, num_tokens: int) -> None:
        _check(lib().pkv_alloc_seq_new(self._h, seq, num_tokens), "alloc_seq_new")

    def fork(self, parent: int, child: int) -> None:
        _check(lib().pkv_alloc_fork(self._h, parent, child), "alloc_fork")

    def append_slot(self, seq: int):
        slot, cs, cd = ctypes.c_int64(), ctypes.c_int32(), ctypes.c_int32()
        _check(lib().pkv_alloc_append_slot(self._h, seq, ctypes.byref(slot), ctypes.byref(cs), ctypes.byref(cd)),
               "alloc_append_slot")
        return slot.value, (None if cs.value < 0 else (cs.value, cd.value))

    def extend(self, seq: int, num_tokens: int) -> None:
        _check(lib().pkv_alloc_seq_extend(self._h, seq, num_tokens), "alloc_seq_extend")

    def free(self, seq: int) -> None:
        _check(lib().pkv_alloc_free(self._h, seq), "alloc_free")

    def append_batch(self, seq_ids):
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        n = ids.shape[0]
        slots = np.empty(n, np.int64)
        pairs = np.empty((max(n, 1), 2), np.int32)
        npairs = ctypes.c_int32(0)
        _check(lib().pkv_alloc_append_batch(self._h, _np_ptr(ids), n, _np_ptr(slots), _np_ptr(pairs), max(n, 1),
                                            ctypes.byref(npairs)), "alloc_append_batch")
        return slots, pairs[: npairs.value].copy()

    def append_tokens(self, seq_ids, counts):
        """Reserves counts[i] new token slots for seq_ids[i] (chunked
        prefill); returns (slots [sum counts], copy-on-write pairs [n, 2])."""
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        cnt = np.ascontiguousarray(counts, dtype=np.int32)
        n = ids.shape[0]
        if cnt.shape != (n,):
            raise ValueError("seq_ids and counts differ in length")
        total = int(cnt.sum()) if n else 0
        slots = np.empty(max(total, 1), np.int64)
        pairs = np.empty((max(n, 1), 2), np.int32)
        npairs = ctypes.c_int32(0)
        _check(lib().pkv_alloc_append_tokens(self._h, _np_ptr(ids), _np_ptr(cnt), n, _np_ptr(slots), total,
                                             _np_ptr(pairs), max(n, 1), ctypes.byref(npairs)), "alloc_append_tokens")
        return slots[:total].copy(), pairs[: npairs.value].copy()

    # -- automatic prefix caching
    def lookup(self, hashes) -> int:
        h = np.ascontiguousarray(hashes, dtype=np.uint64)
        k = lib().pkv_alloc_lookup(self._h, _np_ptr(h), int(h.shape[0]))
        if k < 0:
            raise PagedKVError(ERR_INVALID, "alloc_lookup")
        return int(k)

    def seq_new_prefix(self, seq: int, hashes, num_tokens: int) -> int:
        """New sequence sharing its cached leading blocks; returns their count."""
        h = np.ascontiguousarray(hashes, dtype=np.uint64)
        hits = ctypes.c_int32(0)
        _check(lib().pkv_alloc_seq_new_prefix(self._h, int(seq), _np_ptr(h), int(h.shape[0]), int(num_tokens),
                                              ctypes.byref(hits)), "alloc_seq_new_prefix")
        return int(hits.value)

    def commit(self, seq: int, hashes) -> int:
        h = np.ascontiguousarray(hashes, dtype=np.uint64)
        c = ctypes.c_int32(0)
        _check(lib().pkv_alloc_commit(self._h, int(seq), _np_ptr(h), int(h.shape[0]), ctypes.byref(c)),
               "alloc_commit")
        return int(c.value)

    def num_cached(self) -> int:
        return int(lib().pkv_alloc_num_cached(self._h))

    def block_hash_of(self, block: int):
        out = ctypes.c_uint64(0)
        r = lib().pkv_alloc_block_hash_of(self._h, int(block), ctypes.byref(out))
        if r < 0:
            raise PagedKVError(ERR_INVALID, "alloc_block_hash_of")
        return int(out.value) if r else None

    def reset_prefix_cache(self) -> None:
        lib().pkv_alloc_reset_prefix_cache(self._h)

    def export(self, seq_ids, max_blocks: int):
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        n = ids.shape[0]
        tables = np.empty((n, max_blocks), np.int32)
        lens = np.empty(n, np.int32)
        _check(lib().pkv_alloc_export(self._h, _np_ptr(ids), n, _np_ptr(tables), max_blocks, _np_ptr(lens)),
               "alloc_export")
        return tables, lens

    def block_table(self, seq: int):
        n = ctypes.c_int32(0)
        cap = self.num_blocks
        out = np.empty(max(cap, 1), np.int32)
        _check(lib().pkv_alloc_block_table(self._h, seq, _np_ptr(out), cap, ctypes.byref(n)), "alloc_block_table")
        return out[: n.value].tolist()

    def seq_len(self, seq: int) -> int:
        n = ctypes.c_int64(0)
        _check(lib().pkv_alloc_seq_len(self._h, seq, ctypes.byref(n)), "alloc_seq_len")
        return n.value

    def refcount(self, block: int) -> int:
        return int(lib().pkv_alloc_refcount(self._h, block))

    def num_free(self) -> int:
        return int(lib().pkv_alloc_num_free(self._h))

    def num_seqs(self) -> int:
        return int(lib().pkv_alloc_num_seqs(self._h))

    def prefix_groups(self, seq_ids, min_blocks: int = 16) -> PrefixGroups:
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        n = ids.shape[0]
        sg = np.empty(max(n, 1), np.int32)
        gb = np.empty(max(n, 1), np.int32)
        go = np.empty(n + 1, np.int32)
        gm = np.empty(max(n, 1), np.int32)
        ng, mm, mb = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
        _check(lib().pkv_alloc_prefix_groups(self._h, _np_ptr(ids), n, int(min_blocks), _np_ptr(sg), _np_ptr(gb),
                                             _np_ptr(go), _np_ptr(gm), ctypes.byref(ng), ctypes.byref(mm),
                                             ctypes.byref(mb)), "alloc_prefix_groups")
        k = ng.value
        return PrefixGroups(sg[:n].copy(), gb[:k].copy(), go[:k + 1].copy(), gm[:go[k] if k else 0].copy(),
                            mm.value, mb.value)

    def swap_out(self, host: "Allocator", seq: int) -> np.ndarray:
        """Moves seq to the host allocator; returns (device, host) block pairs."""
        pairs = np.empty((max(self.num_blocks, 1), 2), np.int32)
        n = ctypes.c_int32(0)
        _check(lib().pkv_alloc_swap_out(self._h, host._h, seq, _np_ptr(pairs), pairs.shape[0], ctypes.byref(n)),
               "alloc_swap_out")
        return pairs[: n.value].copy()

    def swap_in(self, host: "Allocator", seq: int) -> np.ndarray:
        """Moves seq back from the host allocator; returns (device, host) pairs."""
        pairs = np.empty((max(host.num_blocks, 1), 2), np.int32)
        n = ctypes.c_int32(0)
        _check(lib().pkv_alloc_swap_in(self._h, host._h, seq, _np_ptr(pairs), pairs.shape[0], ctypes.byref(n)),
               "alloc_swap_in")
        return pairs[: n.value].copy()

    def fail_after(self, k: int) -> None:
        lib().pkv_alloc_fail_after(self._h, int(k))


def apply_setup(alloc: Allocator, ops) -> None:
    """Runs an allocator script of ("new", seq, n) / ("fork", parent, child) /
    ("extend", seq, n) / ("free", seq) operations."""
    for op in ops:
        if op[0] == "new":
            alloc.seq_new(op[1], op[2])
        elif op[0] == "fork":
            alloc.fork(op[1], op[2])
        elif op[0] == "extend":
            alloc.extend(op[1], op[2])
        elif op[0] == "free":
            alloc.free(op[1])
        else:
            raise ValueError(f"unknown allocator op {op[0]!r}")
