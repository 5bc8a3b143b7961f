"""CPU oracle for the paged KV cache hot path (float64).

TEST INFRASTRUCTURE ONLY: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product library never loads it, and it never loads the product
library: the two share no code (see ``pkv_oracle.c`` for the formats, each
decoded from its published definition).

``pkv_oracle.c`` holds the arithmetic (plain loops, float64, OpenMP over the
(sequence, query head) rows); this module only marshals numpy arrays into it.
``allocator_model.py`` is an independent pure-Python model of the host block
allocator.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

F16, BF16, E4M3 = 0, 1, 2
DTYPE_CODE = {"f16": F16, "bf16": BF16, "e4m3": E4M3}


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` with gcc (OpenMP if the compiler has it)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    base = ["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-Wall", _SRC, "-o", _LIB, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True)
    return _LIB


_lib = None


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = bind(ctypes.CDLL(_LIB))
    return _lib


def bind(lib):
    """Declares the C signatures on a loaded oracle library and returns it."""
    if True:
        P = ctypes.c_void_p
        i32, i64, f64, f32 = ctypes.c_int, ctypes.c_int64, ctypes.c_double, ctypes.c_float
        lib.pkvo_f16_to_double.argtypes = [ctypes.c_uint16]
        lib.pkvo_f16_to_double.restype = f64
        lib.pkvo_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.pkvo_bf16_to_double.restype = f64
        lib.pkvo_e4m3_to_double.argtypes = [ctypes.c_uint8]
        lib.pkvo_e4m3_to_double.restype = f64
        lib.pkvo_e4m3_encode.argtypes = [f32]
        lib.pkvo_e4m3_encode.restype = ctypes.c_uint8
        lib.pkvo_paged_decode.argtypes = [P, i32, i32, i32, P, P, i32, i32, i32, i32, i32, f64, f64,
                                          P, i32, P, f64, P]
        lib.pkvo_paged_decode.restype = i32
        lib.pkvo_paged_decode_partials.argtypes = [P, i32, i32, i32, P, P, i32, i32, i32, i32, i32,
                                                   f64, f64, P, i32, P, f64, i32, i32, P, P, P]
        lib.pkvo_paged_decode_partials.restype = i32
        lib.pkvo_paged_prefill.argtypes = [P, i32, i32, i32, i32, P, P, P, i32, i32, i32, i32, i32, f64, f64,
                                           P, i32, P, f64, P]
        lib.pkvo_paged_prefill.restype = i32
        lib.pkvo_lse_merge.argtypes = [i64, i32, i32, P, P, P, P]
        lib.pkvo_lse_merge.restype = None
        lib.pkvo_append.argtypes = [P, P, i32, i32, P, P, P, i32, i32, i32, i32, i32, f32, f32]
        lib.pkvo_append.restype = i32
        lib.pkvo_copy_blocks.argtypes = [P, P, i32, i32, i32, i32, i32, P, i32]
        lib.pkvo_copy_blocks.restype = i32
        lib.pkvo_num_threads.argtypes = []
        lib.pkvo_num_threads.restype = i32
        lib.pkvo_set_num_threads.argtypes = [i32]
        lib.pkvo_set_num_threads.restype = None
    return lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return int(_load().pkvo_num_threads())


def set_num_threads(n: int) -> None:
    """Threads of the oracle's parallel loops from now on (timing only)."""
    _load().pkvo_set_num_threads(int(n))


# ----------------------------------------------------------------- formats
def f16_to_double(bits: int) -> float:
    return float(_load().pkvo_f16_to_double(int(bits)))


def bf16_to_double(bits: int) -> float:
    return float(_load().pkvo_bf16_to_double(int(bits)))


def e4m3_to_double(code: int) -> float:
    return float(_load().pkvo_e4m3_to_double(int(code)))


def e4m3_encode(x: float) -> int:
    return int(_load().pkvo_e4m3_encode(float(np.float32(x))))


_TABLES: dict = {}


def dequantize(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Element-wise decode of raw storage bits to float64, through a table of
    the oracle's per-code decoder."""
    if dtype not in _TABLES:
        fn = {"f16": f16_to_double, "bf16": bf16_to_double, "e4m3": e4m3_to_double}[dtype]
        n = 256 if dtype == "e4m3" else 65536
        _TABLES[dtype] = np.array([fn(c) for c in range(n)], dtype=np.float64)
    return _TABLES[dtype][np.asarray(bits).astype(np.int64)]


# --------------------------------------------------------------- attention
def paged_decode(q, q_dtype, k_pool, v_pool, kv_dtype, block_tables, seq_lens, scale,
                 k_scale=1.0, v_scale=1.0) -> np.ndarray:
    """float64 out[S, Hq, D] of the plain definition (see pkv_oracle.c).

    q: raw bits [S, Hq, D]; k_pool/v_pool: raw bits [NB, Hkv, b, D];
    block_tables: int32 [S, MB]; seq_lens: int32 [S].
    """
    S, Hq, D = q.shape
    NB, Hkv, b, D2 = k_pool.shape
    assert D == D2 and v_pool.shape == k_pool.shape
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    out = np.zeros((S, Hq, D), dtype=np.float64)
    rc = _load().pkvo_paged_decode(_ptr(q), DTYPE_CODE[q_dtype], S, Hq, _ptr(k_pool), _ptr(v_pool),
                                   DTYPE_CODE[kv_dtype], NB, b, Hkv, D, float(k_scale), float(v_scale),
                                   _ptr(bt), bt.shape[1], _ptr(sl), float(scale), _ptr(out))
    if rc:
        raise ValueError("oracle: invalid argument or block id")
    return out


def paged_prefill(q, q_dtype, query_start, k_pool, v_pool, kv_dtype, block_tables, seq_lens, scale,
                  k_scale=1.0, v_scale=1.0) -> np.ndarray:
    """float64 out[T, Hq, D] of causal paged prefill (see pkv_oracle.c).

    q: raw bits [T, Hq, D]; query_start: int32 [S + 1] (rows of each sequence's
    new tokens); seq_lens: int32 [S], each counting the new tokens.
    """
    T, Hq, D = q.shape
    NB, Hkv, b, D2 = k_pool.shape
    assert D == D2 and v_pool.shape == k_pool.shape
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    qs = np.ascontiguousarray(query_start, dtype=np.int32)
    S = sl.shape[0]
    assert qs.shape == (S + 1,)
    out = np.zeros((T, Hq, D), dtype=np.float64)
    rc = _load().pkvo_paged_prefill(_ptr(np.ascontiguousarray(q)), DTYPE_CODE[q_dtype], T, Hq, S, _ptr(qs),
                                    _ptr(k_pool), _ptr(v_pool), DTYPE_CODE[kv_dtype], NB, b, Hkv, D,
                                    float(k_scale), float(v_scale), _ptr(bt), bt.shape[1] if bt.ndim == 2 else 0,
                                    _ptr(sl), float(scale), _ptr(out))
    if rc:
        raise ValueError("oracle: invalid argument or block id")
    return out


def paged_decode_partials(q, q_dtype, k_pool, v_pool, kv_dtype, block_tables, seq_lens, scale,
                          partition_tokens, num_partitions=None, k_scale=1.0, v_scale=1.0):
    """Split-K partials (m, l, o) of shape [S, Hq, NP], [S, Hq, NP], [S, Hq, NP, D]."""
    S, Hq, D = q.shape
    NB, Hkv, b, _ = k_pool.shape
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    P = int(partition_tokens)
    NP = num_partitions or max(1, max((int(x) + P - 1) // P for x in sl) if S else 1)
    m = np.zeros((S, Hq, NP), np.float64)
    l = np.zeros((S, Hq, NP), np.float64)
    o = np.zeros((S, Hq, NP, D), np.float64)
    rc = _load().pkvo_paged_decode_partials(_ptr(q), DTYPE_CODE[q_dtype], S, Hq, _ptr(k_pool),
                                            _ptr(v_pool), DTYPE_CODE[kv_dtype], NB, b, Hkv, D,
                                            float(k_scale), float(v_scale), _ptr(bt), bt.shape[1],
                                            _ptr(sl), float(scale), P, NP, _ptr(m), _ptr(l), _ptr(o))
    if rc:
        raise ValueError("oracle: invalid argument or block id")
    return m, l, o


def lse_merge(m, l, o) -> np.ndarray:
    """Merge partials from ``paged_decode_partials`` into out[S, Hq, D]."""
    S, Hq, NP, D = o.shape
    m = np.ascontiguousarray(m, np.float64)
    l = np.ascontiguousarray(l, np.float64)
    o = np.ascontiguousarray(o, np.float64)
    out = np.zeros((S, Hq, D), np.float64)
    _load().pkvo_lse_merge(S * Hq, NP, D, _ptr(m), _ptr(l), _ptr(o), _ptr(out))
    return out


# ------------------------------------------------------------ append / copy
def append(k_new, v_new, in_dtype, slot_mapping, k_pool, v_pool, kv_dtype,
           k_scale=1.0, v_scale=1.0) -> None:
    """In-place slot-mapped write into numpy pools (raw bits)."""
    T = k_new.shape[0]
    NB, Hkv, b, D = k_pool.shape
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    rc = _load().pkvo_append(_ptr(k_new), _ptr(v_new), DTYPE_CODE[in_dtype], T, _ptr(sm),
                             _ptr(k_pool), _ptr(v_pool), DTYPE_CODE[kv_dtype], NB, b, Hkv, D,
                             float(np.float32(k_scale)), float(np.float32(v_scale)))
    if rc:
        raise ValueError("oracle: slot outside the pool")


def copy_blocks(k_pool, v_pool, kv_dtype, pairs) -> None:
    """In-place copy-on-write block copy on numpy pools (raw bits)."""
    NB, Hkv, b, D = k_pool.shape
    pr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
    rc = _load().pkvo_copy_blocks(_ptr(k_pool), _ptr(v_pool), DTYPE_CODE[kv_dtype], NB, b, Hkv, D,
                                  _ptr(pr), pr.shape[0])
    if rc:
        raise ValueError("oracle: block id outside the pool")
