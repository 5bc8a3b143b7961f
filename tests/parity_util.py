"""Shared helpers for the GPU parity tests: run one decode step through the C
ABI and recompute it with the oracle (independent allocator model, float64
attention, byte-level append / copy)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from oracle.allocator_model import AllocatorModel

TOL = {"f16": 2e-3, "bf16": 1e-2, "e4m3": 1e-2}
# explicit significand bits of the 16-bit output formats
_MANT = {"f16": 10, "bf16": 7}


def output_ulp(ref: np.ndarray, out_dtype: str) -> np.ndarray:
    """One unit in the last place of the output format at |ref| (normal range)."""
    a = np.maximum(np.abs(ref), np.finfo(np.float64).tiny)
    return np.exp2(np.floor(np.log2(a)) - _MANT[out_dtype])


# Bound on the kernels' float32 error before the final rounding, as a
# fraction of the largest |value| the output averages: every kernel forms
# sum_t p_t v_t / sum_t p_t with float32 products and sums (the tensor-core
# kernels feed P V with P split into a 16-bit head and a 16-bit tail, so the
# probabilities keep 16 or more significant bits), exp2 within 2^-22
# relative, and, at the tested lengths (up to 32768 tokens), fewer than
# 2^9 + 16 dependent float32 additions per output element (one per block of
# a warp's range, the cross-warp and split-K merges, the 16 products of an
# MMA): (2^9 + 16) * 2^-24 < 2^-14.
FP32_TERM = 2.0 ** -14


def relaxed_bound(ref: np.ndarray, out_dtype: str, tol: float, vmax: float) -> np.ndarray:
    """Per-element bound on |got - ref|.  The output is rounded once to q's
    16-bit format; where half a unit in the last place of that format at the
    exact value exceeds `tol` (bf16 |out| >= 4 at 1e-2, f16 |out| >= 8 at
    2e-3) not even the correctly rounded result meets `tol`, and the bound
    is that half unit plus twice the float32 error allowance (rounding a
    value e away from ref lands within half an ulp + 2e of ref).  Everywhere
    else the bound is `tol` itself."""
    half = 0.5 * output_ulp(ref, out_dtype)
    return np.where(half > tol, half + 2.0 * FP32_TERM * vmax, tol)


def max_error(got: np.ndarray, ref: np.ndarray, out_dtype: str, tol: float, vmax: float | None = None) -> float:
    """Max-abs error against the float64 oracle, shifted so that it compares
    with `tol`: max(|got - ref| - (relaxed_bound - tol)).  `vmax`: the largest
    |V| the outputs average (default: the largest |ref|, a lower bound of it,
    which only makes the check stricter)."""
    if ref.size == 0:
        return 0.0
    if vmax is None:
        vmax = float(np.max(np.abs(ref)))
    return float(np.max(np.abs(got - ref) - (relaxed_bound(ref, out_dtype, tol, vmax) - tol)))


def host_bits(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu()
    if t.element_size() == 2:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.view(torch.uint8).numpy()


def model_step(wl):
    """Replays the workload's allocator script in the Python model."""
    m = AllocatorModel(wl.NB, wl.b, wl.free_order)
    for op in wl.setup:
        if op[0] == "new":
            m.seq_new(op[1], op[2])
        elif op[0] == "fork":
            m.fork(op[1], op[2])
        elif op[0] == "extend":
            for _ in range(op[2]):
                assert m.append_slot(op[1])[1] is None
        elif op[0] == "free":
            m.free_seq(op[1])
    slots = np.full(wl.S, -1, np.int64)
    pairs = []
    for s in wl.step_seqs:
        slot, cow = m.append_slot(s)
        slots[s] = slot
        if cow:
            pairs.append(cow)
    MB = wl.max_blocks
    tables = np.full((wl.S, MB), -1, np.int32)
    lens = np.zeros(wl.S, np.int32)
    for s in range(wl.S):
        t = m.block_table(s)
        tables[s, :len(t)] = t
        lens[s] = m.lens[s]
    return slots, np.array(pairs, np.int32).reshape(-1, 2), tables, lens


def oracle_pools(wl, pairs, slots):
    kp, vp = wl.k_pool.copy(), wl.v_pool.copy()
    if len(pairs):
        oracle.copy_blocks(kp, vp, wl.kv_dtype, pairs)
    oracle.append(wl.k_new, wl.v_new, wl.in_dtype, slots, kp, vp, wl.kv_dtype, wl.k_scale, wl.v_scale)
    return kp, vp


def check_step(step, rows=None, check_pools=True):
    """Compares one executed DecodeStep with the oracle.  ``rows``: subset of
    batch rows whose attention output is recomputed (None = all).  Returns
    (max-abs error with the output-format allowance of ``max_error``, max
    |oracle|)."""
    wl = step.wl
    slots, pairs, tables, lens = model_step(wl)
    # host bookkeeping: bit-exact against the independent model
    assert np.array_equal(step.slots, slots)
    assert np.array_equal(step.pairs.reshape(-1, 2), pairs)
    assert np.array_equal(step.tables, tables)
    assert np.array_equal(step.seq_lens, lens)
    kp, vp = oracle_pools(wl, pairs, slots)
    if check_pools:
        assert np.array_equal(host_bits(step.k_cache), kp), "K pool differs from the oracle"
        assert np.array_equal(host_bits(step.v_cache), vp), "V pool differs from the oracle"
    rows = np.arange(wl.S) if rows is None else np.asarray(rows)
    ref = oracle.paged_decode(np.ascontiguousarray(wl.q[rows]), wl.q_dtype, kp, vp, wl.kv_dtype,
                              np.ascontiguousarray(tables[rows]), np.ascontiguousarray(lens[rows]), wl.scale,
                              wl.k_scale, wl.v_scale)
    got = oracle.dequantize(host_bits(step.out)[rows], wl.q_dtype)
    assert np.all(np.isfinite(got))
    err = max_error(got, ref, wl.q_dtype, TOL[wl.kv_dtype])
    return err, float(np.max(np.abs(ref))) if ref.size else 0.0
