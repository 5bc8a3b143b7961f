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


# unit roundoff of the probabilities' 16-bit type in the tensor-core products
P_ROUNDOFF = {"bf16": 2.0 ** -8, "f16": 2.0 ** -11}


def p_rounding_allowance(p_dtype: str, vmax: float) -> float:
    """Error a kernel that rounds the softmax probabilities to a 16-bit MMA
    operand may add when few keys dominate a row: each weight moves by at
    most the unit roundoff u, so the output by at most u * max|V|.  (Rows
    spread over many keys, as with the configs' N(0,1) queries, average it
    out.)"""
    return P_ROUNDOFF[p_dtype] * float(vmax)


def max_error(got: np.ndarray, ref: np.ndarray, out_dtype: str, tol: float) -> float:
    """Max-abs error against the float64 oracle, with the allowance of an
    output whose format cannot meet the absolute bound: where one unit in
    the last place of the output format at the oracle value exceeds `tol`
    (|out| >= 2 for bf16 at 1e-2, >= 4 for f16 at 2e-3), that unit is the
    bound, so even the correctly rounded result may differ by up to it.
    Returns a number to compare with `tol`: max(|got - ref| - max(0, ulp - tol))."""
    if ref.size == 0:
        return 0.0
    slack = np.maximum(output_ulp(ref, out_dtype) - tol, 0.0)
    return float(np.max(np.abs(got - ref) - slack))


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
