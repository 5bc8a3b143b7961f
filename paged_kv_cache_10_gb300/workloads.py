"""Seeded synthetic workloads for paged decode attention.

This module only draws inputs: element values, a free-list order for the
block allocator and a script of allocator operations (new / fork / extend /
free, then the step's batch of appends).  It holds none of the method's
arithmetic -- no slot or block-table computation, no attention, no encoding
logic of its own -- so both the CUDA path (``bench.py`` and the GPU tests) and
the float64 oracle (tests) consume exactly the same draws.

Values are N(0, 1) drawn with numpy's PCG64 in fixed 16 Mi-element chunks
(child seeds from one ``SeedSequence``), so the result does not depend on the
number of threads used; they are rounded to the storage type by torch's CPU
casts (round to nearest even).  fp8 E4M3 pools store ``x / scale`` with one
per-tensor scale ``max|x| / 448`` so that the N(0, 1) source fills the E4M3
range.

The five named workloads follow the sizes the pages' PagedAttention
description implies (16-token blocks, block tables over a shared pool,
prefix sharing with reference counts) on Llama-shaped heads:

  tiny_fp16       4 seqs, lens {1,17,50,64}, 4/4 heads, D 64, fp16, 64-block pool
  llama7b_mha     64 seqs, lens U[512,4096], 32/32 heads, D 128, bf16
  llama3_8b_gqa   256 seqs, lens U[128,2048], 32/8 heads, D 128, bf16
  longctx_fp8     8 seqs x 32768 tokens, 64/8 heads, D 128, fp8 E4M3 KV, bf16 q,
                  512-token partitions, 5 % of the pool free
  prefix_share    64 parallel-sampling pairs over one 2048-token prefix
                  (refcount 128); each pair shares a U[0,512] suffix, every
                  sequence appends one token (copy-on-write where the pair's
                  last block is partial); 32/8 heads, D 128, bf16

In every decode workload each sequence appends exactly one new token in the
step and ``seq_len`` counts it.

Prefill workloads (``PREFILL``) append a chunk of new tokens per sequence and
run causal attention for them:

  prefill_chunked_gqa  8 chunks of 512 tokens after U[0,3584] tokens of
                       context each (a 4096-token batch), 32/8 heads, bf16
  prefill_prompt_gqa   4 whole prompts of 4096 tokens, 32/8 heads, bf16
  prefill_prompt_mha   4 whole prompts of 2048 tokens, 32/32 heads, bf16
  prefill_chunked_gqa_fp8  prefill_chunked_gqa over an fp8 E4M3 cache with
                       per-tensor scales (bf16 queries and output)
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np
import torch

BLOCK_SIZE = 16
_CHUNK = 16 << 20

_TORCH_DT = {"f16": torch.float16, "bf16": torch.bfloat16}


@dataclass
class Workload:
    name: str
    S: int
    Hq: int
    Hkv: int
    D: int
    NB: int
    q_dtype: str          # "f16" | "bf16"
    kv_dtype: str         # "f16" | "bf16" | "e4m3"
    in_dtype: str         # dtype of the appended k/v ("bf16" for an fp8 cache)
    scale: float
    k_scale: float
    v_scale: float
    partition_tokens: int  # 0 = let the library choose
    q: np.ndarray          # raw bits [S, Hq, D]
    k_pool: np.ndarray     # raw bits [NB, Hkv, b, D]
    v_pool: np.ndarray
    k_new: np.ndarray      # raw bits [S, Hkv, D], one token per sequence
    v_new: np.ndarray
    free_order: np.ndarray  # int32 [NB], allocation takes from the end
    setup: list = field(default_factory=list)   # [("new", seq, n) | ("fork", p, c) | ("extend", seq, n) | ("free", seq)]
    step_seqs: list = field(default_factory=list)  # sequence ids of the batch, in order
    seq_lens: list = field(default_factory=list)   # intended seq_len per batch row (counts the new token)
    b: int = BLOCK_SIZE

    @property
    def max_seq_len(self) -> int:
        return max(self.seq_lens) if self.seq_lens else 0

    @property
    def max_blocks(self) -> int:
        return max(1, -(-self.max_seq_len // self.b))

    def kv_elem_bytes(self) -> int:
        return 1 if self.kv_dtype == "e4m3" else 2


def _normal_f32(seed_seq: np.random.SeedSequence, n: int, threads: int = 16) -> np.ndarray:
    out = np.empty(n, np.float32)
    nch = max(1, -(-n // _CHUNK))
    kids = seed_seq.spawn(nch)

    def work(i):
        lo, hi = i * _CHUNK, min(n, (i + 1) * _CHUNK)
        g = np.random.Generator(np.random.PCG64(kids[i]))
        g.standard_normal(hi - lo, dtype=np.float32, out=out[lo:hi])

    with ThreadPoolExecutor(min(threads, nch)) as ex:
        list(ex.map(work, range(nch)))
    return out


def _to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float32 -> f16/bf16 storage bits (uint16), chunked."""
    out = np.empty(x.shape, np.uint16)
    xf, of = x.reshape(-1), out.reshape(-1)
    for lo in range(0, xf.size, _CHUNK):
        hi = min(xf.size, lo + _CHUNK)
        t = torch.from_numpy(xf[lo:hi]).to(_TORCH_DT[dtype])
        of[lo:hi] = t.view(torch.int16).numpy().view(np.uint16)
    return out


def _to_e4m3(x: np.ndarray, scale: float) -> np.ndarray:
    out = np.empty(x.shape, np.uint8)
    xf, of = x.reshape(-1), out.reshape(-1)
    s = torch.tensor(scale, dtype=torch.float32)
    for lo in range(0, xf.size, _CHUNK):
        hi = min(xf.size, lo + _CHUNK)
        t = (torch.from_numpy(xf[lo:hi]) / s).to(torch.float8_e4m3fn)
        of[lo:hi] = t.view(torch.uint8).numpy()
    return out


def _values(ss, shape, dtype):
    """N(0,1) values rounded to ``dtype`` storage bits; returns (bits, scale)."""
    n = int(np.prod(shape))
    x = _normal_f32(ss, n).reshape(shape)
    if dtype == "e4m3":
        scale = float(np.float32(np.abs(x).max()) / np.float32(448.0))
        return _to_e4m3(x, scale), scale
    return _to_bits(x, dtype), 1.0


def build(name, seed, S, Hq, Hkv, D, NB, q_dtype, kv_dtype, setup, step_seqs, seq_lens,
          partition_tokens=0, in_dtype=None, rng=None) -> Workload:
    """Draws the values for a workload whose allocator script is given."""
    ss = np.random.SeedSequence(seed)
    s_q, s_k, s_v, s_kn, s_vn, s_free = ss.spawn(6)
    in_dtype = in_dtype or (kv_dtype if kv_dtype != "e4m3" else "bf16")
    b = BLOCK_SIZE
    k_pool, k_scale = _values(s_k, (NB, Hkv, b, D), kv_dtype)
    v_pool, v_scale = _values(s_v, (NB, Hkv, b, D), kv_dtype)
    q, _ = _values(s_q, (S, Hq, D), q_dtype)
    k_new, _ = _values(s_kn, (S, Hkv, D), in_dtype)
    v_new, _ = _values(s_vn, (S, Hkv, D), in_dtype)
    free_order = np.random.Generator(np.random.PCG64(s_free)).permutation(NB).astype(np.int32)
    return Workload(name=name, S=S, Hq=Hq, Hkv=Hkv, D=D, NB=NB, q_dtype=q_dtype, kv_dtype=kv_dtype,
                    in_dtype=in_dtype, scale=1.0 / math.sqrt(D), k_scale=k_scale, v_scale=v_scale,
                    partition_tokens=partition_tokens, q=q, k_pool=k_pool, v_pool=v_pool,
                    k_new=k_new, v_new=v_new, free_order=free_order, setup=setup,
                    step_seqs=list(step_seqs), seq_lens=list(seq_lens))


def _independent(lens):
    """Setup script: every sequence prefilled with len-1 tokens, then one append each."""
    setup = [("new", s, int(L) - 1) for s, L in enumerate(lens)]
    return setup, list(range(len(lens))), [int(x) for x in lens]


def _blocks(n):
    return -(-int(n) // BLOCK_SIZE)


def tiny_fp16(seed=1001) -> Workload:
    lens = [1, 17, 50, 64]
    setup, step, sl = _independent(lens)
    return build("tiny_fp16", seed, 4, 4, 4, 64, 64, "f16", "f16", setup, step, sl)


def llama7b_mha(seed=1002) -> Workload:
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed).spawn(7)[6]))
    lens = rng.integers(512, 4096, size=64, endpoint=True)
    U = sum(_blocks(L) for L in lens)
    NB = U + math.ceil(0.10 * U)
    setup, step, sl = _independent(lens)
    return build("llama7b_mha", seed, 64, 32, 32, 128, NB, "bf16", "bf16", setup, step, sl)


def llama3_8b_gqa(seed=1003) -> Workload:
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed).spawn(7)[6]))
    lens = rng.integers(128, 2048, size=256, endpoint=True)
    U = sum(_blocks(L) for L in lens)
    NB = U + math.ceil(0.10 * U)
    setup, step, sl = _independent(lens)
    return build("llama3_8b_gqa", seed, 256, 32, 8, 128, NB, "bf16", "bf16", setup, step, sl)


def longctx_fp8(seed=1004) -> Workload:
    lens = [32768] * 8
    U = sum(_blocks(L) for L in lens)
    NB = math.ceil(U / 0.95)
    setup, step, sl = _independent(lens)
    return build("longctx_fp8", seed, 8, 64, 8, 128, NB, "bf16", "e4m3", setup, step, sl,
                 partition_tokens=512)


def prefix_share(seed=1005, pairs=64, prefix=2048, literal=False, kv_dtype="bf16") -> Workload:
    """Parallel sampling over one shared prefix.

    Default: ``pairs`` pairs (2j, 2j+1); both members share the prefix and a
    pair suffix of U[0,512] tokens, so the first member's append hits a shared
    partial block (copy-on-write) unless the suffix is a whole number of
    blocks.  ``literal=True``: 2*pairs sequences with independent suffixes
    (no block but the prefix is shared, so no copy-on-write).  kv_dtype:
    the pool's element type (queries stay bf16; an fp8 pool takes per-tensor
    scales from its values)."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed).spawn(7)[6]))
    S = 2 * pairs
    T = 1 << 30  # template sequence id, freed before the step
    setup = [("new", T, prefix)]
    lens = []
    if literal:
        suf = rng.integers(0, 512, size=S, endpoint=True)
        for s in range(S):
            setup += [("fork", T, s), ("extend", s, int(suf[s]))]
            lens.append(prefix + int(suf[s]) + 1)
        nblk = _blocks(prefix) + sum(_blocks(prefix + x + 1) - _blocks(prefix) for x in suf)
    else:
        suf = rng.integers(0, 512, size=pairs, endpoint=True)
        for j in range(pairs):
            setup += [("fork", T, 2 * j), ("extend", 2 * j, int(suf[j])), ("fork", 2 * j, 2 * j + 1)]
            lens += [prefix + int(suf[j]) + 1] * 2
        nblk = _blocks(prefix) + sum(_blocks(x) + 2 for x in suf)
    setup.append(("free", T))
    NB = nblk + math.ceil(0.10 * nblk)
    name = ("prefix_share_literal" if literal else "prefix_share") + ("" if kv_dtype == "bf16" else "_" + kv_dtype)
    return build(name, seed, S, 32, 8, 128, NB, "bf16", kv_dtype, setup, list(range(S)), lens)


def custom(name, seed, lens, Hq, Hkv, D, kv_dtype="bf16", q_dtype=None, NB=None,
           partition_tokens=0) -> Workload:
    """Independent sequences of the given final lengths (a length-0 sequence
    gets no append: it stays empty)."""
    q_dtype = q_dtype or ("bf16" if kv_dtype == "e4m3" else kv_dtype)
    setup, step, sl = [], [], []
    for s, L in enumerate(lens):
        L = int(L)
        setup.append(("new", s, max(L - 1, 0)))
        sl.append(L)
    step = [s for s, L in enumerate(lens) if int(L) > 0]
    need = sum(_blocks(L) for L in lens)
    NB = NB or max(4, need + math.ceil(0.25 * need))
    return build(name, seed, len(lens), Hq, Hkv, D, NB, q_dtype, kv_dtype, setup, step, sl,
                 partition_tokens=partition_tokens)


def fork_groups(name, seed, groups, singles, Hq, Hkv, D=128, kv_dtype="bf16", partition_tokens=0,
                q_dtype=None) -> Workload:
    """Fork trees: for each (prefix_tokens, members) in ``groups`` a template
    sequence of prefix_tokens (a multiple of 16) is forked into ``members``
    sequences, each extended by its own U[0, 300] tokens; ``singles``
    independent sequences of U[1, 600] tokens join the batch.  Every sequence
    appends one token in the step."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed).spawn(7)[6]))
    setup, lens, s = [], [], 0
    need = 0
    for gi, (prefix, members) in enumerate(groups):
        assert prefix % BLOCK_SIZE == 0
        T = (1 << 30) + gi
        setup.append(("new", T, prefix))
        need += _blocks(prefix)
        for _ in range(members):
            suf = int(rng.integers(0, 300, endpoint=True))
            setup += [("fork", T, s), ("extend", s, suf)]
            lens.append(prefix + suf + 1)
            need += _blocks(prefix + suf + 1) - _blocks(prefix) + 1
            s += 1
        setup.append(("free", T))
    for _ in range(singles):
        L = int(rng.integers(1, 600, endpoint=True))
        setup.append(("new", s, L - 1))
        lens.append(L)
        need += _blocks(L) + 1
        s += 1
    NB = need + math.ceil(0.25 * need)
    q_dtype = q_dtype or ("bf16" if kv_dtype == "e4m3" else kv_dtype)
    return build(name, seed, s, Hq, Hkv, D, NB, q_dtype, kv_dtype, setup, list(range(s)), lens,
                 partition_tokens=partition_tokens)


@dataclass
class PrefillWorkload:
    """Inputs of one paged (chunked) prefill step: sequence s already holds
    ctx[s] tokens in the pool (allocator script "new"), then appends qlens[s]
    new tokens (k_new / v_new rows, packed sequence after sequence) and runs
    causal attention for those rows (q rows, packed the same way)."""
    name: str
    S: int
    Hq: int
    Hkv: int
    D: int
    NB: int
    dtype: str            # "f16" | "bf16" (q, appended k/v, output; the pool too unless kv_dtype says)
    scale: float
    ctx: list
    qlens: list
    q: np.ndarray          # raw bits [T, Hq, D]
    k_pool: np.ndarray     # raw bits [NB, Hkv, b, D]
    v_pool: np.ndarray
    k_new: np.ndarray      # raw bits [T, Hkv, D]
    v_new: np.ndarray
    free_order: np.ndarray
    b: int = BLOCK_SIZE
    kv_dtype: str = ""     # pool element type; "" = dtype; "e4m3" with the per-tensor scales below
    k_scale: float = 1.0
    v_scale: float = 1.0

    def __post_init__(self):
        self.kv_dtype = self.kv_dtype or self.dtype

    @property
    def T(self) -> int:
        return int(sum(self.qlens))

    @property
    def seq_lens(self) -> list:
        return [int(c) + int(n) for c, n in zip(self.ctx, self.qlens)]

    @property
    def max_blocks(self) -> int:
        return max(1, max(_blocks(L) for L in self.seq_lens))

    @property
    def max_query_len(self) -> int:
        return max(self.qlens) if self.qlens else 0


def prefill(name, seed, ctx, qlens, Hq, Hkv, D=128, dtype="bf16", NB=None, kv_dtype=None) -> PrefillWorkload:
    """kv_dtype: the pool's element type (default dtype); for "e4m3" each pool
    draws its per-tensor scale from its values (max |x| / 448) and the new
    tokens, drawn in dtype, are encoded with it by the append."""
    ss = np.random.SeedSequence(seed)
    s_q, s_k, s_v, s_kn, s_vn, s_free = ss.spawn(6)
    ctx = [int(c) for c in ctx]
    qlens = [int(n) for n in qlens]
    T = sum(qlens)
    kv_dtype = kv_dtype or dtype
    need = sum(_blocks(c + n) for c, n in zip(ctx, qlens))
    NB = NB or max(4, need + math.ceil(0.10 * need))
    k_pool, k_scale = _values(s_k, (NB, Hkv, BLOCK_SIZE, D), kv_dtype)
    v_pool, v_scale = _values(s_v, (NB, Hkv, BLOCK_SIZE, D), kv_dtype)
    q, _ = _values(s_q, (T, Hq, D), dtype)
    k_new, _ = _values(s_kn, (T, Hkv, D), dtype)
    v_new, _ = _values(s_vn, (T, Hkv, D), dtype)
    free_order = np.random.Generator(np.random.PCG64(s_free)).permutation(NB).astype(np.int32)
    return PrefillWorkload(name=name, S=len(ctx), Hq=Hq, Hkv=Hkv, D=D, NB=NB, dtype=dtype, scale=1.0 / math.sqrt(D),
                           ctx=ctx, qlens=qlens, q=q, k_pool=k_pool, v_pool=v_pool, k_new=k_new, v_new=v_new,
                           free_order=free_order, kv_dtype=kv_dtype, k_scale=k_scale, v_scale=v_scale)


def prefill_chunked_gqa(seed=1010) -> PrefillWorkload:
    """Chunked prefill, Llama-3-8B-shaped heads (32 / 8, D 128, bf16): a
    4096-token batch of 8 chunks of 512 tokens, each continuing a prompt with
    U[0, 3584] tokens already in the pool."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed).spawn(7)[6]))
    ctx = rng.integers(0, 3584, size=8, endpoint=True)
    return prefill("prefill_chunked_gqa", seed, ctx, [512] * 8, 32, 8)


def prefill_prompt_gqa(seed=1011) -> PrefillWorkload:
    """Whole-prompt prefill, Llama-3-8B-shaped heads: 4 prompts of 4096 tokens."""
    return prefill("prefill_prompt_gqa", seed, [0] * 4, [4096] * 4, 32, 8)


def prefill_prompt_mha(seed=1012) -> PrefillWorkload:
    """Whole-prompt prefill, Llama-7B-shaped heads (32 / 32, D 128, bf16): 4
    prompts of 2048 tokens."""
    return prefill("prefill_prompt_mha", seed, [0] * 4, [2048] * 4, 32, 32)


def prefill_chunked_gqa_fp8(seed=1010) -> PrefillWorkload:
    """prefill_chunked_gqa (same seed, context lengths and queries) over an fp8 E4M3 cache
    (per-tensor scales), bf16 queries and output."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed).spawn(7)[6]))
    ctx = rng.integers(0, 3584, size=8, endpoint=True)
    return prefill("prefill_chunked_gqa_fp8", seed, ctx, [512] * 8, 32, 8, kv_dtype="e4m3")


PREFILL = {
    "prefill_chunked_gqa": prefill_chunked_gqa,
    "prefill_chunked_gqa_fp8": prefill_chunked_gqa_fp8,
    "prefill_prompt_gqa": prefill_prompt_gqa,
    "prefill_prompt_mha": prefill_prompt_mha,
}


NAMED = {
    "tiny_fp16": tiny_fp16,
    "llama7b_mha": llama7b_mha,
    "llama3_8b_gqa": llama3_8b_gqa,
    "longctx_fp8": longctx_fp8,
    "prefix_share": prefix_share,
}
