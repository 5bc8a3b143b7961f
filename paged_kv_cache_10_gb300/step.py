"""One decode step of the paged KV cache through the C ABI.

Host side (C++ allocator): ``append_batch`` reserves one slot per sequence
(copy-on-write pairs where a sequence writes into a shared partial block),
``export`` writes the padded block tables and lengths.  Device side, in
stream order: ``copy_blocks`` (only when there are pairs) ->
``paged_attention_decode_append`` (the decode kernel makes the copy-on-write
copies and writes the new tokens' K/V itself; + its merge kernel when a
sequence spans several partitions).
With ``fused=False`` (or for cascade decode) the append is its own kernel,
``paged_kv_append``, before the decode.

Re-running the device part is idempotent (the same slots get the same
values, the same copies are made), which is what timing loops rely on.
"""
from __future__ import annotations

import numpy as np
import torch

from . import pagedkv as pk

_STORE = {"f16": torch.uint16, "bf16": torch.uint16, "e4m3": torch.uint8}


def _to_dev(a: np.ndarray, device) -> torch.Tensor:
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.uint16)
    return torch.from_numpy(a).to(device)


class DecodeStep:
    """Device state and launch sequence of one workload's decode step."""

    def __init__(self, wl, device="cuda", partition_tokens=None, alloc: pk.Allocator | None = None,
                 cascade: bool = False, cascade_min_blocks: int = 16, fused: bool = True, plan="auto"):
        self.wl = wl
        self.device = torch.device(device)
        self.desc = pk.CacheDesc(num_blocks=wl.NB, num_kv_heads=wl.Hkv, head_size=wl.D, kv_dtype=wl.kv_dtype,
                                 k_scale=wl.k_scale, v_scale=wl.v_scale, block_size=wl.b)
        self.partition_tokens = wl.partition_tokens if partition_tokens is None else partition_tokens
        # -- host allocator: prefill script, then this step's appends
        self.alloc = alloc or pk.Allocator(wl.NB, wl.b, wl.free_order)
        pk.apply_setup(self.alloc, wl.setup)
        rows = np.arange(wl.S, dtype=np.int64)
        appending = np.full(wl.S, -1, np.int64)
        appending[np.asarray(wl.step_seqs, dtype=np.int64)] = np.asarray(wl.step_seqs, dtype=np.int64)
        self.slots, self.pairs = self.alloc.append_batch(appending)
        self.max_blocks = wl.max_blocks
        self.tables, self.seq_lens = self.alloc.export(rows, self.max_blocks)
        self.max_seq_len = int(self.seq_lens.max()) if wl.S else 0
        # -- device buffers
        dev = self.device
        self.k_cache = _to_dev(wl.k_pool, dev)
        self.v_cache = _to_dev(wl.v_pool, dev)
        self.q = _to_dev(wl.q, dev)
        self.k_new = _to_dev(wl.k_new, dev)
        self.v_new = _to_dev(wl.v_new, dev)
        self.d_slots = torch.from_numpy(self.slots).to(dev)
        self.d_pairs = torch.from_numpy(np.ascontiguousarray(self.pairs)).to(dev)
        # per batch row: the copy-on-write source of its last block (the
        # pair whose destination is the block its new token goes to), or -1
        cow = np.full(wl.S, -1, np.int32)
        if len(self.pairs):
            dst_row = {int(self.slots[r]) // wl.b: r for r in range(wl.S) if self.slots[r] >= 0}
            for src, dst in np.asarray(self.pairs).reshape(-1, 2):
                cow[dst_row[int(dst)]] = src
        self.cow_src = cow
        self.d_cow_src = torch.from_numpy(cow).to(dev)
        self.d_tables = torch.from_numpy(self.tables).to(dev)
        self.d_lens = torch.from_numpy(self.seq_lens).to(dev)
        self.out = torch.empty((wl.S, wl.Hq, wl.D), dtype=torch.uint16, device=dev)
        self.cascade = cascade
        self.fused = fused and not cascade
        if cascade:
            # groups of rows sharing leading blocks (host), decoded with one
            # pass over each shared prefix
            self.groups = self.alloc.prefix_groups(rows, cascade_min_blocks)
            g = self.groups
            self.d_seq_group = torch.from_numpy(g.seq_group).to(dev)
            self.d_group_blocks = torch.from_numpy(g.group_blocks).to(dev)
            self.d_group_offsets = torch.from_numpy(g.group_offsets).to(dev)
            self.d_group_members = torch.from_numpy(g.group_members).to(dev)
            ws = pk.decode_cascade_total_workspace_bytes(wl.kv_dtype, wl.S, wl.Hq, wl.Hkv, wl.D, self.max_seq_len,
                                                         self.max_blocks, self.partition_tokens, g.num_groups,
                                                         g.max_blocks)
        else:
            ws = pk.decode_workspace_bytes(wl.S, wl.Hq, wl.D, self.max_seq_len, self.partition_tokens)
        self.workspace = torch.empty(max(ws, 16), dtype=torch.uint8, device=dev) if ws else None
        self.launches = 0
        # the fused decode's CTAs in the host plan's order (longest unit
        # first).  "auto": where that order can pay, i.e. there is more than
        # a wave of CTAs, the units' lengths differ (by a block or more) and
        # no two rows share a block (CTAs of rows sharing blocks are better
        # co-scheduled in grid order, for L2).
        self.work = None
        if plan == "auto":
            plan = self._plan_pays()
        if plan and self.fused and wl.S:
            self.work_host = pk.decode_plan(self.seq_lens, wl.Hkv, self.max_seq_len, self.partition_tokens)
            self.work = torch.from_numpy(self.work_host).to(dev)

    def _plan_pays(self) -> bool:
        if not self.fused or self.wl.S == 0:
            return False
        used = self.tables[self.tables >= 0]
        if len(self.pairs) or np.unique(used).size != used.size:
            return False  # blocks shared between rows
        P = self.effective_partition(planned=True)
        lens = self.seq_lens.astype(np.int64)
        full = lens // P  # full partitions, plus one partial of lens % P tokens
        units = np.concatenate([np.full(int(full.sum()), P), (lens % P)[lens % P > 0]])
        sms = torch.cuda.get_device_properties(self.device).multi_processor_count if self.device.type == "cuda" else 1
        if units.size * self.wl.Hkv <= 2 * sms:
            return False  # one wave: the order does not matter
        return int(units.max() - units.min()) >= self.wl.b

    def effective_partition(self, planned=None) -> int:
        """Tokens per split-K partition of this step's decode (a planned
        launch's automatic size has no cap)."""
        if self.partition_tokens:
            return self.partition_tokens
        if planned is None:
            planned = getattr(self, "work", None) is not None
        return pk.decode_auto_partition(self.wl.S, self.wl.Hq, self.wl.Hkv, self.wl.D, self.max_seq_len, planned)

    def kernel_launches(self) -> int:
        """Number of kernels one ``run`` enqueues."""
        n = 1 if self.fused else 2  # (append +) decode
        if len(self.pairs) and not self.fused:
            n += 1
        if self.cascade:
            # merge, prefix pass (and the 16-bit staging of an fp8 pool's prefixes)
            n += 1 + ((2 if self.wl.kv_dtype == "e4m3" else 1) if self.groups.num_groups else 0)
            return n
        P = self.effective_partition()
        if self.max_seq_len > P:
            n += 1  # merge
        return n

    # -- device work (stream order)
    def copy(self, stream=None):
        if len(self.pairs) and not self.fused:  # the fused decode copies itself
            pk.copy_blocks(self.k_cache, self.v_cache, self.desc, self.d_pairs, stream=stream)

    def append(self, stream=None, k=None, v=None, slots=None):
        if self.fused:
            return  # done by decode()
        pk.paged_kv_append(self.k_new if k is None else k, self.v_new if v is None else v,
                           self.d_slots if slots is None else slots, self.k_cache, self.v_cache, self.desc,
                           in_dtype=self.wl.in_dtype, stream=stream)

    def decode(self, stream=None, q=None, tables=None, lens=None, out=None, k=None, v=None, slots=None,
               cow_src=None, work=None):
        if self.fused:
            pk.paged_attention_decode_append(
                self.k_new if k is None else k, self.v_new if v is None else v, self.d_slots if slots is None else slots,
                self.q if q is None else q, self.k_cache, self.v_cache, self.desc,
                self.d_tables if tables is None else tables, self.d_lens if lens is None else lens, self.max_seq_len,
                self.wl.scale, self.out if out is None else out, workspace=self.workspace,
                partition_tokens=self.partition_tokens, q_dtype=self.wl.q_dtype, in_dtype=self.wl.in_dtype,
                cow_src=(self.d_cow_src if cow_src is None else cow_src) if len(self.pairs) else None, stream=stream,
                work_units=self.work if work is None else work)
            return
        if self.cascade:
            g = self.groups
            pk.paged_attention_decode_cascade(
                self.q if q is None else q, self.k_cache, self.v_cache, self.desc,
                self.d_tables if tables is None else tables, self.d_lens if lens is None else lens,
                self.max_seq_len, self.wl.scale, self.out if out is None else out, self.d_seq_group,
                self.d_group_blocks, self.d_group_offsets, self.d_group_members, g.max_members, g.max_blocks,
                self.workspace, partition_tokens=self.partition_tokens, q_dtype=self.wl.q_dtype, stream=stream)
            return
        pk.paged_attention_decode(self.q if q is None else q, self.k_cache, self.v_cache, self.desc,
                                  self.d_tables if tables is None else tables,
                                  self.d_lens if lens is None else lens, self.max_seq_len, self.wl.scale,
                                  self.out if out is None else out, workspace=self.workspace,
                                  partition_tokens=self.partition_tokens, q_dtype=self.wl.q_dtype, stream=stream)

    def run(self, stream=None):
        self.copy(stream)
        self.append(stream)
        self.decode(stream)

    def capture(self):
        """Records one step (copy, append, decode and its merge) into a CUDA
        graph and returns it; ``graph.replay()`` re-issues the same kernels
        with one launch.  Run the step eagerly once first, so every
        one-time set-up (kernel attributes, device addresses) is done."""
        self.run()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            self.run()
        torch.cuda.synchronize()
        return graph


class PrefillStep:
    """Device state and launch sequence of one paged (chunked) prefill step.

    Host: the allocator holds every sequence's earlier context, then reserves
    one slot per new token (``append_tokens``).  Device, in stream order: ``paged_kv_append`` of the new
    tokens' K/V -> ``paged_attention_prefill`` for their query rows, its CTAs
    in the order of the host plan (``prefill_plan``: longest causal key range
    first) unless ``plan`` is False.  Over an fp8 pool the attention call
    first copies the blocks it reaches into 16-bit blocks in ``workspace``."""

    def __init__(self, wl, device="cuda", alloc: pk.Allocator | None = None, plan: bool = True):
        self.wl = wl
        self.device = torch.device(device)
        self.desc = pk.CacheDesc(num_blocks=wl.NB, num_kv_heads=wl.Hkv, head_size=wl.D, kv_dtype=wl.kv_dtype,
                                 k_scale=wl.k_scale, v_scale=wl.v_scale, block_size=wl.b)
        self.alloc = alloc or pk.Allocator(wl.NB, wl.b, wl.free_order)
        for s, c in enumerate(wl.ctx):
            self.alloc.seq_new(s, int(c))
        self.slots, self.pairs = self.alloc.append_tokens(np.arange(wl.S), wl.qlens)
        assert len(self.pairs) == 0  # no block is shared
        self.tables, self.seq_lens = self.alloc.export(np.arange(wl.S, dtype=np.int64), wl.max_blocks)
        self.query_start = np.zeros(wl.S + 1, np.int32)
        self.query_start[1:] = np.cumsum(np.asarray(wl.qlens, dtype=np.int64))
        dev = self.device
        self.k_cache = _to_dev(wl.k_pool, dev)
        self.v_cache = _to_dev(wl.v_pool, dev)
        self.q = _to_dev(wl.q, dev)
        self.k_new = _to_dev(wl.k_new, dev)
        self.v_new = _to_dev(wl.v_new, dev)
        self.d_slots = torch.from_numpy(self.slots).to(dev)
        self.d_tables = torch.from_numpy(self.tables).to(dev)
        self.d_lens = torch.from_numpy(self.seq_lens).to(dev)
        self.d_query_start = torch.from_numpy(self.query_start).to(dev)
        self.out = torch.empty((wl.T, wl.Hq, wl.D), dtype=torch.uint16, device=dev)
        ws = pk.prefill_workspace_bytes(wl.kv_dtype, wl.S, wl.Hkv, wl.D, wl.max_blocks)
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=dev) if ws else None
        self.work = None
        if plan:
            self.work_host = pk.prefill_plan(self.query_start, self.seq_lens, wl.Hq, wl.Hkv, wl.max_query_len)
            self.work = torch.from_numpy(self.work_host).to(dev)

    def kernel_launches(self) -> int:
        # append + prefill attention (+ the 16-bit staging of an fp8 pool)
        return 3 if self.workspace is not None else 2

    def append(self, stream=None):
        pk.paged_kv_append(self.k_new, self.v_new, self.d_slots, self.k_cache, self.v_cache, self.desc,
                           in_dtype=self.wl.dtype, stream=stream)

    def attend(self, stream=None, q=None, out=None):
        pk.paged_attention_prefill(self.q if q is None else q, self.k_cache, self.v_cache, self.desc,
                                   self.d_query_start, self.wl.max_query_len, self.d_tables, self.d_lens,
                                   self.wl.scale, self.out if out is None else out, q_dtype=self.wl.dtype,
                                   stream=stream, work_units=self.work, workspace=self.workspace)

    def run(self, stream=None):
        self.append(stream)
        self.attend(stream)
