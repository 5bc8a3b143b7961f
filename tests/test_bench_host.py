"""Host-side logic of bench.py without a GPU: the multi-rank aggregation
(whole-job bytes summed over ranks, time = slowest rank) over a gloo process
group of two CPU ranks, the algorithmic byte count of a step, the
recorded traffic rows, and the reference arm (the oracle) run on the CPU."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    b, s = bench.aggregate(1000.0 * (rank + 1), 0.5 + rank)
    q.put((rank, b, s))
    dist.destroy_process_group()


def test_aggregate_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for _, b, s in res:
        assert b == 3000.0 and s == 1.5


def test_single_process_aggregate_is_identity():
    import bench
    assert bench.aggregate(12.0, 3.0) == (12.0, 3.0)


def test_step_bytes_counts_the_gathered_kv():
    import bench

    class WL:
        S, Hq, Hkv, D, b = 2, 8, 2, 128, 16
        def kv_elem_bytes(self):
            return 2

    class Step:
        wl = WL()
        seq_lens = np.array([17, 40], np.int32)
        slots = np.array([5, -1], np.int64)
        pairs = np.zeros((1, 2), np.int32)
        # row 1 shares its first block (full in both) with row 0
        tables = np.array([[7, 3, -1], [7, 9, 4]], np.int32)

    nb = bench.step_bytes(Step())
    assert nb["kv"] == (17 + 40) * 2 * 2 * 128 * 2
    assert nb["decode"] == nb["kv"] + 2 * 2 * 8 * 128 * 2 + (2 + 3) * 4 + 2 * 4
    assert nb["append"] == 1 * 2 * 2 * 128 * (2 + 2) + 2 * 8
    assert nb["copy"] == 1 * (2 * 2 * (2 * 16 * 128 * 2) + 8)
    assert nb["total"] == nb["decode"] + nb["append"] + nb["copy"]
    # distinct tokens: block 7 (16), block 3 (1), block 9 (16), block 4 (8)
    assert nb["unique_kv"] == (16 + 1 + 16 + 8) * 2 * 2 * 128 * 2
    assert nb["decode_unique"] == nb["decode"] - nb["kv"] + nb["unique_kv"]


def test_prefill_flops_count_every_causal_pair():
    import bench

    class WL:
        D, Hq = 128, 8
        ctx = [0, 5, 33]
        qlens = [3, 4, 1]

    # brute force: each new row at position p sees keys 0..p; 4 * D flops per key and head
    pairs = sum(c + j + 1 for c, n in zip(WL.ctx, WL.qlens) for j in range(n))
    assert bench.prefill_flops(WL()) == 4.0 * 128 * 8 * pairs


def test_kernel_hash_ignores_comments_but_not_code():
    """Recorded DRAM traffic is keyed by a hash of the kernel sources; an edit
    to // comments or blank lines must keep the key, any code edit must not."""
    import bench
    src = "int a = 1;  // one\n\n// a comment line\nint b = 2;\n"
    assert bench.code_only(src) == bench.code_only("int a = 1;\nint b = 2;  // two, reworded\n")
    assert bench.code_only(src) != bench.code_only("int a = 1;\nint b = 3;\n")
    for kind in bench.KERNEL_SOURCES:
        assert len(bench.kernel_hash(kind)) == 12


def test_kv_utilisation_counts_distinct_blocks_and_the_last_block_waste():
    """The b - 1 waste bound of the paged pool ("vLLM 高性能大语言模型推理引擎深度技术评估与分布式架构展望",
    physical blocks and the paging analogy): every sequence wastes at most the
    slots of its last block, and a block several sequences share counts once."""
    from types import SimpleNamespace
    import bench
    wl = SimpleNamespace(b=16, S=4)
    lens = np.array([1, 16, 33, 20], np.int32)
    tables = np.array([[3, -1, -1], [7, -1, -1], [4, 5, 6], [7, 9, -1]], np.int32)  # rows 1 and 3 share block 7
    got = bench.kv_utilisation(SimpleNamespace(wl=wl, seq_lens=lens, tables=tables))
    # distinct blocks 3, 7, 4, 5, 6, 9 hold 1, 16, 16, 16, 1, 4 tokens
    assert got["distinct_blocks"] == 6
    assert got["utilisation"] == round(54 / (6 * 16), 5)
    assert got["max_waste_tokens_per_seq"] == 15  # the 1-token row and the 33-token row
    assert 0 <= got["max_waste_tokens_per_seq"] <= wl.b - 1


def test_bench_parity_bound_is_the_tests_bound():
    """bench.py reports each config's error against the same per-element
    bound the parity tests assert (its own copy, since bench.py imports
    nothing from tests/)."""
    import bench
    from parity_util import relaxed_bound
    rng = np.random.default_rng(5)
    ref = np.concatenate([rng.normal(0, 3, 4000), rng.uniform(-20, 20, 4000), [0.0, 1e-30, 3.99, 4.0, 8.0]])
    for dt, tol in (("bf16", 1e-2), ("f16", 2e-3)):
        np.testing.assert_array_equal(bench.error_bound(ref, dt, tol, 7.5), relaxed_bound(ref, dt, tol, 7.5))


def test_recorded_traffic_covers_every_reported_kernel():
    """profiles/ncu_traffic.txt holds a row, for the current kernel sources,
    for every workload whose line carries roofline.traffic: each decode
    config (the cascade by its own source hash) and each prefill row."""
    import types
    import bench
    heads = {"tiny_fp16": (4, 4, 64), "llama7b_mha": (32, 32, 128), "llama3_8b_gqa": (32, 8, 128),
             "longctx_fp8": (64, 8, 128), "prefix_share": (32, 8, 128)}  # (query heads, KV heads, head size)
    for name, cascade, _ in bench.DECODE_CONFIGS:
        Hq, Hkv, D = heads[name]
        kind = "cascade" if cascade else bench.decode_kernel_kind(types.SimpleNamespace(Hq=Hq, Hkv=Hkv, D=D))
        t = bench.recorded_traffic(name, kind)
        assert t is not None and t > 0, (name, kind)
    from paged_kv_cache_10_gb300 import workloads
    for name in bench.NEXT_PREFILL + ("prefill_prompt_gqa", "prefill_prompt_mha"):
        assert name in workloads.PREFILL, name
        assert bench.recorded_traffic(name, "prefill"), name
    # the plain and the cascade rows of prefix_share are told apart by their hash
    assert bench.recorded_traffic("prefix_share", "cascade") != bench.recorded_traffic("prefix_share", "tensor_core")


@pytest.mark.parametrize("workload", ["tiny_fp16", "prefill_chunked_gqa"])
def test_reference_arm_line_and_no_product_code(workload):
    """bench.py --impl reference (the oracle as the reference arm) prints one
    JSON line with the arm's contract fields, on the CPU, and its process
    never loads the product library."""
    import json
    import subprocess
    import sys
    code = ("import json, sys, bench; bench.main(['--impl', 'reference', '--steps', '1', '--warmup', '1', "
            f"'--workload', '{workload}']); "
            "maps = open('/proc/self/maps').read(); "
            "print('PRODUCT_LOADED' if 'libpagedkv' in maps else 'PRODUCT_NOT_LOADED')")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert lines[-1] == "PRODUCT_NOT_LOADED"
    line = json.loads(lines[-2])
    assert line["impl"] == "reference" and line["value"] > 0 and line["higher_is_better"] is True
    assert line["unit"] == line["e2e"]["unit"] and line["e2e"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["config"]["workload"] == workload
