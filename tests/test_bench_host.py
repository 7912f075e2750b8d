"""Host-side logic of bench.py on the CPU: the replica launch path at world size 2 (gloo),
the max-over-ranks reduction, the FLOP bookkeeping and the JSON contract of the oracle arm."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank)
    bench.dist_barrier(w)
    m = bench.dist_max(float(rank + 1) * 1.5, w, torch.device("cpu"))
    out.put((rank, m))
    dist.destroy_process_group()


def test_max_over_ranks_with_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == {0: 3.0, 1: 3.0}


def test_reference_arm_under_torchrun_prints_one_line_from_rank0():
    port = free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.join(ROOT, "bench.py"), "--gpus", "2", "--impl", "reference",
           "--workload", "tiny_fwd_fp16", "--steps", "2", "--warmup", "1"]
    res = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    for key in ("metric", "value", "unit", "steps", "warmup", "ms_per_step", "higher_is_better",
                "cpu_baseline", "e2e", "config"):
        assert key in line
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    assert line["cpu_baseline"]["kind"] == "oracle"


def test_flop_convention():
    f = bench.flops(1, 32, 8192, 128, causal=True)
    fwd = 4 * 32 * 8192 ** 2 * 128 / 2
    assert f["fa_fwd_kernel"] == fwd
    assert f["fa_bwd_dkdv_kernel"] + f["fa_bwd_dq_kernel"] == 2.5 * fwd
    assert abs(fwd / 1e9 - 549.76) < 0.01  # the 8k causal forward is 549.8 GFLOP
    g = bench.flops(1, 8, 16384, 64, causal=False, density=0.25)
    assert g["fa_fwd_kernel"] == 4 * 8 * 16384 ** 2 * 64 * 0.25


def test_warmup_floor_is_enforced():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "1"])


def test_mufu_bound_counts_one_exponential_per_live_tile_element():
    # brute force over the tile grid: causal keeps j <= i, the block mask keeps M[i][j] != 0
    from exact_attention_staged_gb300.workloads import Workload
    T = 5
    mask = torch.tensor([[1, 0, 1, 1, 0], [0, 1, 0, 0, 1], [1, 1, 1, 0, 0], [0, 0, 1, 1, 1],
                         [1, 0, 0, 1, 1]], dtype=torch.uint8)
    for causal in (False, True):
        for m in (None, mask):
            w = Workload("t", 2, 3, T * 128 - 7, 64, "bf16", causal, 1)
            live = sum(1 for i in range(T) for j in range(T)
                       if (not causal or j <= i) and (m is None or m[i, j] != 0))
            r = bench.mufu_bound(w, m, 1.0, {"sm_mhz": 1000.0, "sm_max_mhz": 2070.0})
            assert r["exps_per_launch"] == live * 128 * 128 * 2 * 3
            assert r["peak"] == pytest.approx(32 * 152 * 1000e6 / 1e12)
            assert r["achieved"] == pytest.approx(r["exps_per_launch"] / 1e-3 / 1e12)


def test_cpu_model_is_named():
    assert isinstance(bench.cpu_model(), str) and bench.cpu_model()


def test_stored_traffic_is_used_only_while_the_kernel_sources_match(monkeypatch):
    # every stored record names a kernel bench.py knows and carries its sources' hash
    with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
        stored = json.load(f)
    for workload, kernels in stored.items():
        for kernel, rec in kernels.items():
            assert kernel in bench.KERNEL_SOURCES, kernel
            assert rec["dram_bytes_per_launch"] == rec["dram_read"] + rec["dram_write"]
            assert rec["command"].startswith("ncu ") and "--clock-control none" in rec["command"]
    # the decode step's figure is the decode kernel plus the merge, the merge only when split
    one = bench.ncu_traffic("fa_decode_kernel", "decode_gqa_d128_kv8k")
    merge = bench.ncu_traffic("fa_decode_combine_kernel", "decode_gqa_d128_kv8k")
    if one is not None and merge is not None:
        assert bench.decode_traffic("decode_gqa_d128_kv8k", 1) == one + merge
        assert bench.decode_traffic("decode_gqa_d128_kv8k", 0) == one
    # a changed source (here: the hash taken over another file) voids the stored figure
    monkeypatch.setitem(bench.KERNEL_SOURCES, "fa_decode_kernel", ("bench.py",))
    assert bench.ncu_traffic("fa_decode_kernel", "decode_gqa_d128_kv8k") is None
    assert bench.decode_traffic("decode_gqa_d128_kv8k", 1) is None


def test_call_traffic_is_the_sum_of_its_kernels_records(monkeypatch):
    # a backward call (the dominant unit of the grouped-query and dropout lines) counts every
    # recorded kernel of its workload but the forward; any kernel without a valid record voids it
    with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
        stored = json.load(f)
    for workload in ("dropout_causal_d128_n8k", "gqa_causal_d128_n8k"):
        kernels = [k for k in stored.get(workload, {}) if k != "fa_fwd_kernel"]
        parts = [bench.ncu_traffic(k, workload) for k in kernels]
        if kernels and all(x is not None for x in parts):
            assert bench.backward_call_traffic(workload) == sum(parts)
    assert bench.calls_traffic("no_such_workload", ["fa_fwd_kernel"]) is None
    assert bench.calls_traffic("gpt_causal_d128_n8k", []) is None
    monkeypatch.setitem(bench.KERNEL_SOURCES, "fa_bwd_dq_kernel", ("bench.py",))
    assert bench.backward_call_traffic("dropout_causal_d128_n8k") is None


def test_source_hash_ignores_comments_but_not_code(tmp_path, monkeypatch):
    src = 'int f(int x) {  // doubles\n  /* "quoted" */ return 2 * x; }\nconst char *s = "a // b";\n'
    (tmp_path / "a.cu").write_text(src)
    (tmp_path / "b.cu").write_text("// header comment\n\n" + src.replace("// doubles", "// twice"))
    (tmp_path / "c.cu").write_text(src.replace("2 * x", "3 * x"))
    (tmp_path / "d.cu").write_text(src.replace('"a // b"', '"a // c"'))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = {n: bench.source_hash((n,)) for n in ("a.cu", "b.cu", "c.cu", "d.cu")}
    assert h["a.cu"] == h["b.cu"]        # comments and blank lines only
    assert h["a.cu"] != h["c.cu"]        # code
    assert h["a.cu"] != h["d.cu"]        # a string literal that holds comment markers


def test_clock_summary_keeps_only_samples_inside_the_timed_regions():
    clk = bench.ClockSampler(0)
    line = "{},2070,Not Active,Not Active,Not Active,{}"
    clk.samples = [(0.5, line.format(1500, "Not Active")),   # before the first region
                   (1.2, line.format(2070, "Not Active")),
                   (1.8, line.format(2000, "Active")),
                   (2.5, line.format(900, "Active")),        # between regions
                   (3.1, line.format(1980, "Not Active"))]
    clk.windows = [(1.0, 2.0), (3.0, 3.5)]
    s = clk.summary()
    assert s["samples"] == 3
    assert s["sm_mhz"] == 2000 and s["sm_mhz_min"] == 1980 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"]
