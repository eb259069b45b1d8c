"""Host-side logic of bench.py (CPU only): FLOP convention, clock parsing, the
reference arm's rank handling, and the cross-rank reductions under gloo (world size 2)."""

import json
import os
import subprocess
import sys

import pytest
import torch

import bench

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_flop_convention_matches_the_pages_figure():
    # hada.io FA3 summary, "Überlappung von GEMM und Softmax": at head dimension 128 there are
    # 512 times more matmul FLOPs than exponentials (one exponential per score element).
    with open(os.path.join(HERE, "golden", "pages_figures.json")) as f:
        g = json.load(f)
    B, H, S, D = 3, 5, 64, 128
    exps = B * H * S * S
    assert bench.attention_flops(B, H, S, D) / exps == g["matmul_flops_per_exp_at_head_dim_128"]["value"]
    assert bench.attention_flops(B, H, S, D, causal=True) * 2 == bench.attention_flops(B, H, S, D)


def test_quant_bytes():
    assert bench.quant_bytes(1, 128, 1, 128) == 128 * 128 * 3 + 4
    assert bench.quant_bytes(2, 300, 3, 64) == 2 * 300 * 3 * 64 * 3 + 4 * 2 * 3 * 3


def test_clock_sampler_parsing():
    cs = bench.ClockSampler.__new__(bench.ClockSampler)
    cs.proc = None
    assert cs.stop()["sm_mhz"] is None
    cs.lines = ["0, 2000, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Not Active",
                "0, 1980, 2070, 1300.0, 0x4, Not Active, Not Active, Not Active, Active",
                "0, 2010, 2070, 1100.0, 0x0, Not Active, Not Active, Not Active, Not Active"]

    class _P:
        def terminate(self): pass
        def wait(self, timeout=None): pass

    class _T:
        def join(self, timeout=None): pass

    cs.proc, cs.thread = _P(), _T()
    r = cs.stop()
    assert r["sm_mhz"] == 2000 and r["sm_max_mhz"] == 2070 and r["reasons"] == ["sw_power_cap"]


def test_reference_arm_non_zero_rank_does_no_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "2", "--warmup", "3"], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOPS" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    dev = torch.device("cpu")
    mx = bench.max_over_ranks(1.0 + rank, True, dev)
    sm = bench.sum_over_ranks(10.0 * (rank + 1), True, dev)
    torch.distributed.barrier()
    out.put((rank, mx, sm))
    torch.distributed.destroy_process_group()


def test_cross_rank_max_and_sum_under_gloo():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == [(0, 2.0, 30.0), (1, 2.0, 30.0)]
