"""Host-side logic of bench.py: multi-rank plumbing (gloo, world size 2, CPU),
token sharding, workload parsing, byte counts, and the reference arm."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

import bench
from tp_reduce_residual_gb300 import inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    r, w = bench.dist_init("gloo")
    bench.barrier()
    m = bench.max_over_ranks(10.0 + r)          # each rank reports a different time
    span = bench.row_range(1023, w, r)
    q.put((r, w, m, span))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_time_and_split_rows():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [2, 2]
    assert [r[2] for r in res] == [11.0, 11.0]      # max over ranks on every rank
    assert res[0][3] == (0, 512) and res[1][3] == (512, 1023)


@pytest.mark.parametrize("T,world", [(1, 1), (7, 2), (4096, 8), (3, 8)])
def test_row_ranges_partition_the_batch(T, world):
    spans = [bench.row_range(T, world, r) for r in range(world)]
    assert spans[0][0] == 0 and spans[-1][1] == T
    for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
        assert a1 == b0 and a0 <= a1
    assert max(b - a for a, b in spans) - min(b - a for a, b in spans) <= 1


def test_workload_parsing_and_bytes():
    wl, T = bench.parse_workload("C4:1024")
    assert (wl.R, wl.H, wl.k, T) == (8, 8192, 10, 1024)
    # T*H*(2Rk + 2R + 6) + 8RkT + 8H bytes for R=8, H=8192, k=10, T=1024: 1.527 GB
    assert abs(bench.workload_bytes(wl, T) / 1e9 - 1.527) < 0.001
    wl2, T2 = bench.parse_workload("C2:4096")
    assert abs(bench.workload_bytes(wl2, T2) / 1e6 - 738.3) < 0.1
    assert bench.workload_bytes(wl, T, split=True) - bench.workload_bytes(wl, T) == 8 * T * wl.H


def test_reference_arm_runs_on_cpu_and_prints_one_line():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "C1:64", "--steps", "3", "--warmup", "1", "--ref-seconds", "2"],
                       capture_output=True, text=True, env=env, timeout=600, cwd=ROOT)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_measured_peak_is_read_or_falls_back():
    peak, kind = bench.measured_peak()
    assert peak > 1000 and kind in ("measured", "fallback")


def test_kernel_hash_ignores_comments_only():
    a = 'int f(int x) { return x + 1; }  // add one\n'
    b = '/* the successor */\nint f(int x)\n{\n    return x + 1;  // comment changed\n}\n'
    c = 'int f(int x) { return x + 2; }\n'
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)
    assert bench._code_only('const char *s = "a // b";') == 'const char *s = "a // b";'


def test_headline_rotates_input_sets_below_twice_l2():
    """The headline loop replays one input set only when a call's inputs are
    at least twice L2; a smaller workload rotates over enough sets to pass 8x
    L2 (at most 64), and the config says which."""
    l2 = 136 * 1024 * 1024
    wl, T = bench.parse_workload("C4:1024")
    B = bench.workload_bytes(wl, T)
    assert bench.headline_sets(B, l2) == 1
    assert bench.l2_label(B, l2).endswith("no flush") and "> L2" in bench.l2_label(B, l2)
    wl, T = bench.parse_workload("C2:256")
    B = bench.workload_bytes(wl, T)
    n = bench.headline_sets(B, l2)
    assert n > 1 and n * B >= 8 * l2 and (n - 1) * B < 8 * l2
    assert "rotate over" in bench.l2_label(B, l2) and "warm" not in bench.l2_label(B, l2)
    wl, T = bench.parse_workload("C4:1")
    B = bench.workload_bytes(wl, T)
    assert bench.headline_sets(B, l2) == 64
    assert "partly L2-warm" in bench.l2_label(B, l2)
