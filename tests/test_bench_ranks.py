"""Host logic of bench.py's multi-process path, on CPU: two gloo ranks time
rank 0's number of steps, a job's time is its slowest rank's, the whole-job
rate counts every rank's units; under torchrun the reference arm prints one
line from rank 0 and every rank exits 0."""

import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        steps = bench.rank0_value(100 + 7 * rank, "cpu")
        times = bench.max_over_ranks([1.0 + rank, 5.0 - rank, 3.0], "cpu")
        q.put((rank, steps, times))
    finally:
        dist.destroy_process_group()


def test_rank_reductions_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, steps, times in got:
        assert steps == 100, (rank, steps)            # rank 0's step count everywhere
        assert times == [2.0, 5.0, 3.0], (rank, times)  # each time's maximum over the ranks


def test_whole_job_rate_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench
    # 64 rows x 10 steps on each of 2 ranks in 1000 ms
    assert bench.whole_job_rate(64 * 10, 2, 1000.0) == pytest.approx(1280.0)
    assert bench.whole_job_rate(64 * 10, 1, 500.0) == pytest.approx(1280.0)
    # no process group: the values come back unchanged
    assert bench.max_over_ranks([1.5, 2.5], "cpu") == [1.5, 2.5]
    assert bench.rank0_value(17, "cpu") == 17


def test_reference_arm_under_torchrun_two_ranks():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3", "--reference-seconds", "2"]
    res = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, res.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"], "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_algorithmic_bytes_of_quantized_base():
    """The GEMM's algorithmic bytes count 1 byte (int8) or half a byte (int4)
    per base weight plus one fp32 scale per row; the rest is unchanged."""
    sys.path.insert(0, ROOT)
    import bench
    from workloads import make_config
    wl = make_config("decode_bgmv")
    N, K = wl.projections[0].N, wl.K
    bf16 = bench.algorithmic(wl)
    i8 = bench.algorithmic(wl, 8)
    i4 = bench.algorithmic(wl, 4)
    assert bf16["gemm_bytes"] - i8["gemm_bytes"] == N * K - N * 4
    assert bf16["gemm_bytes"] - i4["gemm_bytes"] == N * K * 3 // 2 - N * 4
    assert bf16["gemm_flops"] == i8["gemm_flops"] == i4["gemm_flops"] == 2 * wl.M * N * K
    assert bf16["lora_bytes"] == i8["lora_bytes"] == i4["lora_bytes"]


def test_algorithmic_bytes_follow_the_method():
    """The base GEMM's bytes are (NK + MK + MN) * 2 with no implementation
    intermediate (34,603,008 for 64 x 4096 -> 4096, as worked out by hand);
    the standalone LoRA bytes count each distinct adapter once, the adapted
    rows of x and of y (read and written) and V written and read; the fp32
    correction array is reported apart as an intermediate."""
    import numpy as np
    sys.path.insert(0, ROOT)
    import bench
    from workloads import make_config
    wl = make_config("decode_bgmv")
    a = bench.algorithmic(wl)
    M, K, N = 64, 4096, 4096
    assert a["gemm_bytes"] == (N * K + M * K + M * N) * 2 == 34_603_008
    assert a["gemm_flops"] == 2 * M * N * K
    distinct = np.unique(wl.row_adapter[wl.row_adapter >= 0]).size
    Ma = int((wl.row_adapter >= 0).sum())
    assert (distinct, Ma) == (a["distinct"], a["adapted_rows"])
    assert a["lora_bytes"] == distinct * 16 * (K + N) * 2 + Ma * (K + 2 * N) * 2 + 2 * Ma * 16 * 4
    assert a["lora_bytes_fused"] == distinct * 16 * (K + N) * 2 + 2 * Ma * 16 * 4
    assert a["intermediate_bytes"] == 2 * M * N * 4
    assert a["lora_flops"] == 2 * Ma * 16 * (K + N)
    # large M with the two-SM GEMM (N >= 256): the whole LoRA term is inside
    # the GEMM, whose bytes are the base bytes plus the distinct adapters'
    # A and B and V written and read (x and y shared with the base), and
    # whose flops add 2 r (K + N) per adapted row; before it only the tile
    # plans are made (the row ids read, 48 ints per 256-token tile written)
    wl = make_config("prefill_sgmv")
    a = bench.algorithmic(wl)
    M = 8192
    rd = int(sum(int(wl.ranks[s]) for s in np.unique(wl.row_adapter)))
    rr = int(wl.ranks[wl.row_adapter].sum())
    assert a["orientation"] == "pair"
    assert a["gemm_bytes"] == (N * K + M * K + M * N) * 2 + rd * (K + N) * 2 + 2 * rr * 4
    assert a["gemm_flops"] == 2 * M * N * K + 2 * rr * (K + N)
    assert a["lora_bytes"] == 4 * M + 48 * 4 * (M // 256) and a["lora_flops"] == 0
    # large M with fewer than 256 output columns: the shrink reads the
    # distinct A's and the adapted rows of x and writes V; the GEMM's share
    # adds the distinct B's and reads V
    import copy
    wl2 = copy.deepcopy(wl)
    wl2.projections[0].N = 136
    a = bench.algorithmic(wl2)
    assert a["orientation"] == "rows"
    assert a["lora_bytes"] == rd * K * 2 + M * K * 2 + rr * 4
    assert a["gemm_bytes"] == (136 * K + M * K + M * 136) * 2 + rd * 136 * 2 + rr * 4
    assert a["gemm_flops"] == 2 * M * 136 * K


def test_percentiles():
    sys.path.insert(0, ROOT)
    import bench
    p = bench.percentiles(list(range(1, 101)))
    assert p["p50"] == 50.5 and abs(p["p10"] - 10.9) < 1e-9 and abs(p["p90"] - 90.1) < 1e-9
