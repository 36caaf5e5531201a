"""The multi-process side of bench.py on the CPU: world size 2 over gloo
(127.0.0.1), exercising the same helpers the GPU run uses with NCCL --
process-group set-up from the torchrun environment, the barrier, the maximum
of the per-rank times and the whole-job (replicas) throughput -- plus the
reference arm, which only rank 0 runs."""
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, port, q):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2", MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    ws, r, local = bench.dist_setup()
    bench.barrier(ws)
    secs = bench.max_over_ranks(1.5 + r, ws)          # rank 1 is the slow one
    q.put((r, ws, local, dist.get_backend(), secs, bench.whole_job_gbs(ws, 3e9, secs)))
    bench.barrier(ws)
    dist.destroy_process_group()


def test_two_rank_gloo_helpers():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, (rank, ws, local, backend, secs, gbs) in enumerate(out):
        assert (rank, ws, local, backend) == (r, 2, r, "gloo")
        assert secs == 2.5                              # the max over ranks
        assert gbs == 2 * 3e9 / 2.5 / 1e9               # both replicas' bytes in the slowest time


def test_reference_arm_only_rank0_prints():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_clock_samples_inside_the_load_window():
    """The clock summary keeps the nvidia-smi samples taken while the measured
    work ran (and all samples when none fell inside), with the throttle
    reasons seen there."""
    import datetime
    import time
    sys.path.insert(0, ROOT)
    import bench
    now = time.time()

    def fmt(t):
        return datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    c = bench.ClockSampler(0)
    idle = "Not Active, Not Active, Not Active, Not Active"
    capped = "Not Active, Not Active, Not Active, Active"
    c.lines = [f"{fmt(now - 1)}, 0, 2070, 2070, 300.0, 0x0, {idle}",
               f"{fmt(now + 0.1)}, 0, 1650, 2070, 1390.0, 0x4, {capped}",
               f"{fmt(now + 0.2)}, 0, 1700, 2070, 1385.0, 0x4, {capped}",
               f"{fmt(now + 2)}, 0, 2070, 2070, 300.0, 0x0, {idle}"]
    c.load(now, now + 1)
    s = c.summary()
    assert (s["sm_mhz"], s["samples_under_load"], s["reasons"]) == (1675.0, 2, ["sw_power_cap"])
    c.window = None
    s = c.summary()
    assert (s["samples"], s["samples_under_load"]) == (4, 0)
