"""The multi-GPU path is replicas only (independent layers per rank, no exchange step):
bench.py's ranks meet at barriers and the job's time is the slowest rank's.  Checked here
with two gloo ranks on the CPU."""
import os
import socket


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 10.0 + 5.0 * rank                      # rank 1 is the slow replica
        dist.barrier()
        got = bench.slowest_rank_ms(ms, dist, device="cpu")
        out[rank] = got
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_replicas_report_the_slowest_rank():
    import torch.multiprocessing as mp
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    assert dict(out) == {0: 15.0, 1: 15.0}


def test_single_rank_time_is_its_own():
    import bench
    assert bench.slowest_rank_ms(12.5, None, device="cpu") == 12.5


def test_reference_arm_runs_on_rank_zero_only(capsys):
    import bench
    bench.run_reference(bench.parse(["--impl", "reference"]), rank=1, world=2)     # a non-zero rank returns without work
    assert capsys.readouterr().out == ""


def test_reference_arm_json_line():
    """bench.py --impl reference (the float64 oracle on the host cores) prints one JSON
    line with the keys the contract fixes."""
    import json
    import subprocess
    import sys
    here = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, os.path.join(here, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "1", "--cpu-seconds", "0.5"], capture_output=True, text=True, timeout=600,
                         cwd=here, check=True).stdout.strip().splitlines()
    line = json.loads(out[-1])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in line, k
    assert line["impl"] == "reference" and line["value"] > 0 and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
