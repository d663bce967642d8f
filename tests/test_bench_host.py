"""Host-side logic of bench.py: the max-over-ranks timing and the whole-job
throughput under two gloo ranks on CPU, the reference arm's rank handling,
and the clock-sample parsing. No GPU."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local = 1.0 + rank * 2.5                     # rank 1 is the slow one
        slowest = bench.reduce_max(local)
        bench.barrier()
        q.put((rank, slowest, bench.aggregate_throughput(32, world, slowest)))
    finally:
        dist.destroy_process_group()


def test_reduce_max_and_throughput_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [3.5, 3.5]               # every rank sees the slowest time
    assert res[0][2] == pytest.approx(32 * 2 / 3.5)        # all ranks' units over the max time


def test_reduce_max_without_process_group_is_identity():
    assert bench.reduce_max(1.25) == 1.25
    assert bench.aggregate_throughput(10, 1, 0.5) == 20.0


def test_reference_arm_on_a_non_zero_rank_does_no_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True,
                         timeout=120)
    assert out.returncode == 0 and out.stdout.strip() == ""


def test_reference_arm_prints_one_line(monkeypatch, capsys):
    # a tiny stand-in workload keeps this fast; the line format is what is checked
    monkeypatch.setattr(bench, "oracle_sample_decode", lambda cfg, seed, nseq: (0.5, 4, 1))
    rc = bench.main(["--impl", "reference", "--steps", "2", "--warmup", "3"])
    line = json.loads(capsys.readouterr().out.strip())
    assert rc == 0 and line["impl"] == "reference" and line["unit"] == "tok/s"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 4
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["higher_is_better"] is True


def test_clock_sampler_parses_nvidia_smi_lines():
    c = bench.ClockSampler.__new__(bench.ClockSampler)
    c.samples, c.reasons, c.max_mhz, c.error, c.source = [], set(), None, None, "nvidia-smi"
    c._thread, c.nvml = None, None
    c._stop = __import__("threading").Event()

    class FakeProc:
        def terminate(self):
            pass

        def communicate(self, timeout=None):
            return ("1965, 2032, 0x0000000000000000\n"
                    "210, 2032, 0x0000000000000001\n"        # idle: dropped
                    "1800, 2032, 0x0000000000000004\n"
                    "garbage\n", "")
    c._proc = FakeProc()
    c.__exit__(None, None, None)
    s = c.summary()
    assert s["samples"] == 2 and s["sm_mhz"] == pytest.approx(1882.5) and s["sm_max_mhz"] == 2032
    assert s["reasons"] == ["sw_power_cap"]
