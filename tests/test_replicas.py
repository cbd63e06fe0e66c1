"""Host logic of the multi-GPU launch (one independent replica per GPU), run
as world-size-2 gloo ranks on the CPU: rendezvous from the launcher's
environment, the barrier, the slowest rank's time as every rank's time, the
whole-job rate, and the reference arm's rank-0-only behaviour."""
import json
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    r = bench.Replicas("gloo", torch.device("cpu"))
    r.barrier()
    slowest = r.max(10.0 + rank)  # the last rank is the slowest
    rate = r.total_rate(100.0, slowest)
    r.barrier()
    r.close()
    q.put((rank, r.world, r.rank, slowest, rate))


@pytest.mark.timeout(300)
def test_two_replicas_over_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=240) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[0] for g in got] == [0, 1]
    for rank, world, r_rank, slowest, rate in got:
        assert world == 2 and r_rank == rank
        assert slowest == 11.0  # every rank reports the slowest rank's time
        assert rate == pytest.approx(2 * 100.0 / 11.0)  # all ranks' work / that time


def test_single_process_needs_no_rendezvous(monkeypatch):
    for v in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(v, raising=False)
    import bench
    r = bench.Replicas("gloo", torch.device("cpu"))
    assert (r.world, r.rank, r.local) == (1, 0, 0)
    assert r.max(3.5) == 3.5 and r.total_rate(10.0, 2.0) == 5.0
    r.barrier()
    r.close()


class _Args:
    cpu_tokens, warmup, steps, gpus = 1, 0, 1, 2


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import bench
    from w8a8_int8_quantized_token_gb300 import synth
    cfg = synth.CONFIGS["tiny"]
    monkeypatch.setenv("RANK", "1")
    bench.run_reference(_Args(), cfg)
    assert capsys.readouterr().out == ""  # other ranks exit without work
    monkeypatch.setenv("RANK", "0")
    bench.run_reference(_Args(), cfg)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"], "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
