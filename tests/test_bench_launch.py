"""How `bench.py` is launched (no GPU): our arm refuses a multi-GPU launch
before it loads the library (its pair GEMM engines use TMA multicast within
a cluster, kept to one-GPU runs), the binding refuses to load the library
in a rank of a multi-process launch, and the reference arm (the CPU oracle)
runs on rank 0 only."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _bench(env_extra, *argv):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *argv], env=env,
                          capture_output=True, text=True, timeout=240)


@pytest.mark.parametrize("env,argv", [({"WORLD_SIZE": "2", "RANK": "0", "LOCAL_RANK": "0"}, ()),
                                      ({"WORLD_SIZE": "2", "RANK": "1", "LOCAL_RANK": "1"}, ()),
                                      ({}, ("--gpus", "4"))])
def test_multi_gpu_launch_is_refused(env, argv):
    r = _bench(env, "--steps", "1", "--warmup", "0", *argv)
    assert r.returncode == 2, r.stderr
    assert r.stdout == ""
    assert "refused" in r.stderr and "one GPU only" in r.stderr


def test_binding_refuses_multi_process_rank(monkeypatch):
    from w8a8_int8_quantized_token_gb300 import binding
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setattr(binding, "_lib", None)
    with pytest.raises(binding.WQError, match="one-GPU runs only"):
        binding.lib()


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


def test_reference_arm_under_two_ranks_prints_once():
    env = {"WORLD_SIZE": "2", "RANK": "1", "LOCAL_RANK": "1"}
    r = _bench(env, "--impl", "reference", "--config", "tiny", "--steps", "1", "--warmup", "0",
               "--cpu-tokens", "1")
    assert r.returncode == 0 and r.stdout == ""
    env["RANK"] = env["LOCAL_RANK"] = "0"
    r = _bench(env, "--impl", "reference", "--config", "tiny", "--steps", "1", "--warmup", "0",
               "--cpu-tokens", "1")
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
