"""bench.py's command line on the CPU: the reference arm (the oracle timed on
the host cores) prints one JSON line with the keys the bench contract asks
for; under torchrun only rank 0 prints; too few warm-up steps are refused."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BENCH = os.path.join(ROOT, "bench.py")


def _run(args, timeout=300):
    env = dict(os.environ)
    env.pop("RANK", None)
    env.pop("WORLD_SIZE", None)
    return subprocess.run([sys.executable] + args, cwd=ROOT, capture_output=True, text=True,
                          timeout=timeout, env=env)


def _json_lines(out):
    return [json.loads(line) for line in out.splitlines() if line.startswith("{")]


def test_reference_arm_prints_one_contract_line():
    r = _run([BENCH, "--impl", "reference", "--config", "p5_example", "--steps", "2",
              "--warmup", "3"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    d = lines[0]
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["value"] > 0 and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["n_gpus"] == 1 and d["steps"] == 2 and d["warmup"] == 3
    assert d["config"]["workload"] == "p5_example"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


@pytest.mark.parametrize("extra,rows", [(["--query-tokens", "2"], 6), (["--group", "3"], 3)])
def test_reference_arm_takes_the_workload_options(extra, rows):
    r = _run([BENCH, "--impl", "reference", "--config", "p5_example", "--steps", "2",
              "--warmup", "3"] + extra)
    assert r.returncode == 0, r.stderr[-2000:]
    (d,) = _json_lines(r.stdout)
    assert d["config"]["query_rows_per_step"] == rows
    if "--group" in extra:
        assert d["config"]["H"] == 3 * d["config"]["Hkv"]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_reference_arm_under_two_ranks_prints_once():
    r = _run(["-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
              "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), BENCH,
              "--impl", "reference", "--gpus", "2", "--config", "p5_example", "--steps", "2",
              "--warmup", "3"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1 and lines[0]["n_gpus"] == 2


def test_fewer_than_three_warmup_steps_are_refused():
    r = _run([BENCH, "--impl", "reference", "--config", "p5_example", "--steps", "2",
              "--warmup", "2"])
    assert r.returncode != 0
    assert _json_lines(r.stdout) == []


@pytest.mark.gpu
@pytest.mark.parametrize("extra", [[], ["--query-tokens", "2"], ["--graph"], ["--fused-append"]])
def test_bench_line_on_the_gpu(extra):
    """The GPU arm on a small workload: one JSON line with the contract's keys,
    the roofline against the measured peak, an end-to-end figure with its
    byte counts, the clocks, the launch count and the parity sample."""
    r = _run([BENCH, "--config", "qwen2_b8_g7_d64", "--steps", "20", "--warmup", "3",
              "--cpu-baseline-s", "0.5"] + extra, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    (d,) = _json_lines(r.stdout)
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "cpu_baseline", "e2e", "clocks", "gpu_launches"):
        assert key in d, key
    assert d["value"] > 0 and d["n_gpus"] == 1 and d["steps"] == 20 and d["warmup"] == 3
    rf = d["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["peak"] > 0
    assert rf["frac"] == pytest.approx(rf["achieved"] / rf["peak"], abs=1e-4)  # rounded to 4 places
    # the timed steps do the work: no faster than the device's memory allows
    assert d["value"] < 1.5 * rf["peak"] and rf["frac"] < 1.5
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    # the synchronous host-buffer step costs more than the device step; the
    # pipelined one adds its staging kernel to every step (with --fused-append
    # the timed step also writes the new rows, which the host-buffer step
    # does not, so there the two are not comparable)
    if "--fused-append" not in extra:
        assert e["sync_value"] < d["value"] and e["value"] <= 1.05 * d["value"]
    assert d["gpu_launches"] >= d["steps"]  # one cluster kernel, or split + merge, per step
    assert d["clocks"]["sm_max_mhz"] > 0
    assert d["parity_vs_oracle"]["max_abs_err"] <= 2e-3
    assert d["cpu_baseline"]["kind"] == "oracle"


def test_per_config_selection():
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import bench

    every = [e[0] for e in bench.PER_CONFIG]
    assert bench.per_config_entries("none", True) == []
    assert bench.per_config_entries("auto", False) == []
    assert [e[0] for e in bench.per_config_entries("auto", True)] == every
    assert [e[0] for e in bench.per_config_entries("all", False)] == every
    picked = bench.per_config_entries("qwen2_b8_g7_d64,p5_example", False)
    assert [e[0] for e in picked] == ["qwen2_b8_g7_d64", "p5_example"]
    with pytest.raises(SystemExit):
        bench.per_config_entries("no_such_entry", True)
