"""Host-side logic of bench.py without a GPU: the multi-rank reductions with
the gloo backend (two processes), the clock-record parsing, and that the
reference arm's non-zero ranks exit without output."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_WORKER = r"""
import os, sys, json
sys.path.insert(0, {root!r})
import torch.distributed as dist
import bench
dist.init_process_group("gloo", rank=int(os.environ["RANK"]), world_size=2)
rank = dist.get_rank()
ms = bench.max_over_ranks(10.0 + rank, 2, device="cpu")
tot = bench.sum_over_ranks(1000.0 * (rank + 1), 2, device="cpu")
bench.barrier(2)
print(json.dumps({{"rank": rank, "ms": ms, "tot": tot}}), flush=True)
dist.destroy_process_group()
"""


def test_two_rank_reductions_gloo(tmp_path):
    pytest.importorskip("torch")
    script = tmp_path / "w.py"
    script.write_text(_WORKER.format(root=ROOT))
    procs = []
    for r in range(2):
        env = dict(os.environ, RANK=str(r), WORLD_SIZE="2", MASTER_ADDR="127.0.0.1", MASTER_PORT="29533")
        procs.append(subprocess.Popen([sys.executable, str(script)], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = [p.communicate(timeout=120) for p in procs]
    for p, (o, e) in zip(procs, outs):
        assert p.returncode == 0, e
    res = [json.loads(o.strip().splitlines()[-1]) for o, _ in outs]
    for r in res:
        assert r["ms"] == 11.0          # max over ranks: the slowest rank's time
        assert r["tot"] == 3000.0       # whole-job total


def test_clock_summary_keeps_samples_inside_the_timed_region():
    import datetime

    import bench
    c = bench.ClockSampler(0)
    c.out = ("2026/12/02 10:00:00.100, 1500, 2070, 1200.0, Not Active, Not Active, Not Active, Not Active\n"
             "2026/12/02 10:00:00.300, 1800, 2070, 1350.5, Not Active, Not Active, Not Active, Active\n"
             "2026/12/02 10:00:00.350, 1900, 2070, 1390.1, Not Active, Not Active, Not Active, Not Active\n"
             "garbage line\n"
             "2026/12/02 10:00:00.900, 1200, 2070, 900.0, Active, Not Active, Not Active, Not Active\n")
    t = lambda ms: datetime.datetime(2026, 12, 2, 10, 0, 0, ms * 1000).timestamp()  # noqa: E731
    c.mark(t(200), t(500))
    s = c.summary()
    assert s["sm_mhz"] == 1850.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"] and s["samples"] == 2
    c.mark(t(600), t(700))
    assert c.summary()["samples"] == 0


def test_reference_arm_other_ranks_exit_silently():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_arm_prints_one_contract_line():
    """The reference arm (the C++ oracle on the host cores) prints one JSON
    line with the contract's keys: metric, value, unit, the timed step,
    cpu_baseline with the thread count, and an e2e object with no copies."""
    env = dict(os.environ, LCE_REF_STEP_S="0.2")
    env.pop("RANK", None)
    env.pop("WORLD_SIZE", None)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                        "--steps", "2", "--warmup", "1"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench_metric() and d["unit"] == "valid tokens/s"
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["steps"] == 2 and d["warmup"] == 1
    assert d["higher_is_better"] is True and d["dtype"] == "f64"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def bench_metric():
    import bench
    return bench.METRIC


def test_kernel_hash_ignores_comments_only():
    import bench
    base = bench.kernel_src_sha256(["int a = 1;\nint b = a; // trailing\n", "asm(\"mov\");\n"])
    assert base == bench.kernel_src_sha256(["// header\nint a = 1;\n\nint b = a;\n", "asm(\"mov\"); // note\n"])
    assert base != bench.kernel_src_sha256(["int a = 2;\nint b = a;\n", "asm(\"mov\");\n"])
    assert len(bench.kernel_src_sha256()) == 16


def test_host_tensors_follow_the_workload_dtype():
    import torch

    import bench
    from synth_inputs import bf16_bits_to_f32, make_inputs
    x = make_inputs("tiny", N=8, d=16, V=20)
    H, W = bench.host_tensors(x)
    assert H.dtype == torch.float32 and H.shape == (8, 16) and torch.equal(H, torch.from_numpy(x.H))
    y = make_inputs("gpt1b", N=8, d=16, V=20, seqs=1)
    H, W = bench.host_tensors(y)
    assert H.dtype == torch.bfloat16 and W.shape == (20, 16)
    assert torch.equal(H.float(), torch.from_numpy(bf16_bits_to_f32(y.H)))
