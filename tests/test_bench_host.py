"""Host-side logic of the benchmark: byte accounting, the multi-rank
aggregation (world size 2 over gloo, on CPU) and the reference arm."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_byte_accounting():
    # values + masks + x + y, and the dense counterpart
    assert bench.sparse_bytes(4096, 4096) == 4096 * 4096 * 9 // 8 + 2 * 4096 * 2
    assert bench.dense_bytes(4096, 4096) == 2 * 4096 * 4096 + 4 * 4096
    mats = bench.WORKLOADS["llama33_70b_layer"]
    sp = sum(bench.sparse_bytes(r, c) for _, r, c in mats)
    de = sum(bench.dense_bytes(r, c) for _, r, c in mats)
    assert abs(sp / 1e6 - 962.9) < 0.2 and abs(de / 1e6 - 1711.6) < 0.2
    assert 1.77 < de / sp < 1.78


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


AGG_CHILD = r"""
import os, sys, json
sys.path.insert(0, sys.argv[1])
import torch.distributed as dist
import bench
dist.init_process_group("gloo")
r = dist.get_rank()
units, secs = bench.aggregate(1000.0 * (r + 1), 0.5 + r)
bench.barrier()
print(json.dumps({"rank": r, "units": units, "secs": secs}))
dist.destroy_process_group()
"""


def test_aggregate_two_ranks_gloo(tmp_path):
    script = tmp_path / "agg.py"
    script.write_text(AGG_CHILD)
    port = _free_port()
    procs = []
    for r in range(2):
        env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(r),
                   WORLD_SIZE="2", LOCAL_RANK=str(r))
        procs.append(subprocess.Popen([sys.executable, str(script), ROOT], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = [p.communicate(timeout=120) for p in procs]
    for p, (o, e) in zip(procs, outs):
        assert p.returncode == 0, e
    res = [json.loads(o.strip().splitlines()[-1]) for o, _ in outs]
    for d in res:
        assert d["units"] == 3000.0 and d["secs"] == 1.5  # sum of units, slowest rank


def test_reference_arm_prints_one_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "3", "--warmup", "3", "--ref-seconds", "2",
                          "--workload", "single_4096"],
                         capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"


def test_reference_arm_at_a_small_batch_names_the_spmm_metric():
    """--batch B: the oracle runs one SpMV per token on the row sample, and the
    line carries the same metric and batch as the GPU arm's --batch line."""
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--batch", "4", "--steps", "3", "--warmup", "3", "--ref-seconds", "2",
                          "--workload", "single_4096"],
                         capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr
    d = json.loads([l for l in out.stdout.splitlines() if l.strip()][-1])
    assert d["metric"] == bench.batch_metric(4) != bench.METRIC
    assert "batch 4" in d["config"]["workload"] and "4 tokens" in d["cpu_baseline"]["sample"]
    assert d["value"] > 0
    assert bench.batch_metric(1) == bench.METRIC


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="1")
    out = subprocess.run([sys.executable, "-c",
                          f"import sys; sys.path.insert(0, {ROOT!r}); import bench; "
                          "a = bench.parse(['--impl', 'reference', '--steps', '3', '--warmup', '3']);"
                          "print(bench.run_reference(a))"],
                         capture_output=True, text=True, env=env, timeout=120)
    assert out.returncode == 0 and out.stdout.strip() == "None"


def test_warmup_floor():
    with pytest.raises(SystemExit):
        bench.parse(["--warmup", "2"])


def test_prefill_reference_arm_and_flop_accounting():
    mats = bench.WORKLOADS["llama33_70b_layer"]
    assert bench.prefill_flops(mats, 2) == 2 * 2 * sum(r * c for _, r, c in mats)
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--prefill", "512", "--ref-seconds", "4", "--workload", "single_4096"],
                         capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    d = json.loads(lines[-1])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["metric"] == bench.PREFILL_METRIC


def test_prefill_argument_checks():
    assert bench.parse(["--prefill", "2048"]).prefill == 2048
    with pytest.raises(SystemExit):
        bench.parse(["--prefill", "64", "--batch", "4"])
    with pytest.raises(SystemExit):
        bench.parse(["--prefill", "-1"])


def test_default_line_sections_can_be_switched_off():
    """The default run times the headline plus the other workloads, the step at
    2..8 tokens, the fused SwiGLU step and the layer's prefill; each extra
    section has a switch, and the slot widths the small-batch section times are
    the ones nm_spmm pads to."""
    a = bench.parse([])
    assert a.side and a.small_batch and a.prefill_summary and a.batch == 1
    b = bench.parse(["--no-side", "--no-small-batch", "--no-prefill-summary"])
    assert not (b.side or b.small_batch or b.prefill_summary)
    assert bench.SMALL_BATCHES == (2, 4, 6, 8)
    assert bench.PREFILL_SUMMARY_TOKENS == (64, 256)


def test_clock_record_keeps_the_headline_window_apart(tmp_path):
    """nvidia-smi samples are kept only inside the timed windows; the first
    window (the headline's) gets a record of its own, so a power cap reached by
    a later section (the dense GEMMs) does not hide a clean headline record."""
    import datetime
    cs = bench.ClockSampler.__new__(bench.ClockSampler)
    cs.proc = object()
    t0 = datetime.datetime(2026, 1, 1, 12, 0, 0)
    rows = []
    for k in range(30):
        ts = t0 + datetime.timedelta(milliseconds=100 * k)
        cap = "Active" if k >= 20 else "Not Active"
        rows.append(f"{ts:%Y/%m/%d %H:%M:%S.%f}, 2070, 2070, {900 + k}, 0x0, Not Active, "
                    f"Not Active, Not Active, {cap}")
    p = tmp_path / "clocks.csv"
    p.write_text("\n".join(rows) + "\n")
    cs.path = str(p)
    cs.windows = [[t0, t0 + datetime.timedelta(milliseconds=950)],
                  [t0 + datetime.timedelta(milliseconds=1950), t0 + datetime.timedelta(seconds=3)]]
    s = cs.summary()
    assert s["reasons"] == ["sw_power_cap"] and s["samples"] == 20
    h = s["headline_window"]
    assert h["reasons"] == [] and h["samples"] == 10 and h["sm_mhz"] == 2070.0
