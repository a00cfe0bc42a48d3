"""Host-side logic of bench.py that needs no GPU: the clock sampler.

A fake `nvidia-smi` on PATH prints timestamped samples; the sampler must keep
only those inside the timed region and report throttle reasons from them.
"""
import os
import stat
import sys
import textwrap
import time

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _fake_smi(tmp_path, body):
    exe = tmp_path / "nvidia-smi"
    exe.write_text("#!" + sys.executable + "\n" + textwrap.dedent(body))
    exe.chmod(exe.stat().st_mode | stat.S_IXUSR)
    return str(tmp_path)


FAKE = """
import datetime, sys, time
# one sample every 20 ms; a throttle reason shows only after the first 0.3 s
t0 = time.time()
while True:
    now = time.time()
    stamp = datetime.datetime.fromtimestamp(now).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    hot = "Active" if now - t0 > 0.3 else "Not Active"
    sm = 1500 if now - t0 > 0.3 else 2070
    print(f"{stamp}, 0, {sm}, 2070, 900.5, 0x0, Not Active, {hot}, Not Active, Not Active", flush=True)
    time.sleep(0.02)
"""


def test_clocks_keep_only_timed_region(tmp_path, monkeypatch):
    bench = pytest.importorskip("bench")
    monkeypatch.setenv("PATH", _fake_smi(tmp_path, FAKE) + os.pathsep + os.environ["PATH"])
    c = bench.Clocks(0)
    c.start()
    c.mark(0)
    time.sleep(0.12)
    c.mark(1)
    out = c.stop()
    assert out["samples"] >= 2
    assert out["sm_mhz"] == 2070.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == []


def test_clocks_report_throttle_inside_region(tmp_path, monkeypatch):
    bench = pytest.importorskip("bench")
    monkeypatch.setenv("PATH", _fake_smi(tmp_path, FAKE) + os.pathsep + os.environ["PATH"])
    c = bench.Clocks(0)
    c.start()
    time.sleep(0.4)
    c.mark(0)
    time.sleep(0.1)
    c.mark(1)
    out = c.stop()
    assert out["reasons"] == ["hw_thermal_slowdown"]
    assert out["sm_mhz"] == 1500.0


def test_clocks_without_nvidia_smi(tmp_path, monkeypatch):
    bench = pytest.importorskip("bench")
    monkeypatch.setenv("PATH", str(tmp_path))
    c = bench.Clocks(0)
    c.start()
    c.mark(0)
    c.mark(1)
    assert c.stop()["reasons"] == ["nvidia-smi unavailable"]


def test_ctx_len_override():
    """--ctx-len replaces a fixed-length workload's context length only."""
    import argparse
    bench = pytest.importorskip("bench")
    w = bench._workload(argparse.Namespace(workload="qwen35_a3b_32k", ctx_len=2048))
    assert w.ctx_len == 2048 and w.draft.D == 2048 and w.batch == 4
    w0 = bench._workload(argparse.Namespace(workload="qwen35_a3b_32k", ctx_len=0))
    assert w0.ctx_len == 32768
    with pytest.raises(SystemExit):
        bench._workload(argparse.Namespace(workload="qwen3_8b_b32_ragged", ctx_len=2048))
