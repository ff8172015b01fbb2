"""Host logic of bench.py, no GPU: the max-over-ranks timing reduction on two
gloo ranks, the reference arm's rank rule, the kernel hash that keys the
stored ncu traffic, and the peaks the figures are reported against."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

_RANK_SCRIPT = r"""
import os, sys
sys.path.insert(0, {root!r})
import torch.distributed as dist
import bench
rank, world, _ = bench.dist_env()
dist.init_process_group("gloo")
v = bench._max_over_ranks(1.5 + 2.0 * rank, world)
print("MAX", v, flush=True)
dist.destroy_process_group()
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_max_over_ranks_two_gloo_ranks():
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2",
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, "-c", _RANK_SCRIPT.format(root=ROOT)], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True))
    outs = [p.communicate(timeout=120)[0] for p in procs]
    for p, out in zip(procs, outs):
        assert p.returncode == 0, out
        vals = [float(l.split()[1]) for l in out.splitlines() if l.startswith("MAX ")]
        assert vals == [3.5], out   # max(1.5, 3.5) on every rank


def test_reference_arm_other_ranks_do_no_work(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        steps, warmup, gpus = 2, 3, 2

    assert bench.run_reference(A()) == 0
    assert capsys.readouterr().out == ""


def test_kernel_hash_ignores_comments_not_code():
    src = "int a = 1; // one\n/* block\n comment */\nint b = 2;\n"
    assert bench._code_only(src) == bench._code_only("int a = 1;\nint b = 2; // two\n")
    assert bench._code_only(src) != bench._code_only("int a = 1;\nint b = 3;\n")


def test_stored_traffic_only_for_the_hashed_kernel(tmp_path, monkeypatch):
    rec = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    assert rec["dram_bytes_per_forward"] > 0
    (tmp_path / "profiles").mkdir()
    stale = dict(rec, kernel_hash="0" * 16)
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(stale))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_hash", lambda: "f" * 16)
    assert bench.stored_traffic() is None
    fresh = dict(rec, kernel_hash="f" * 16)
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(fresh))
    assert bench.stored_traffic() == rec["dram_bytes_per_forward"]


def test_tensor_peaks_follow_the_measured_bf16_figure(tmp_path, monkeypatch):
    """The batched figures' tensor peaks: the measured cuBLAS bf16 burst figure
    (MEASURED_PEAKS.json) for the bf16 numerics, and it times 13.5 / 2.25 (the
    dense FP4 to bf16 ratio of the nominal GB300 rates) for the MXFP4 one; the
    stated fallback without a measurement."""
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    bf, src = bench._bf16_peak()
    fp, src4 = bench._fp4_peak()
    assert bf == 1900.0 and "fallback" in src
    assert fp == pytest.approx(1900.0 * 6.0) and "fallback" in src4
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6700.0, "bf16_tflops": 2000.0}))
    bf, src = bench._bf16_peak()
    fp, src4 = bench._fp4_peak()
    assert bf == 2000.0 and "measured" in src
    assert fp == pytest.approx(12000.0) and "measured" in src4
    assert bench.measured_peaks() == (6700.0, "measured")
