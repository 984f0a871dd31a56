"""bench.py's host logic on the CPU: the bytes each path reads (the roofline's
numerator) and when a recorded DRAM-traffic figure may be reported."""
import json
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from speculative_decoding_verification_20_gb300 import workloads  # noqa: E402


def test_bytes_by_path_v128k_is_all_streaming():
    """Every sequence of the v128k recipe streams (top-k 50): (2 * 7 + 1) rows of
    128256 bf16 logits each, 985,006,080 bytes at the bench's B = 256."""
    wl = workloads.make("v128k", seed=0, B=8)
    b = bench.bytes_by_path(wl, 256)
    assert b == {"stream": 8 * 15 * 128256 * 2, "free": 0, "dense": 0}
    assert 256 * 15 * 128256 * 2 == 985_006_080


def test_bytes_by_path_splits_ragged_by_row_parameters():
    """Greedy rows stream; rows with no top-k take the whole-row path; each row
    counts (2 gamma_b + 1) V sizeof bytes."""
    wl = workloads.make("ragged", seed=0)
    b = bench.bytes_by_path(wl, 256)
    T = wl.temperature.numpy()
    gam = wl.gammas()
    row = (2 * gam + 1) * wl.V * 4
    assert b["stream"] == int(row[T == 0].sum()) and b["free"] == int(row[T != 0].sum()) and b["dense"] == 0
    assert b["stream"] > 0 and b["free"] > 0


def test_bytes_by_path_large_top_k_goes_dense():
    wl = workloads.make("v32k", seed=0, B=4)
    wl.top_k = torch.full((4,), 1000, dtype=torch.int32)
    b = bench.bytes_by_path(wl, 256)
    assert b["dense"] == 4 * 11 * 32000 * 2 and b["stream"] == 0 and b["free"] == 0


def test_recorded_traffic_only_for_its_kernel_full_batch_and_sources():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)
    for wl, r in rec.items():
        # a record counts only while its kernel's sources are those it was captured with
        current = r["kernel_hash"] == bench.kernel_hash(r["path"])
        assert bench.recorded_traffic(wl, r["path"], True) == (r["bytes_per_launch"] if current else None)
        assert bench.recorded_traffic(wl, r["path"], False) is None  # another batch size
        other = "free" if r["path"] == "stream" else "stream"
        assert bench.recorded_traffic(wl, other, True) is None  # another kernel
    assert bench.recorded_traffic("tiny", "free", True) is None  # no capture recorded


def test_kernel_hash_covers_each_kernels_sources():
    for path, files in bench.KERNEL_SOURCES.items():
        assert all(os.path.exists(os.path.join(ROOT, f)) for f in files)
        assert len(bench.kernel_hash(path)) == 16
    assert bench.kernel_hash("stream") != bench.kernel_hash("free")


def test_bytes_by_path_shared_noise_splits_unfiltered_rows():
    """Under the shared-noise rule only the gamma_b + 1 target rows are read; rows
    with neither top-k nor top-p (T > 0) take the one-pass kernel, top-p rows the
    whole-row kernel, greedy and top-k rows the streaming path."""
    wl = workloads.make("ragged", seed=0)
    wl.top_p = torch.tensor([1.0 if b % 3 == 0 else 0.9 for b in range(wl.B)], dtype=torch.float32)
    b = bench.bytes_by_path(wl, 256, "gumbel")
    T = wl.temperature.numpy()
    P = wl.top_p.numpy()
    row = (wl.gammas() + 1) * wl.V * 4
    assert b["stream"] == int(row[T == 0].sum())
    assert b["gumbel"] == int(row[(T != 0) & (P >= 1.0)].sum()) > 0
    assert b["free"] == int(row[(T != 0) & (P < 1.0)].sum()) > 0
    assert b["dense"] == 0
    assert "gumbel" not in bench.bytes_by_path(wl, 256)  # the sampling rule has no such path


def test_launches_per_step_counts_the_one_pass_kernel():
    assert bench.launches_per_step("sampling") == 6
    assert bench.launches_per_step("gumbel") == 7
    assert bench.launches_per_step("kseq") == 6


def test_recorded_instructions_only_for_its_kernel_full_batch_and_sources():
    with open(os.path.join(ROOT, "profiles", "instructions.json")) as f:
        rec = json.load(f)
    for key, r in rec.items():
        rule, wl = key.split(":")
        current = r["kernel_hash"] == bench.kernel_hash(r["path"])
        assert bench.recorded_instructions(rule, wl, r["path"], True) == (
            r["thread_inst_per_launch"] if current else None)
        assert bench.recorded_instructions(rule, wl, r["path"], False) is None
        assert bench.recorded_instructions(rule, wl, "stream", True) is None
