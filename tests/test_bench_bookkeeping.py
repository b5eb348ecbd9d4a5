"""The benchmark's bookkeeping on the CPU: the kernels it names exist in the sources,
the committed DRAM-traffic records name known kernels and workloads, and the roofline
arithmetic of each kernel kind follows its algorithmic-bytes definition."""

import json
import os
import types

import numpy as np
import pytest

import bench
from shared_prefix_paged_gb300 import accounting, workloads

CSRC = os.path.join(bench.ROOT, "shared_prefix_paged_gb300", "csrc")


def test_every_named_kernel_is_defined_in_its_sources():
    for kernel, files in bench.KERNEL_SOURCES.items():
        text = ""
        for f in files:
            path = os.path.join(CSRC, f)
            assert os.path.exists(path), (kernel, f)
            with open(path, encoding="utf-8") as fh:
                text += fh.read()
        assert f"{kernel}(" in text, kernel  # the __global__ function itself


def test_traffic_records_name_known_kernels_and_workloads():
    with open(os.path.join(bench.ROOT, "profiles", "dram_traffic.json"), encoding="utf-8") as f:
        table = json.load(f)
    names = {b.name for b in (workloads.by_name(n) for n in ("decode", "chunked", "tiny"))}
    names.add("long_prefix_N256_P16384")
    for key, rec in table.items():
        kernel, workload = key.split("@")
        assert kernel in bench.KERNEL_SOURCES, key
        assert workload in names, key
        assert rec["bytes_per_launch"] > 0
        assert len(rec["source_sha"]) == 16
    # the headline kernel's record, while current (it reads None once the kernel's
    # sources change after the capture), is about its algorithmic bytes
    b = workloads.by_name("decode")
    assert "decode_cascade_kernel@" + b.name in table
    got = bench.committed_traffic("decode_cascade_kernel", b.name)
    if got is not None:
        assert 0.98 < got / accounting.cascade_min_bytes(b, 4096) < 1.02


@pytest.mark.parametrize("kernel", ["decode_cascade_kernel", "prefix_attn_kernel",
                                    "paged_attn_kernel", "paged_tc_kernel",
                                    "merge_slots_kernel"])
def test_roofline_entry_arithmetic(kernel):
    b = workloads.by_name("tiny")
    run = types.SimpleNamespace(cpl=256, prefix_ranges=2)
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0, "source": "test"}
    e = bench.roofline_entry(kernel, 10.0, b, run, peaks, b.name)
    rows = b.total_q * b.num_q_heads
    kvtok = accounting.kv_bytes_per_token(b.num_kv_heads, b.head_dim)
    if kernel == "decode_cascade_kernel":
        want = accounting.cascade_min_bytes(b, 256)
    elif kernel == "merge_slots_kernel":
        want = rows * (3 * (b.head_dim * 2 + 4) + b.head_dim * 2 + 4)
    elif kernel == "prefix_attn_kernel":
        want = 256 * kvtok + rows * b.head_dim * 2 + rows * (b.head_dim * 2 + 4)
    else:
        want = (int((b.seq_lens.astype(np.int64) - 256).sum()) * kvtok +
                rows * b.head_dim * 2 + rows * (b.head_dim * 2 + 4))
    assert e["algorithmic_bytes_per_launch"] == int(want)
    gbs = want / 10e-6 / 1e9
    assert e["frac"] == pytest.approx(max(gbs / 6000.0, e.get("tensor", {}).get("frac", 0.0)),
                                      abs=1e-4)
    assert e["bound"] in ("hbm", "tensor")
