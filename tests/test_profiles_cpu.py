"""The committed ncu evidence matches the kernel source it describes: the
pass-2 DRAM traffic the benchmark reports was captured on the current source
of passes 1 and 2 (the hash recorded beside it), and is close to the
algorithmic 28 bytes per parameter; every profile summary that records a
source hash records the current one."""
import glob
import json
import os
import re

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("workload,params", [("gpt2_1p5b_full", 1_557_611_264),
                                             ("gpt2_1p5b_nd16", 97_350_784)])
def test_traffic_record_is_for_the_current_kernel_source(workload, params):
    path = os.path.join(ROOT, "profiles", f"adam_pass2_{workload}_traffic.json")
    d = json.load(open(path))
    assert d["kernel_source_sha256_16"] == bench.kernel_source_hash(), \
        "the kernels changed since the traffic was captured: recapture it"
    t = bench.committed_traffic(workload)
    assert t is not None
    algorithmic = 28 * params
    assert d["algorithmic_bytes_per_launch"] == algorithmic
    # reads equal the algorithmic 14 B/param; part of the writes are still in
    # L2 when the launch ends
    assert 0.9 * algorithmic <= t <= 1.05 * algorithmic
    assert abs(d["dram_bytes_read"] - 14 * params) <= 0.001 * 14 * params


def test_profile_summaries_record_the_current_source():
    h = bench.kernel_source_hash()
    seen = 0
    for p in glob.glob(os.path.join(ROOT, "profiles", "*.md")):
        for rec in re.findall(r"first 16 hex\): ([0-9a-f]{16})", open(p).read()):
            assert rec == h, f"{os.path.basename(p)} was captured on another kernel source"
            seen += 1
    assert seen >= 3
