"""Host logic of bench.py that needs no GPU: the launch count it claims for
the driver legs follows the library's batching rule (units of at most 2^24
elements batched up to 256 per launch, a unit above that size launched on
its own)."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_model_launches_follow_the_batching_rule():
    # 12 GPT-2 small blocks (7.09 M elements): one group, an update and a gather
    assert bench.model_launches(12, 7087872, 1) == 2
    # units above the size limit: one update and one gather each
    assert bench.model_launches(12, 855654400, 1) == 24
    # 200 units of 50,000: one group, an update and a gather
    assert bench.model_launches(200, 50000, 1) == 2
    assert bench.model_launches(200, 50000, 2) == 3
    assert bench.model_launches(200, 50000, 0) == 1
    # 500 units: groups of 256 and 244
    assert bench.model_launches(500, 20000, 1) == 4
    # 256 fill one group; 257 leave one unit, launched on its own
    assert bench.model_launches(256, 1000, 1) == 2
    assert bench.model_launches(257, 1000, 1) == 4
    # the size limit is inclusive
    assert bench.model_launches(3, 1 << 24, 1) == 2
    assert bench.model_launches(3, (1 << 24) + 8, 1) == 6
    assert bench.GROUP_MAX_UNITS == 256 and bench.GROUP_MAX_NUMEL == 1 << 24


def test_batching_constants_match_the_library():
    import re
    src = open(os.path.join(ROOT, "sharded_fsdp_reduce_gb300", "csrc", "group.cuh")).read()
    assert int(re.search(r"#define FSDP_GROUP_MAX (\d+)", src).group(1)) == bench.GROUP_MAX_UNITS
    assert 1 << int(re.search(r"#define FSDP_GROUP_MAX_NUMEL_LOG2 (\d+)", src).group(1)) == bench.GROUP_MAX_NUMEL


def test_e2e_reports_the_faster_form_with_the_other_beside_it():
    import argparse
    a = argparse.Namespace(e2e_read_params=False)
    e = {"steps": 10, "h2d_bytes_per_step": 13690470400, "d2h_bytes_per_step": 4,
         "copy_pipeline_ms": 86.4, "zero_copy_ms": 69.3, "bare_h2d_ms": 79.4}
    r = bench.e2e_record(e, 66741043200, a)
    assert r["path"] == "zero_copy" and r["ms_per_step"] == 69.3
    assert r["value"] == round(66741043200 / 69.3e-3 / 1e9, 2)
    assert r["copy_pipeline"]["ms_per_step"] == 86.4 and "zero_copy" not in r
    assert r["bare_h2d_over_e2e"] == round(79.4 / 69.3, 4)
    assert r["h2d_bytes_per_step"] == 13690470400 and r["d2h_bytes_per_step"] == 4
    e.update(copy_pipeline_ms=66.4, zero_copy_ms=69.2)
    r = bench.e2e_record(e, 66741043200, argparse.Namespace(e2e_read_params=True))
    assert r["path"] == "copy_pipeline" and r["zero_copy"]["ms_per_step"] == 69.2
    assert r["d2h"] == "compute-dtype parameters"
    assert bench.e2e_record({"unavailable": "pinned host buffers: out of memory"}, 1, a) == {
        "unavailable": "pinned host buffers: out of memory"}
