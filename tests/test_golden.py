"""Checks against the fixtures in tests/golden/.

``page_facts.json`` holds numbers the pages print (shapes, defaults, the gate
bound); the workloads and constants used here must agree with them.
``oracle_regression.json`` is written by ``make_oracle_regression.py`` from
the oracle alone and guards the oracle against unnoticed changes.
"""
import json
import os

import numpy as np

import kda_inputs as ki

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def facts():
    with open(os.path.join(GOLDEN, "page_facts.json")) as f:
        return {k: v["value"] for k, v in json.load(f).items() if not k.startswith("_")}


def test_small_workloads_match_page_shapes():
    f = facts()["bench_small"]
    for name in ("fixed_bf16_h8_t1024", "packed_bf16_h8_t1024_4seg"):
        w = ki.WORKLOADS[name]
        assert (w.B, w.H, w.T, w.K, w.V, w.dtype) == (f["B"], f["H"], f["T"], f["K"], f["V"], f["dtype"])
    segs = ki.WORKLOADS["packed_bf16_h8_t1024_4seg"].segments
    assert len(segs) == f["packed_segments"] and sum(segs) == f["T"]
    bounds = np.cumsum(segs)[:-1]
    assert not np.any(bounds % 64 == 0)   # "four non-64-aligned segments"


def test_representative_workloads_match_page_shapes():
    f = facts()["bench_representative"]
    for name in ("fixed_bf16_h32_t8192", "packed_bf16_h32_t8192_25seg"):
        w = ki.WORKLOADS[name]
        assert (w.B, w.H, w.T, w.K, w.V, w.dtype) == (f["B"], f["H"], f["T"], f["K"], f["V"], f["dtype"])
    segs = ki.WORKLOADS["packed_bf16_h32_t8192_25seg"].segments
    assert len(segs) == f["packed_segments"] and sum(segs) == f["T"]
    assert max(segs) - min(segs) <= 1    # balanced


def test_gate_recipe_within_page_bound():
    lo, hi = facts()["gate_lower_bound_range"]
    x = ki.make_inputs(ki.custom_workload(1, 4096, 2, 32, 8), seed=5)
    assert float(x["g"].min()) >= lo and float(x["g"].max()) <= hi


def test_segment_ids_convention():
    f = facts()["segment_ids_convention"]
    seg = ki.segment_ids_from_lengths(1, 10, [3, ("pad", 2), 4])
    assert int(seg[0, 0]) == f["first_id"] and int(seg[0, 3]) == f["padding_id"]


def test_oracle_regression_fixture():
    import make_oracle_regression as M
    with open(os.path.join(GOLDEN, "oracle_regression.json")) as fh:
        ref = json.load(fh)
    o, fs = M.compute()
    np.testing.assert_allclose(o.ravel(), ref["o"], rtol=1e-14, atol=1e-16)
    np.testing.assert_allclose(fs.ravel(), ref["final_state"], rtol=1e-14, atol=1e-16)
