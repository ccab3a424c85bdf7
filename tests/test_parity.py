"""GPU parity: the CUDA chunked forward (through the C ABI) against the fp64
oracle on the same seeded inputs, element by element, for the five
workloads of the pages and for edge cases of the packed format.
"""
import pytest
import torch

import kda_inputs as ki
from kda_testlib import (assert_parity, check_workload, errors, run_gpu, run_oracle,
                         skip_unless_supported, to_dev)

pytestmark = pytest.mark.gpu

# auto = the split tensor-core path for bf16 K = V = 128 without segment ids
# (its workspace is allocated by the binding), the fused one with them.
IMPLS = ["auto", "tc", "simt"]
NAMED = ["tiny_fp32_h2_t128_d32", "fixed_bf16_h8_t1024", "packed_bf16_h8_t1024_4seg",
         "fixed_bf16_h32_t8192", "packed_bf16_h32_t8192_25seg"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import gated_delta_rule_21_gb300 as kda
    from gated_delta_rule_21_gb300 import build
    build.build()
    kda.lib()


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("name", NAMED)
def test_named_workload(name, impl):
    check_workload(ki.WORKLOADS[name], impl=impl)


EDGE = {
    "ragged_T100": dict(B=1, T=100, H=2, K=128, V=128),
    "T1": dict(B=1, T=1, H=1, K=128, V=128),
    "T63": dict(B=1, T=63, H=1, K=128, V=128),
    "T65_S0": dict(B=1, T=65, H=2, K=128, V=128, init_state_std=0.1),
    "B2_H1": dict(B=2, T=200, H=1, K=128, V=128, init_state_std=0.1),
    "K64_V64": dict(B=1, T=150, H=3, K=64, V=64, init_state_std=0.1),
    "K64_V128": dict(B=1, T=130, H=2, K=64, V=128),
    "K128_V32": dict(B=1, T=130, H=2, K=128, V=32),
    "K32_V64_f32": dict(B=2, T=90, H=2, K=32, V=64, dtype="f32"),
    "f32_K128": dict(B=1, T=200, H=2, K=128, V=128, dtype="f32", init_state_std=0.1),
    "len1_segments": dict(B=1, T=140, H=2, K=128, V=128, init_state_std=0.1,
                          segments=[1, 1, 64, 1, 70, 1]),
    "boundary_at_64": dict(B=1, T=256, H=2, K=128, V=128, segments=[64, 128, 64]),
    "long_run_and_pads": dict(B=2, T=400, H=2, K=128, V=128, init_state_std=0.1,
                              segments=[[("pad", 5), 300, ("pad", 10), 70],
                                        [130, 1, ("pad", 64), 200]]),
    "all_padding_row": dict(B=2, T=96, H=2, K=128, V=128, init_state_std=0.1,
                            segments=[[90], [("pad", 96)]]),
    "repeated_id_after_pad": dict(B=1, T=160, H=1, K=128, V=128, init_state_std=0.1,
                                  segments=[50, ("pad", 3), 100]),
    "padding_rows_between": dict(B=4, T=96, H=2, K=128, V=128, init_state_std=0.1,
                                 segments=[[("pad", 96)], [40, ("pad", 6), 50],
                                           [("pad", 96)], [96]]),
}


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("case", sorted(EDGE))
def test_edge_case(case, impl):
    w = ki.custom_workload(name=case, **EDGE[case])
    skip_unless_supported(w, impl)
    x = ki.make_inputs(w, seed=1)
    if case == "repeated_id_after_pad":
        seg = x["segment_ids"]
        seg[seg == 2] = 1        # same id on both sides of the padding
    o, fs = run_gpu(x, impl=impl)
    o_ref, fs_ref = run_oracle(x)
    bf16 = w.dtype == "bf16"
    assert_parity(o, o_ref, bf16, f"{case} o")
    assert_parity(fs, fs_ref, bf16, f"{case} final_state")
    if x["segment_ids"] is not None:
        pad = (x["segment_ids"] == 0).numpy()
        assert torch.all(o.cpu()[torch.from_numpy(pad)] == 0)


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("gval", [0.0, -5.0])
def test_constant_gate_edges(gval, impl):
    """g = 0 (pure delta rule) and g = -5 on every channel (the contract
    edge, where the chunk-wide exponent span is 320)."""
    w = ki.custom_workload(1, 192, 2, 128, 128, init_state_std=0.1)
    x = ki.make_inputs(w, seed=2)
    x["g"] = torch.full_like(x["g"], gval)
    o, fs = run_gpu(x, impl=impl)
    o_ref, fs_ref = run_oracle(x)
    assert_parity(o, o_ref, True, "o")
    assert_parity(fs, fs_ref, True, "final_state")


@pytest.mark.parametrize("impl", IMPLS)
def test_split_sequence_state_handoff(impl):
    """[0, t) then [t, T) with final -> initial state equals one pass."""
    w = ki.custom_workload(1, 300, 2, 128, 128, init_state_std=0.1)
    x = ki.make_inputs(w, seed=3)
    o, fs = run_gpu(x, impl=impl)
    cut = 137
    xa = {**x, **{n: x[n][:, :cut].contiguous() for n in ("q", "k", "v", "g", "beta")}}
    xb = {**x, **{n: x[n][:, cut:].contiguous() for n in ("q", "k", "v", "g", "beta")}}
    oa, fa = run_gpu(xa, impl=impl)
    ob, fb = run_gpu(xb, impl=impl, initial_state=fa.cpu())
    o_ref, fs_ref = run_oracle(x)
    assert_parity(torch.cat([oa, ob], 1), o_ref, True, "split o")
    assert_parity(fb, fs_ref, True, "split final_state")
    mx, _ = errors(torch.cat([oa, ob], 1).float(), o.double().cpu().numpy())
    assert mx <= 2e-2


@pytest.mark.parametrize("impl", IMPLS)
def test_row_independence_and_determinism(impl):
    w = ki.custom_workload(2, 130, 3, 128, 128, init_state_std=0.1)
    x = ki.make_inputs(w, seed=4)
    o1, f1 = run_gpu(x, impl=impl)
    o2, f2 = run_gpu(x, impl=impl)
    assert torch.equal(o1, o2) and torch.equal(f1, f2)          # bitwise repeatable
    x2 = dict(x)
    x2["v"] = x["v"].clone()
    x2["v"][1] += 1.0
    o3, f3 = run_gpu(x2, impl=impl)
    assert torch.equal(o3[0], o1[0]) and torch.equal(f3[0], f1[0])
    assert not torch.equal(o3[1], o1[1])


def test_no_final_state_requested():
    w = ki.WORKLOADS["packed_bf16_h8_t1024_4seg"]
    x = ki.make_inputs(w, seed=0)
    o, fs = run_gpu(x, output_final_state=False)
    assert fs is None
    o_ref, _ = run_oracle(x)
    assert_parity(o, o_ref, True, "o")


def test_device_status_clean_and_workspace_reuse():
    import gated_delta_rule_21_gb300 as kda
    w = ki.WORKLOADS["packed_bf16_h8_t1024_4seg"]
    x = ki.make_inputs(w, seed=0)
    ws = kda.alloc_workspace(w.B, w.T, w.H, w.K, w.V, torch.bfloat16, True)
    for _ in range(3):   # the run-builder's counters return to zero
        o, fs = run_gpu(x, workspace=ws)
    assert kda.read_device_status(ws) == 0
    o_ref, fs_ref = run_oracle(x)
    assert_parity(o, o_ref, True, "o after workspace reuse")


def test_split_packed_with_explicit_runs_bound():
    """Packed input on the split path with a workspace sized for exactly the
    runs present (four per row)."""
    import gated_delta_rule_21_gb300 as kda
    w = ki.WORKLOADS["packed_bf16_h8_t1024_4seg"]
    x = ki.make_inputs(w, seed=5)
    ws = kda.alloc_workspace(w.B, w.T, w.H, w.K, w.V, torch.bfloat16, True, impl="split",
                             max_runs_per_row=4)
    o, fs = run_gpu(x, impl="split", workspace=ws)
    assert kda.read_device_status(ws) == 0
    o_ref, fs_ref = run_oracle(x)
    assert_parity(o, o_ref, True, "o")
    assert_parity(fs, fs_ref, True, "final_state")


def test_split_packed_overflow_is_reported_not_computed():
    """More runs than the workspace was sized for: the split path reports
    KDA_DEVICE_WORKSPACE in the status word instead of writing garbage past
    its items, and the context stays usable."""
    import gated_delta_rule_21_gb300 as kda
    lens = [1] * 120 + [8]          # 121 runs in one row of 128 tokens
    w = ki.custom_workload(1, 128, 2, 128, 128, segments=lens)
    x = ki.make_inputs(w, seed=6)
    ws = kda.alloc_workspace(w.B, w.T, w.H, w.K, w.V, torch.bfloat16, True, impl="split",
                             max_runs_per_row=1)
    run_gpu(x, impl="split", workspace=ws)
    assert kda.read_device_status(ws) & 0x4
    kda.clear_device_status(ws)
    o, fs = run_gpu(x, impl="tc")      # the same inputs on the fused path
    o_ref, fs_ref = run_oracle(x)
    assert_parity(o, o_ref, True, "o")


def test_misaligned_pointer_rejected_on_gpu():
    import gated_delta_rule_21_gb300 as kda
    w = ki.custom_workload(1, 64, 1, 128, 128)
    x = ki.make_inputs(w)
    buf = torch.zeros(64 * 128 + 8, dtype=torch.bfloat16, device="cuda")
    qm = buf[1:1 + 64 * 128].view(1, 64, 1, 128)      # 2-byte offset
    with pytest.raises(kda.KdaError) as e:
        kda.chunk_fwd(qm, to_dev(x["k"]), to_dev(x["v"]), to_dev(x["g"]), to_dev(x["beta"]))
    assert e.value.status == 3


@pytest.mark.parametrize("v_tile", [32, 64, 128])
@pytest.mark.parametrize("name", ["fixed_bf16_h8_t1024", "packed_bf16_h8_t1024_4seg"])
def test_split_value_tiles(name, v_tile):
    """The split path's recurrence with either value-tile width (32 or 64
    columns per CTA) matches the oracle."""
    import gated_delta_rule_21_gb300 as kda
    w = ki.WORKLOADS[name]
    skip_unless_supported(w, "split")
    x = ki.make_inputs(w, seed=3)
    has_seg = w.segments is not None
    ws = kda.alloc_workspace(w.B, w.T, w.H, w.K, w.V, torch.bfloat16, has_seg, impl="split",
                             max_runs_per_row=len(w.segments) if has_seg else None)
    o, fs = run_gpu(x, impl="split", v_tile=v_tile, workspace=ws)
    assert kda.read_device_status(ws) == 0
    o_ref, fs_ref = run_oracle(x)
    assert_parity(o, o_ref, True, f"{name} v_tile {v_tile} o")
    assert_parity(fs, fs_ref, True, f"{name} v_tile {v_tile} final_state")


PACKED_EDGE = ["len1_segments", "boundary_at_64", "long_run_and_pads", "all_padding_row",
               "repeated_id_after_pad", "padding_rows_between"]


@pytest.mark.parametrize("case", PACKED_EDGE)
def test_split_packed_edge_cases(case):
    """The packed edge cases on the split path, whose work items come from a
    per-row chunk table: rows without a run before, between and after rows
    with runs, runs of one token, run boundaries on chunk edges."""
    import gated_delta_rule_21_gb300 as kda
    w = ki.custom_workload(name=case, **EDGE[case])
    skip_unless_supported(w, "split")
    x = ki.make_inputs(w, seed=1)
    seg = x["segment_ids"]
    if case == "repeated_id_after_pad":
        seg[seg == 2] = 1
    prev = torch.cat([torch.zeros_like(seg[:, :1]), seg[:, :-1]], 1)
    max_runs = int(((seg != 0) & (seg != prev)).sum(1).max())
    ws = kda.alloc_workspace(w.B, w.T, w.H, w.K, w.V, torch.bfloat16, True, impl="split",
                             max_runs_per_row=max(max_runs, 1))
    o, fs = run_gpu(x, impl="split", workspace=ws)
    assert kda.read_device_status(ws) == 0
    o_ref, fs_ref = run_oracle(x)
    assert_parity(o, o_ref, True, f"{case} o")
    assert_parity(fs, fs_ref, True, f"{case} final_state")
    pad = (seg == 0).numpy()
    assert torch.all(o.cpu()[torch.from_numpy(pad)] == 0)


@pytest.mark.parametrize("name", ["packed_bf16_h8_t1024_4seg", "packed_bf16_h32_t8192_25seg"])
def test_packed_in_benchmark_configuration(name):
    """The packed workloads through AUTO with a workspace sized for their runs
    per row, the configuration the benchmark times (the split path), against
    the oracle on every output."""
    import gated_delta_rule_21_gb300 as kda
    w = ki.WORKLOADS[name]
    skip_unless_supported(w, "split")
    x = ki.make_inputs(w, seed=0)
    ws = kda.alloc_workspace(w.B, w.T, w.H, w.K, w.V, torch.bfloat16, True, impl="auto",
                             max_runs_per_row=len(w.segments))
    o, fs = run_gpu(x, workspace=ws)
    assert kda.read_device_status(ws) == 0
    o_ref, fs_ref = run_oracle(x)
    assert_parity(o, o_ref, True, f"{name} o")
    assert_parity(fs, fs_ref, True, f"{name} final_state")


def _bf16_order_key(t):
    """bf16 bit patterns as integers ordered like the values (+0 and -0 equal)."""
    import numpy as np
    u = t.contiguous().view(torch.int16).numpy().astype(np.int32) & 0xFFFF
    mag = u & 0x7FFF
    return np.where(u & 0x8000, -mag, mag)


@pytest.mark.parametrize("name", ["fixed_bf16_h8_t1024", "packed_bf16_h8_t1024_4seg"])
def test_bf16_ulp_distance_report(name, capsys):
    """Diagnostic: the distance in bf16 ULPs between the kernel's o and the
    fp64 oracle rounded to bf16 (via fp32), over outputs with |o| at least
    1e-3 of the largest (near zero a ULP means nothing).  The only bound
    asserted follows from the rel-L2 tolerance of 1e-2: a relative error of
    1e-2 is at most about 5 ULPs of bf16 (8 significand bits), so the median
    must not exceed that."""
    import numpy as np
    w = ki.WORKLOADS[name]
    x = ki.make_inputs(w, seed=0)
    o, _ = run_gpu(x)
    o_ref, _ = run_oracle(x)
    ref = torch.from_numpy(np.asarray(o_ref)).to(torch.float32).to(torch.bfloat16)
    d_all = np.abs(_bf16_order_key(o.cpu()) - _bf16_order_key(ref))
    mag = np.abs(np.asarray(o_ref))
    # a distance across zero counts every binade in between, so the maximum
    # over small outputs says little; |o| >= 0.1 max is the well-scaled part
    for frac in (1e-3, 1e-1):
        d = d_all[mag >= frac * mag.max()]
        p50, p99, mx = np.percentile(d, 50), np.percentile(d, 99), d.max()
        exact = float(np.mean(d == 0))
        with capsys.disabled():
            print(f"\n{name}: bf16 ULP distance of o over the {d.size} outputs with |o| >= "
                  f"{frac:g} max: median {p50:.0f}, p99 {p99:.0f}, max {mx}, "
                  f"exact {100 * exact:.1f} %")
        if frac == 1e-3:
            assert p50 <= 5
