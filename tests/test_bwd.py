"""GPU parity of the CUDA-core backward (kda_chunk_bwd_ex with KDA_IMPL_SIMT,
through the C ABI) against the fp64 backward oracle on the same seeded
inputs and upstream gradients, for every gradient, on fixed and packed
shapes, all supported (K, V), and heads sampled from the B1 H32 T8192
workload.  The tensor-core backward has its own file (test_bwd_tc.py).

Tolerance: the kernel computes in fp32 from the same (bf16 or fp32) input
values the oracle upcasts exactly, so the difference is fp32 rounding only
(unit 6e-8) accumulated over sums of K or V terms per token and over the
run's tokens; per gradient, max-abs <= 1e-3 * max|ref| + 1e-6 and
rel-L2 <= 1e-3.
"""
import numpy as np
import pytest
import torch

import kda_inputs as ki
import oracle
from kda_testlib import to_dev

pytestmark = pytest.mark.gpu

NAMES = ("dq", "dk", "dv", "dg", "dbeta", "d_initial")


def _run_both(w, seed=0, heads=None, impl="simt"):
    import gated_delta_rule_21_gb300 as kda
    x = ki.make_inputs(w, seed=seed)
    u = ki.make_upstream_grads(w, seed=seed)
    got = kda.chunk_bwd(to_dev(x["q"]), to_dev(x["k"]), to_dev(x["v"]), to_dev(x["g"]),
                        to_dev(x["beta"]), to_dev(u["d_o"]), scale=x["scale"],
                        initial_state=to_dev(x["initial_state"]),
                        segment_ids=to_dev(x["segment_ids"]), d_final=to_dev(u["d_final"]),
                        impl=impl)
    torch.cuda.synchronize()
    got = [t.cpu().numpy() for t in got]
    if heads is not None:   # heads are independent problems: the oracle takes a few
        hs = list(heads)
        sel = lambda a, axis: None if a is None else a[(slice(None),) * axis + (hs,)]
        x = dict(x, q=sel(x["q"], 2), k=sel(x["k"], 2), v=sel(x["v"], 2), g=sel(x["g"], 2),
                 beta=sel(x["beta"], 2), initial_state=sel(x["initial_state"], 1))
        u = dict(d_o=sel(u["d_o"], 2), d_final=sel(u["d_final"], 1))
        got = [sel(got[0], 2), sel(got[1], 2), sel(got[2], 2), sel(got[3], 2), sel(got[4], 2),
               sel(got[5], 1)]
    ref = oracle.kda_backward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"],
                              initial_state=x["initial_state"], segment_ids=x["segment_ids"],
                              d_o=u["d_o"], d_final=u["d_final"])
    return x, got, ref


def _check(name, got, ref, what):
    d = np.abs(got - ref)
    mx = float(d.max()) if d.size else 0.0
    scale = float(np.abs(ref).max()) if ref.size else 0.0
    nref = np.linalg.norm(ref)
    rel = float(np.linalg.norm(got - ref) / nref) if nref > 0 else float(np.linalg.norm(got - ref))
    assert mx <= 1e-3 * scale + 1e-6 and rel <= 1e-3, \
        f"{what} {name}: max-abs {mx:.3e} (ref max {scale:.3e}), rel-L2 {rel:.3e}"


CASES = {
    "f32_k32_v32_t128_s0": dict(B=1, T=128, H=2, K=32, V=32, dtype="f32", init_state_std=0.1),
    "bf16_k128_t200_s0": dict(B=1, T=200, H=2, K=128, V=128, init_state_std=0.1),
    "f32_k64_v128_t130": dict(B=2, T=130, H=2, K=64, V=128, dtype="f32"),
    "bf16_k128_v64_t77": dict(B=1, T=77, H=3, K=128, V=64, init_state_std=0.1),
    "T1": dict(B=1, T=1, H=1, K=128, V=128, init_state_std=0.1),
    "bf16_k32_v64_t70": dict(B=1, T=70, H=2, K=32, V=64, init_state_std=0.1),
    "f32_k128_v32_t9": dict(B=3, T=9, H=1, K=128, V=32, dtype="f32"),
    "len1_runs_only": dict(B=1, T=12, H=2, K=64, V=64, init_state_std=0.1,
                           segments=[1, 1, 1, ("pad", 1), 1, 1, 1, 1, 1, 1, 1, 1]),
    "packed": dict(B=2, T=300, H=2, K=128, V=128, init_state_std=0.1,
                   segments=[[("pad", 3), 100, 1, 1, ("pad", 5), 120, 70],
                             [64, 64, ("pad", 2), 170]]),
    "all_padding_row": dict(B=2, T=96, H=2, K=64, V=64, dtype="f32", init_state_std=0.1,
                            segments=[[90], [("pad", 96)]]),
    "padding_rows_between": dict(B=4, T=96, H=2, K=128, V=128, init_state_std=0.1,
                                 segments=[[("pad", 96)], [40, ("pad", 6), 50],
                                           [("pad", 96)], [96]]),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_backward_matches_oracle(case):
    w = ki.custom_workload(name=case, **CASES[case])
    x, got, ref = _run_both(w, seed=3)
    for name, a, b in zip(NAMES, got, ref):
        _check(name, a, b, case)
    if x["segment_ids"] is not None:
        pad = (x["segment_ids"] == 0).numpy()
        for name, a in zip(NAMES[:5], got[:5]):
            assert np.all(a[pad] == 0), f"{case} {name} not zero on padding"


@pytest.mark.parametrize("name", ["fixed_bf16_h32_t8192", "packed_bf16_h32_t8192_25seg"])
def test_backward_full_size_sampled_heads(name):
    """The full B1 H32 T8192 workload on the GPU; the oracle checks two heads."""
    x, got, ref = _run_both(ki.WORKLOADS[name], seed=0, heads=(0, 31))
    for n, a, b in zip(NAMES, got, ref):
        _check(n, a, b, name)


def test_backward_is_deterministic_and_workspace_reusable():
    import gated_delta_rule_21_gb300 as kda
    w = ki.custom_workload(B=1, T=150, H=2, K=128, V=128, init_state_std=0.1,
                           segments=[40, 60, 50])
    x = ki.make_inputs(w, seed=5)
    u = ki.make_upstream_grads(w, seed=5)
    ws = torch.zeros(kda.bwd_workspace_size(1, 150, 2, 128, 128, torch.bfloat16, True,
                                            impl="simt"),
                     dtype=torch.uint8, device="cuda")
    args = (to_dev(x["q"]), to_dev(x["k"]), to_dev(x["v"]), to_dev(x["g"]), to_dev(x["beta"]),
            to_dev(u["d_o"]))
    kw = dict(scale=x["scale"], initial_state=to_dev(x["initial_state"]),
              segment_ids=to_dev(x["segment_ids"]), d_final=to_dev(u["d_final"]), workspace=ws,
              impl="simt")
    a = kda.chunk_bwd(*args, **kw)
    b = kda.chunk_bwd(*args, **kw)
    for s, t in zip(a, b):
        assert torch.equal(s, t)
