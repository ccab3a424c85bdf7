"""Shared helpers for the GPU parity tests: run the CUDA path through the C
ABI and the fp64 oracle on the same seeded inputs, and compare them with the
tolerances of the method's precision contract:

* fp32 q/k/v: max-abs error <= 1e-4 on o and final_state;
* bf16 q/k/v (fp32 accumulation): max-abs <= 2e-2 and relative L2
  ||x - x_ref|| / ||x_ref|| <= 1e-2 on o and final_state.
"""
from __future__ import annotations

import numpy as np
import torch

import kda_inputs as ki
import oracle

TOL_F32_MAXABS = 1e-4
TOL_BF16_MAXABS = 2e-2
TOL_BF16_RELL2 = 1e-2


def to_dev(x, dev="cuda"):
    return None if x is None else x.to(dev)


def run_gpu(x, impl="auto", v_tile=0, output_final_state=True, device="cuda",
            initial_state=None, workspace=None):
    import gated_delta_rule_21_gb300 as kda
    S0 = x["initial_state"] if initial_state is None else initial_state
    o, fs = kda.chunk_fwd(to_dev(x["q"], device), to_dev(x["k"], device), to_dev(x["v"], device),
                          to_dev(x["g"], device), to_dev(x["beta"], device), scale=x["scale"],
                          initial_state=to_dev(S0, device),
                          segment_ids=to_dev(x["segment_ids"], device),
                          output_final_state=output_final_state, impl=impl, v_tile=v_tile,
                          workspace=workspace)
    torch.cuda.synchronize()
    return o, fs


def run_oracle(x, initial_state=None):
    S0 = x["initial_state"] if initial_state is None else initial_state
    return oracle.kda_forward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"],
                              initial_state=S0, segment_ids=x["segment_ids"])


def errors(got, ref):
    got = got.detach().to("cpu", torch.float64).numpy() if isinstance(got, torch.Tensor) else got
    d = np.abs(got - ref)
    nref = np.linalg.norm(ref)
    rel = np.linalg.norm(got - ref) / nref if nref > 0 else float(np.linalg.norm(got - ref))
    return float(d.max()) if d.size else 0.0, float(rel)


def assert_parity(got, ref, bf16, what):
    mx, rel = errors(got, ref)
    if bf16:
        assert mx <= TOL_BF16_MAXABS and rel <= TOL_BF16_RELL2, \
            f"{what}: max-abs {mx:.3e} (tol {TOL_BF16_MAXABS}), rel-L2 {rel:.3e} (tol {TOL_BF16_RELL2})"
    else:
        assert mx <= TOL_F32_MAXABS, f"{what}: max-abs {mx:.3e} (tol {TOL_F32_MAXABS})"
    return mx, rel


def skip_unless_supported(w, impl):
    """Skip a test whose implementation does not serve the shape (the ABI
    rejects it with KDA_ERR_UNSUPPORTED, which test_abi covers)."""
    import pytest
    import gated_delta_rule_21_gb300 as kda
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    if impl == "split":
        ok = kda.workspace_size(w.B, w.T, w.H, w.K, w.V, dt, w.segments is not None,
                                impl="split") > 0
    else:
        ok = kda.impl_available(impl, w.B, w.T, w.H, w.K, w.V, dt)
    if not ok:
        pytest.skip(f"{impl} does not serve {w.name}")


def check_workload(w, seed=0, impl="auto", v_tile=0):
    skip_unless_supported(w, impl)
    x = ki.make_inputs(w, seed=seed)
    o, fs = run_gpu(x, impl=impl, v_tile=v_tile)
    o_ref, fs_ref = run_oracle(x)
    bf16 = w.dtype == "bf16"
    e1 = assert_parity(o, o_ref, bf16, f"{w.name} o")
    e2 = assert_parity(fs, fs_ref, bf16, f"{w.name} final_state")
    return e1, e2
