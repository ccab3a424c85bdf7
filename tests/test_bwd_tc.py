"""GPU parity of the tensor-core backward (kda_chunk_bwd_ex with KDA_IMPL_TC,
and KDA_IMPL_AUTO, which picks it for bf16 K = V = 128) against the fp64
backward oracle on the same seeded inputs and upstream gradients: every
gradient, on one chunk, several chunks, ragged last chunks, two rows, gates
at the contract's lower bound, with and without an initial state and
d_final, packed rows (runs of one token, runs across chunk boundaries,
padding, rows without a run), the item overflow report, and two heads of
the fixed and the packed B1 H32 T8192 workloads.

Tolerance: the bounds the forward's bf16 parity uses (relative L2 <= 1e-2;
max-abs <= 2e-2, here relative to each gradient's largest magnitude, since
gradients are not O(1) like o).  The kernels round to bf16 (unit 2^-9)
the operands of every product: the saved states S and dS', U and dU, the
items' w, Q e^G, A_qk, K e^{G_C-G}, T and K e^G, and the intermediate dT,
P, dw and dA tiles; each gradient sums such products over K = 128 or
C = 64 terms with fp32 accumulation, so its error is a few times 2^-9
relative to the sum of magnitudes (measured: rel-L2 2e-3 .. 7e-3).
"""
import numpy as np
import pytest
import torch

import kda_inputs as ki
import oracle
from kda_testlib import to_dev

pytestmark = pytest.mark.gpu

NAMES = ("dq", "dk", "dv", "dg", "dbeta", "d_initial")
TOL_RELL2 = 1e-2
TOL_MAXABS_REL = 2e-2


def _inputs(w, seed, g_fill=None, no_s0=False, no_dfinal=False):
    x = ki.make_inputs(w, seed=seed)
    u = ki.make_upstream_grads(w, seed=seed)
    if g_fill is not None:
        x["g"] = torch.full_like(x["g"], g_fill)
    if no_s0:
        x["initial_state"] = None
    if no_dfinal:
        u["d_final"] = None
    return x, u


def _gpu(x, u, impl="tc", want_d_initial=True, workspace=None):
    import gated_delta_rule_21_gb300 as kda
    dev = lambda t: None if t is None else to_dev(t)
    got = kda.chunk_bwd(dev(x["q"]), dev(x["k"]), dev(x["v"]), dev(x["g"]), dev(x["beta"]),
                        dev(u["d_o"]), scale=x["scale"], initial_state=dev(x["initial_state"]),
                        segment_ids=dev(x["segment_ids"]), d_final=dev(u["d_final"]),
                        want_d_initial=want_d_initial, impl=impl, workspace=workspace)
    torch.cuda.synchronize()
    return got


def _oracle(x, u, heads=None):
    if heads is not None:
        hs = list(heads)
        sel = lambda a, axis: None if a is None else a[(slice(None),) * axis + (hs,)]
        x = dict(x, q=sel(x["q"], 2), k=sel(x["k"], 2), v=sel(x["v"], 2), g=sel(x["g"], 2),
                 beta=sel(x["beta"], 2), initial_state=sel(x["initial_state"], 1))
        u = dict(d_o=sel(u["d_o"], 2), d_final=sel(u["d_final"], 1))
    return oracle.kda_backward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"],
                               initial_state=x["initial_state"], segment_ids=x["segment_ids"],
                               d_o=u["d_o"], d_final=u["d_final"])


def _check(name, got, ref, what):
    d = np.abs(got - ref)
    mx = float(d.max()) if d.size else 0.0
    scale = float(np.abs(ref).max()) if ref.size else 0.0
    nref = np.linalg.norm(ref)
    rel = float(np.linalg.norm(got - ref) / nref) if nref > 0 else float(np.linalg.norm(got - ref))
    assert np.all(np.isfinite(got)), f"{what} {name}: non-finite values"
    assert mx <= TOL_MAXABS_REL * scale + 1e-6 and rel <= TOL_RELL2, \
        f"{what} {name}: max-abs {mx:.3e} (ref max {scale:.3e}), rel-L2 {rel:.3e}"
    return mx / max(scale, 1e-30), rel


CASES = {
    "one_chunk": (dict(B=1, T=64, H=1, K=128, V=128, init_state_std=0.1), {}),
    "two_chunks": (dict(B=1, T=128, H=2, K=128, V=128, init_state_std=0.1), {}),
    "ragged_t200": (dict(B=1, T=200, H=2, K=128, V=128, init_state_std=0.1), {}),
    "two_rows_ragged": (dict(B=2, T=130, H=3, K=128, V=128, init_state_std=0.1), {}),
    "short_row_t9": (dict(B=3, T=9, H=1, K=128, V=128, init_state_std=0.1), {}),
    "t1000_h3": (dict(B=1, T=1000, H=3, K=128, V=128, init_state_std=0.1), {}),
    "no_state_no_dfinal": (dict(B=1, T=300, H=2, K=128, V=128),
                           dict(no_s0=True, no_dfinal=True)),
    "gate_lower_bound": (dict(B=1, T=256, H=2, K=128, V=128, init_state_std=0.1),
                         dict(g_fill=-5.0)),
    "gate_zero": (dict(B=1, T=256, H=2, K=128, V=128, init_state_std=0.1), dict(g_fill=0.0)),
    # B*H picks the chain's and the saving recurrence's value tile (152 SMs):
    # up to 38 units 32 columns, up to 76 64 columns, above that 128
    "bh40_tile64": (dict(B=2, T=130, H=20, K=128, V=128, init_state_std=0.1), {}),
    "bh80_tile128": (dict(B=2, T=70, H=40, K=128, V=128, init_state_std=0.1), {}),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_tc_backward_matches_oracle(case):
    shape, opts = CASES[case]
    w = ki.custom_workload(name=case, **shape)
    x, u = _inputs(w, seed=3, **opts)
    got = [t.cpu().numpy() for t in _gpu(x, u)]
    ref = _oracle(x, u)
    for name, a, b in zip(NAMES, got, ref):
        _check(name, a, b, case)


def test_tc_backward_full_size_sampled_heads():
    """The full B1 H32 T8192 workload through the tensor-core path; the
    oracle checks two heads."""
    w = ki.WORKLOADS["fixed_bf16_h32_t8192"]
    x, u = _inputs(w, seed=0)
    got = _gpu(x, u)
    hs = [0, 31]
    got = [g[:, :, hs].cpu().numpy() if i < 5 else g[:, hs].cpu().numpy()
           for i, g in enumerate(got)]
    ref = _oracle(x, u, heads=hs)
    for name, a, b in zip(NAMES, got, ref):
        _check(name, a, b, "B1 H32 T8192")


def test_auto_backward_is_the_tc_path_and_deterministic():
    """AUTO takes the tensor-core path for this shape: its results equal the
    explicit TC call bit for bit, and a second call with the same workspace
    repeats them (no atomics, no state kept between calls)."""
    import gated_delta_rule_21_gb300 as kda
    w = ki.custom_workload(B=1, T=320, H=2, K=128, V=128, init_state_std=0.1, name="det")
    x, u = _inputs(w, seed=9)
    ws = torch.zeros(kda.bwd_workspace_size(1, 320, 2, 128, 128), dtype=torch.uint8,
                     device="cuda")
    a = _gpu(x, u, impl="auto", workspace=ws)
    b = _gpu(x, u, impl="tc", workspace=ws)
    c = _gpu(x, u, impl="tc", workspace=ws)
    for s, t, r in zip(a, b, c):
        assert torch.equal(s, t) and torch.equal(t, r)
    assert kda.read_device_status(ws) == 0


def test_tc_backward_without_d_initial_output():
    w = ki.custom_workload(B=1, T=192, H=2, K=128, V=128, init_state_std=0.1, name="nodi")
    x, u = _inputs(w, seed=4)
    got = _gpu(x, u, want_d_initial=False)
    assert got[5] is None
    ref = _oracle(x, u)
    for name, a, b in zip(NAMES[:5], got[:5], ref[:5]):
        _check(name, a.cpu().numpy(), b, "no d_initial")


def test_tc_and_simt_backward_agree():
    """The two implementations on the same call, at the tensor-core path's
    tolerance (the CUDA-core path is fp32 throughout)."""
    w = ki.custom_workload(B=2, T=260, H=2, K=128, V=128, init_state_std=0.1, name="both")
    x, u = _inputs(w, seed=12)
    tc = [t.cpu().numpy() for t in _gpu(x, u, impl="tc")]
    simt = [t.cpu().numpy() for t in _gpu(x, u, impl="simt")]
    for name, a, b in zip(NAMES, tc, simt):
        _check(name, a, b, "tc vs simt")


PACKED = {
    "packed_pads": dict(B=2, T=300, H=2, K=128, V=128, init_state_std=0.1,
                        segments=[[("pad", 3), 100, 1, 1, ("pad", 5), 120, 70],
                                  [64, 64, ("pad", 2), 170]]),
    "padding_rows_between": dict(B=4, T=96, H=2, K=128, V=128, init_state_std=0.1,
                                 segments=[[("pad", 96)], [40, ("pad", 6), 50],
                                           [("pad", 96)], [96]]),
    "short_runs": dict(B=1, T=40, H=2, K=128, V=128, init_state_std=0.1,
                       segments=[1, 1, 3, ("pad", 1), 7, 1, 2, 24]),
    "runs_across_chunks": dict(B=1, T=400, H=3, K=128, V=128,
                               segments=[65, 63, 1, 130, ("pad", 13), 128]),
}


@pytest.mark.parametrize("case", sorted(PACKED))
def test_tc_backward_packed_matches_oracle(case):
    """Packed rows (segment ids): every run from a reset state, only the
    row's first run sees the initial state and only its last run d_final;
    padding tokens get zero gradients."""
    import gated_delta_rule_21_gb300 as kda
    w = ki.custom_workload(name=case, **PACKED[case])
    x, u = _inputs(w, seed=5)
    # room for every run (rows with more runs than ceil(T/64) need more than
    # the default size)
    runs = int(max(len(torch.unique(r[r > 0])) for r in x["segment_ids"]))
    ws = torch.zeros(kda.bwd_workspace_size_packed(w.B, w.T, w.H, w.K, w.V, max(runs, 1)),
                     dtype=torch.uint8, device="cuda")
    got = [t.cpu().numpy() for t in _gpu(x, u, workspace=ws)]
    assert kda.read_device_status(ws) == 0
    ref = _oracle(x, u)
    for name, a, b in zip(NAMES, got, ref):
        _check(name, a, b, case)
    pad = (x["segment_ids"] == 0).numpy()
    for name, a in zip(NAMES[:5], got[:5]):
        assert np.all(a[pad] == 0), f"{case} {name} not zero on padding"


def test_tc_backward_packed_full_size_sampled_heads():
    """The packed B1 H32 T8192 workload (25 runs) through the tensor-core
    path; the oracle checks two heads."""
    w = ki.WORKLOADS["packed_bf16_h32_t8192_25seg"]
    x, u = _inputs(w, seed=0)
    got = _gpu(x, u)
    hs = [0, 31]
    got = [g[:, :, hs].cpu().numpy() if i < 5 else g[:, hs].cpu().numpy()
           for i, g in enumerate(got)]
    ref = _oracle(x, u, heads=hs)
    for name, a, b in zip(NAMES, got, ref):
        _check(name, a, b, "packed B1 H32 T8192")


def test_tc_backward_packed_overflow_is_reported():
    """A workspace sized for one run per row, inputs with four: the kernels
    compute nothing and the status word says KDA_DEVICE_WORKSPACE (the
    status read returns KDA_ERR_WORKSPACE); nothing faults."""
    import gated_delta_rule_21_gb300 as kda
    w = ki.custom_workload(B=1, T=128, H=2, K=128, V=128, init_state_std=0.1,
                           segments=[32, 32, 32, 32], name="overflow")
    x, u = _inputs(w, seed=2)
    ws = torch.zeros(kda.bwd_workspace_size_packed(1, 128, 2, 128, 128, 1), dtype=torch.uint8,
                     device="cuda")
    _gpu(x, u, workspace=ws)
    assert kda.read_device_status(ws) == 4
    ws2 = torch.zeros(kda.bwd_workspace_size_packed(1, 128, 2, 128, 128, 4), dtype=torch.uint8,
                      device="cuda")
    got = [t.cpu().numpy() for t in _gpu(x, u, workspace=ws2)]
    assert kda.read_device_status(ws2) == 0
    ref = _oracle(x, u)
    for name, a, b in zip(NAMES, got, ref):
        _check(name, a, b, "four runs, room for four")


TRAIN = {
    "fixed_t300": dict(B=2, T=300, H=2, K=128, V=128, init_state_std=0.1),
    "fixed_bh40_tile64": dict(B=2, T=130, H=20, K=128, V=128, init_state_std=0.1),
    "packed": dict(B=2, T=300, H=2, K=128, V=128, init_state_std=0.1,
                   segments=[[("pad", 3), 100, 1, 1, ("pad", 5), 120, 70],
                             [64, 64, ("pad", 2), 170]]),
}


@pytest.mark.parametrize("case", sorted(TRAIN))
def test_training_step_pair_equals_separate_calls(case):
    """kda_chunk_fwd_save gives chunk_fwd's split-path o and final state bit
    for bit, and kda_chunk_bwd_from_saved on its workspace gives the
    tensor-core chunk_bwd's gradients bit for bit (the same kernels on the
    same items and saves); run twice on one workspace, the backward repeats."""
    import gated_delta_rule_21_gb300 as kda
    w = ki.custom_workload(name=case, **TRAIN[case])
    x, u = _inputs(w, seed=21)
    dev = lambda t: None if t is None else to_dev(t)
    d = {n: dev(x[n]) for n in ("q", "k", "v", "g", "beta", "initial_state", "segment_ids")}
    o_s, fs_s, ws = kda.chunk_fwd_save(d["q"], d["k"], d["v"], d["g"], d["beta"],
                                       scale=x["scale"], initial_state=d["initial_state"],
                                       segment_ids=d["segment_ids"])
    o, fs = kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=x["scale"],
                          initial_state=d["initial_state"], segment_ids=d["segment_ids"],
                          output_final_state=True, impl="split")
    torch.cuda.synchronize()
    assert torch.equal(o_s, o) and torch.equal(fs_s, fs)
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"], dev(u["d_o"]))
    kw = dict(scale=x["scale"], initial_state=d["initial_state"],
              segment_ids=d["segment_ids"], d_final=dev(u["d_final"]))
    a = kda.chunk_bwd_from_saved(*args, ws, **kw)
    b = kda.chunk_bwd_from_saved(*args, ws, **kw)
    c = kda.chunk_bwd(*args, impl="tc", **kw)
    torch.cuda.synchronize()
    assert kda.read_device_status(ws) == 0
    for s_, t_, r_ in zip(a, b, c):
        assert torch.equal(s_, t_) and torch.equal(s_, r_)
    ref = _oracle(x, u)
    for name, got, r in zip(NAMES, a, ref):
        _check(name, got.cpu().numpy(), r, f"{case} from saved")
