"""The chunk-parallel state scan (kda_chunk_fwd_scan): rows without segment
ids are cut into segments whose affine state maps S -> M S + B are built in
parallel, chained in fp32, and then every segment is finished from its
entering state.  The GPU tests compare it with the fp64 oracle at the bf16
tolerances of the parity tests, for several segment counts (including one
chunk per segment), a ragged last chunk, two rows and an initial state; the
CPU tests cover the workspace query and the argument checks."""
import ctypes

import pytest
import torch

import kda_inputs as ki
from kda_testlib import assert_parity, run_oracle, to_dev

FAKE = 0x10000  # never dereferenced: rejected on the host


@pytest.fixture(scope="module")
def kda():
    import gated_delta_rule_21_gb300 as kda
    from gated_delta_rule_21_gb300 import build
    build.build()
    kda.lib()
    return kda


def test_scan_workspace_query(kda):
    split = kda.workspace_size(1, 8192, 32, 128, 128, impl="split")
    n2 = kda.scan_workspace_size(1, 8192, 32, 128, 128, n_segments=2)
    n4 = kda.scan_workspace_size(1, 8192, 32, 128, 128, n_segments=4)
    # the items, then (P - 1) maps of K x (V + K) and P entering states of
    # K x V per (row, head), fp32
    per_bh = 128 * 256 * 4
    assert n2 == (split + 255) // 256 * 256 + 1 * 32 * per_bh + 2 * 32 * 128 * 128 * 4
    assert n4 > n2
    assert kda.scan_workspace_size(1, 8192, 32, 64, 64) == 0                 # K, V
    assert kda.scan_workspace_size(1, 8192, 32, 128, 128, torch.float32) == 0
    assert kda.scan_workspace_size(1, 64, 32, 128, 128) == 0                 # one chunk
    assert kda.scan_workspace_size(1, 8192, 32, 128, 128, n_segments=1) == 0
    # segment counts: requested ones capped at the chunks and rounded so
    # every segment holds a chunk; 0 fills the SMs (at least 2)
    assert kda.scan_segments(1, 1024, 2, 128, 128, n_segments=16) == 16
    assert kda.scan_segments(1, 1024, 2, 128, 128, n_segments=40) == 16
    assert kda.scan_segments(1, 320, 2, 128, 128, n_segments=4) == 3   # 5 chunks: 2+2+1
    assert kda.scan_segments(1, 8192, 32, 128, 128) >= 2
    assert kda.scan_segments(1, 8192, 32, 64, 64) == 0


def test_scan_rejects_bad_arguments(kda):
    L = kda.lib()
    vp = ctypes.c_void_p

    def call(shape=(1, 1024, 2, 128, 128, 1), q=FAKE, o=FAKE, nseg=2, chunk=64, ws=FAKE,
             nbytes=1 << 30, s0=None):
        s = kda.kda_shape(*shape)
        return L.kda_chunk_fwd_scan(ctypes.byref(s), vp(q), vp(FAKE), vp(FAKE), vp(FAKE),
                                    vp(FAKE), 0.1, chunk, vp(s0), vp(o), None, nseg, vp(ws),
                                    nbytes, None)
    assert call(q=None) == 1
    assert call(o=None) == 1
    assert call(nseg=1) == 1
    assert call(nseg=-3) == 1
    assert call(chunk=32) == 2
    assert call(shape=(1, 1024, 2, 64, 64, 1)) == 2
    assert call(q=FAKE + 2) == 3
    assert call(s0=FAKE + 4) == 3
    assert call(nbytes=1024) == 4
    assert call(ws=None) == 4
    assert call(ws=FAKE + 16) == 3


CASES = [
    (ki.custom_workload(1, 1024, 2, 128, 128, name="h2_t1024"), 2),
    (ki.custom_workload(1, 1024, 2, 128, 128, name="h2_t1024"), 4),
    (ki.custom_workload(1, 1024, 2, 128, 128, init_state_std=0.1, name="h2_t1024_s0"), 16),
    (ki.custom_workload(1, 1000, 3, 128, 128, init_state_std=0.1, name="h3_t1000_ragged"), 3),
    (ki.custom_workload(2, 640, 3, 128, 128, init_state_std=0.1, name="b2_h3_t640"), 0),
]


@pytest.mark.gpu
@pytest.mark.parametrize("w,nseg", CASES, ids=[f"{w.name}-P{p}" for w, p in CASES])
def test_scan_matches_oracle(kda, w, nseg):
    x = ki.make_inputs(w, seed=31)
    d = {n: to_dev(x[n]) for n in ("q", "k", "v", "g", "beta", "initial_state")}
    ws = torch.zeros(kda.scan_workspace_size(w.B, w.T, w.H, w.K, w.V, n_segments=nseg),
                     dtype=torch.uint8, device="cuda")
    o, fs = kda.chunk_fwd_scan(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=x["scale"],
                               initial_state=d["initial_state"], output_final_state=True,
                               n_segments=nseg, workspace=ws)
    torch.cuda.synchronize()
    assert kda.read_device_status(ws) == 0
    o_ref, fs_ref = run_oracle(x)
    assert_parity(o, o_ref, True, f"{w.name} P={nseg} o")
    assert_parity(fs, fs_ref, True, f"{w.name} P={nseg} final_state")


@pytest.mark.gpu
def test_scan_gate_edges_g_minus5():
    """Every gate at the contract's lower bound: the maps M are products of
    strongly decaying factors, the combine must still hand over the right
    states."""
    import gated_delta_rule_21_gb300 as kda
    w = ki.custom_workload(1, 768, 2, 128, 128, init_state_std=0.1, name="gmin")
    x = ki.make_inputs(w, seed=7)
    x["g"] = torch.full_like(x["g"], -5.0)
    d = {n: to_dev(x[n]) for n in ("q", "k", "v", "g", "beta", "initial_state")}
    o, fs = kda.chunk_fwd_scan(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=x["scale"],
                               initial_state=d["initial_state"], output_final_state=True,
                               n_segments=4)
    torch.cuda.synchronize()
    o_ref, fs_ref = run_oracle(x)
    assert_parity(o, o_ref, True, "g=-5 o")
    assert_parity(fs, fs_ref, True, "g=-5 final_state")


@pytest.mark.gpu
def test_scan_in_benchmark_configuration():
    """The B1 H32 T8192 shape with a random initial state, as a 2-segment
    scan (the count the automatic choice gives there), against the oracle."""
    import gated_delta_rule_21_gb300 as kda
    w = ki.WORKLOADS["fixed_bf16_h32_t8192"]
    x = ki.make_inputs(w, seed=0)
    d = {n: to_dev(x[n]) for n in ("q", "k", "v", "g", "beta", "initial_state")}
    o, fs = kda.chunk_fwd_scan(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=x["scale"],
                               initial_state=d["initial_state"], output_final_state=True,
                               n_segments=0)
    torch.cuda.synchronize()
    o_ref, fs_ref = run_oracle(x)
    assert_parity(o, o_ref, True, "B1 H32 T8192 scan o")
    assert_parity(fs, fs_ref, True, "B1 H32 T8192 scan final_state")


@pytest.mark.gpu
def test_auto_workspace_covers_the_scan_on_long_few_head_rows(kda):
    """AUTO's default workspace is the scan's on long rows with few heads
    (there it runs the scan), the split path's elsewhere.  The choice counts
    the SMs of the current device, so this needs one."""
    long_ = kda.workspace_size(1, 32768, 8, 128, 128)
    assert long_ == kda.scan_workspace_size(1, 32768, 8, 128, 128) > \
        kda.workspace_size(1, 32768, 8, 128, 128, impl="split")
    assert kda.workspace_size(1, 8192, 32, 128, 128) == \
        kda.workspace_size(1, 8192, 32, 128, 128, impl="split")
    assert kda.workspace_size(1, 1024, 8, 128, 128) == \
        kda.workspace_size(1, 1024, 8, 128, 128, impl="split")       # short rows
    # 152 SMs: 9 segments of 15 chunks (8 or more per segment suffice with 8
    # or more segments) against 4 segments of 16 (32 needed with fewer)
    assert kda.workspace_size(1, 8192, 8, 128, 128) == \
        kda.scan_workspace_size(1, 8192, 8, 128, 128)
    assert kda.workspace_size(1, 4096, 16, 128, 128) == \
        kda.workspace_size(1, 4096, 16, 128, 128, impl="split")


@pytest.mark.gpu
def test_auto_on_long_few_head_rows_matches_oracle():
    """kda_chunk_fwd (AUTO) on B1 H8 T32768, which it runs as the scan."""
    import gated_delta_rule_21_gb300 as kda
    w = ki.WORKLOADS["fixed_bf16_h8_t32768"]
    x = ki.make_inputs(w, seed=4)
    d = {n: to_dev(x[n]) for n in ("q", "k", "v", "g", "beta", "initial_state")}
    o, fs = kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=x["scale"],
                          initial_state=d["initial_state"], output_final_state=True)
    torch.cuda.synchronize()
    o_ref, fs_ref = run_oracle(x)
    assert_parity(o, o_ref, True, "B1 H8 T32768 auto o")
    assert_parity(fs, fs_ref, True, "B1 H8 T32768 auto final_state")
