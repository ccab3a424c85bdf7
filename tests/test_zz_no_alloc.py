"""kda_chunk_fwd_noalloc: the forward entry point for callers that cannot
allocate device memory (for instance a plugin that is handed only the
tensors it works on, or code on a path where allocating is not allowed).

It keeps its scratch in a fixed device array inside libkda instead of a
caller-provided workspace.  This test calls it through the C ABI and checks
its output against the ordinary entry point (kda_chunk_fwd with a workspace)
within the bf16 tolerances the parity tests use, on two calls in a row with
different packed inputs, so the second call also shows that the shared
array carries nothing over from the first.  The file is named so that pytest
collects it last.
"""
import ctypes

import pytest
import torch

import kda_inputs as ki
from kda_testlib import assert_parity, to_dev

pytestmark = pytest.mark.gpu


def noalloc_fn():
    import gated_delta_rule_21_gb300 as kda
    from gated_delta_rule_21_gb300 import build
    build.build()
    L = kda.lib()
    vp = ctypes.c_void_p
    f = L.kda_chunk_fwd_noalloc
    f.argtypes = [ctypes.POINTER(kda.kda_shape), vp, vp, vp, vp, vp, ctypes.c_float,
                  ctypes.c_int, vp, vp, vp, vp, vp]
    f.restype = ctypes.c_int
    return kda, f


def call_noalloc(kda, f, d, w, scale):
    o = torch.empty(w.B, w.T, w.H, w.V, dtype=d["q"].dtype, device="cuda")
    fs = torch.empty(w.B, w.H, w.K, w.V, dtype=torch.float32, device="cuda")
    s = kda.make_shape(w.B, w.T, w.H, w.K, w.V, d["q"].dtype)
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    st = f(ctypes.byref(s), p(d["q"]), p(d["k"]), p(d["v"]), p(d["g"]), p(d["beta"]),
           scale, 64, p(d["initial_state"]), p(d["segment_ids"]), p(o), p(fs),
           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, kda.status_string(st)
    return o, fs


def test_noalloc_matches_workspace_entry_point_two_calls():
    kda, f = noalloc_fn()
    cases = [
        ki.custom_workload(1, 1024, 8, 128, 128, init_state_std=0.1,
                           segments=[197, 301, 259, 267], name="packed4"),
        ki.custom_workload(2, 700, 4, 128, 128, init_state_std=0.1,
                           segments=[[("pad", 3), 64, 1, 200, 150, ("pad", 7), 275],
                                     [699]], name="packed_mixed"),
    ]
    for w in cases:                 # two noalloc calls in a row
        x = ki.make_inputs(w, seed=21)
        d = {n: to_dev(x[n]) for n in ("q", "k", "v", "g", "beta", "initial_state",
                                        "segment_ids")}
        o_n, fs_n = call_noalloc(kda, f, d, w, x["scale"])
        o_w, fs_w = kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=x["scale"],
                                  initial_state=d["initial_state"],
                                  segment_ids=d["segment_ids"], output_final_state=True)
        torch.cuda.synchronize()
        assert_parity(o_n, o_w.double().cpu().numpy(), True, f"{w.name} o")
        assert_parity(fs_n, fs_w.double().cpu().numpy(), True, f"{w.name} final_state")


def test_noalloc_rejects_shapes_beyond_its_scratch():
    kda, f = noalloc_fn()
    fake = ctypes.c_void_p(0x10000)   # never dereferenced: rejected on the host
    s = kda.make_shape(1, 200000, 1, 32, 32, torch.bfloat16)
    st = f(ctypes.byref(s), fake, fake, fake, fake, fake, 0.1, 64, None, fake, fake, None, None)
    assert st == 4   # KDA_ERR_WORKSPACE: the run list would not fit
