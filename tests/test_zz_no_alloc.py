"""kda_chunk_fwd_noalloc: the forward entry point for callers that cannot
allocate device memory (for instance a plugin that is handed only the
tensors it works on, or code on a path where allocating is not allowed).

It keeps its scratch in a fixed device array inside libkda instead of a
caller-provided workspace.  These tests call it through the C ABI and check
its output against the fp64 oracle at the parity tests' bf16 tolerances, and
against the ordinary entry point (kda_chunk_fwd with a workspace), on calls
in a row with different inputs, so that later calls also show that the
shared array carries nothing over.  The cases cover both kernels the fixed
array can hold: the fused tensor-core kernel (shapes whose per-chunk
operands do not fit the array) and the split kernels with their operands
inside the array (small B*ceil(T/64)*H), with and without segment ids.
After every call, kda_chunk_fwd_noalloc_status must report a clean status
word.  The file is named so that pytest collects it last.
"""
import ctypes

import pytest
import torch

import kda_inputs as ki
from kda_testlib import assert_parity, run_oracle, to_dev

pytestmark = pytest.mark.gpu


def noalloc_lib():
    import gated_delta_rule_21_gb300 as kda
    from gated_delta_rule_21_gb300 import build
    build.build()
    return kda, kda.lib()


def call_noalloc(kda, L, d, w, scale):
    o = torch.empty(w.B, w.T, w.H, w.V, dtype=d["q"].dtype, device="cuda")
    fs = torch.empty(w.B, w.H, w.K, w.V, dtype=torch.float32, device="cuda")
    s = kda.make_shape(w.B, w.T, w.H, w.K, w.V, d["q"].dtype)
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = L.kda_chunk_fwd_noalloc(ctypes.byref(s), p(d["q"]), p(d["k"]), p(d["v"]), p(d["g"]),
                                 p(d["beta"]), scale, 64, p(d["initial_state"]),
                                 p(d["segment_ids"]), p(o), p(fs), stream)
    assert st == 0, kda.status_string(st)
    bits = ctypes.c_uint32(0xFFFF)
    st = L.kda_chunk_fwd_noalloc_status(stream, ctypes.byref(bits))
    assert st == 0 and bits.value == 0, (kda.status_string(st), bits.value)
    return o, fs


CASES = [
    # fused kernel: the per-chunk operands of these shapes do not fit 1 MiB
    ki.custom_workload(1, 1024, 8, 128, 128, init_state_std=0.1,
                       segments=[197, 301, 259, 267], name="packed4"),
    ki.custom_workload(2, 700, 4, 128, 128, init_state_std=0.1,
                       segments=[[("pad", 3), 64, 1, 200, 150, ("pad", 7), 275],
                                 [699]], name="packed_mixed"),
    ki.custom_workload(1, 1024, 4, 128, 128, init_state_std=0.1, name="fixed_h4"),
    # split kernels with their operands inside the array
    ki.custom_workload(1, 640, 1, 128, 128, init_state_std=0.1,
                       segments=[197, 301, 142], name="packed_h1_split"),
    ki.custom_workload(1, 640, 1, 128, 128, init_state_std=0.1, name="fixed_h1_split"),
]


def test_noalloc_matches_oracle_and_workspace_entry_point_calls_in_a_row():
    kda, L = noalloc_lib()
    for i, w in enumerate(CASES):
        x = ki.make_inputs(w, seed=21 + i)
        d = {n: to_dev(x[n]) for n in ("q", "k", "v", "g", "beta", "initial_state",
                                        "segment_ids")}
        o_ref, fs_ref = run_oracle(x)
        for rep in range(2):        # the same inputs twice more in a row
            o_n, fs_n = call_noalloc(kda, L, d, w, x["scale"])
            torch.cuda.synchronize()
            assert_parity(o_n, o_ref, True, f"{w.name} call {rep} o vs oracle")
            assert_parity(fs_n, fs_ref, True, f"{w.name} call {rep} final_state vs oracle")
        o_w, fs_w = kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=x["scale"],
                                  initial_state=d["initial_state"],
                                  segment_ids=d["segment_ids"], output_final_state=True)
        torch.cuda.synchronize()
        assert_parity(o_n, o_w.double().cpu().numpy(), True, f"{w.name} o vs workspace call")
        assert_parity(fs_n, fs_w.double().cpu().numpy(), True,
                      f"{w.name} final_state vs workspace call")


def test_noalloc_rejects_shapes_beyond_its_scratch():
    kda, L = noalloc_lib()
    fake = ctypes.c_void_p(0x10000)   # never dereferenced: rejected on the host
    s = kda.make_shape(1, 200000, 1, 32, 32, torch.bfloat16)
    st = L.kda_chunk_fwd_noalloc(ctypes.byref(s), fake, fake, fake, fake, fake, 0.1, 64, None,
                                 fake, fake, None, None)
    assert st == 4   # KDA_ERR_WORKSPACE: the run list would not fit
