"""The host-buffer entry point (copies in, forward, copies out, pipelined
over token ranges without segment ids and over head groups with them):
argument checks on the host, and on the GPU bitwise equality with the device
entry point on the same inputs (each range's forward enters with the exact
fp32 state the previous range left; each head group's forward runs the same
kernels on the same per-head data) plus oracle parity."""
import ctypes

import pytest
import torch

import kda_inputs as ki
from kda_testlib import assert_parity, run_gpu, run_oracle


def test_host_buffer_size_and_argument_checks():
    import gated_delta_rule_21_gb300 as kda
    L = kda.lib()
    n = kda.host_buffer_size(1, 8192, 32, 128, 128)
    inputs = 8192 * 32 * (3 * 128 * 2 + 128 * 4 + 4) + 8192 * 32 * 128 * 2
    assert n > inputs
    assert kda.host_buffer_size(1, 100, 2, 128, 128, has_segment_ids=True) > \
        kda.host_buffer_size(1, 100, 2, 128, 128)
    assert kda.host_buffer_size(1, 0, 2, 128, 128) == 0
    s = kda.make_shape(1, 64, 2, 128, 128, torch.bfloat16)
    nb = kda.host_buffer_size(1, 64, 2, 128, 128)
    x = ctypes.c_void_p(16)
    args = [ctypes.byref(s), x, x, x, x, x, 0.1, 64, None, None, x, None, x, nb, None]
    bad = list(args); bad[1] = None
    assert L.kda_chunk_fwd_host(*bad) == 1            # NULL q
    bad = list(args); bad[7] = 32
    assert L.kda_chunk_fwd_host(*bad) == 2            # chunk size
    bad = list(args); bad[13] = nb - 1
    assert L.kda_chunk_fwd_host(*bad) == 4            # small device buffer
    bad = list(args); bad[12] = ctypes.c_void_p(16)
    assert L.kda_chunk_fwd_host(*bad) == 3            # buffer not 256-byte aligned
    bad = list(args); bad[6] = float("nan")
    assert L.kda_chunk_fwd_host(*bad) == 1            # NaN scale


def _pinned(x):
    return None if x is None else x.contiguous().pin_memory()


# Several token ranges (512 tokens each, a ragged last one), B > 1, with and
# without an initial state, and the fp32 paths.
HOST_CASES = {
    "b2_bf16_h4_t1600_s0": dict(B=2, T=1600, H=4, K=128, V=128, dtype="bf16", init_state_std=0.1),
    "b3_bf16_h2_t1100": dict(B=3, T=1100, H=2, K=128, V=128, dtype="bf16"),
    "b2_fp32_h2_t1030_d64_s0": dict(B=2, T=1030, H=2, K=64, V=64, dtype="f32", init_state_std=0.1),
    "b1_fp32_h1_t8200_d32_s0": dict(B=1, T=8200, H=1, K=32, V=32, dtype="f32", init_state_std=0.1),
}


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["fixed_bf16_h8_t1024", "packed_bf16_h8_t1024_4seg",
                                  "tiny_fp32_h2_t128_d32"] + sorted(HOST_CASES))
def test_host_matches_device_path(name):
    import gated_delta_rule_21_gb300 as kda
    w = ki.WORKLOADS[name] if name in ki.WORKLOADS else ki.custom_workload(**HOST_CASES[name])
    x = ki.make_inputs(w, seed=7)
    o_d, fs_d = run_gpu(x)
    h = {n: _pinned(x[n]) for n in ("q", "k", "v", "g", "beta", "initial_state", "segment_ids")}
    buf = torch.zeros(kda.host_buffer_size(w.B, w.T, w.H, w.K, w.V, x["q"].dtype,
                                           x["segment_ids"] is not None),
                      dtype=torch.uint8, device="cuda")
    for _ in range(2):  # the device buffer is reusable
        o_h, fs_h = kda.chunk_fwd_host(h["q"], h["k"], h["v"], h["g"], h["beta"], scale=x["scale"],
                                       initial_state=h["initial_state"],
                                       segment_ids=h["segment_ids"], output_final_state=True,
                                       device_buffer=buf)
        torch.cuda.synchronize()
        assert torch.equal(o_h, o_d.cpu()) and torch.equal(fs_h, fs_d.cpu())
    o_ref, fs_ref = run_oracle(x)
    bf16 = w.dtype == "bf16"
    assert_parity(o_h, o_ref, bf16, f"{name} host o")
    assert_parity(fs_h, fs_ref, bf16, f"{name} host final_state")
