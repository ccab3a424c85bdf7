"""GPU parity of the short-conv prologue (kda_short_conv_silu) against the
fp64 oracle, alone and composed with the chunked forward."""
import numpy as np
import pytest
import torch

import kda_inputs as ki
import oracle
from kda_testlib import assert_parity, to_dev

pytestmark = pytest.mark.gpu


def oracle_prologue(x, w, seg, l2, H, K, V, store_bf16):
    """Conv + SiLU (+ L2 on q, k) in fp64; optionally rounded to the bf16
    storage the GPU prologue writes."""
    B, T = x["q"].shape[:2]
    outs = []
    for i, name in enumerate(("q", "k", "v")):
        D = K if i < 2 else V
        xi = oracle._f64(x[name]).reshape(B, T, H * D)
        wi = w[i].double().numpy()
        y = oracle.short_conv_silu(xi, wi, seg)
        if l2 and i < 2:
            y = oracle.l2norm(y, D, eps=1e-6)
        y = y.reshape(B, T, H, D)
        outs.append(oracle.round_bf16(y) if store_bf16 else y)
    return outs


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("l2", [True, False])
@pytest.mark.parametrize("shape", [(1, 100, 2, 128, 128), (2, 70, 3, 64, 64), (1, 45, 4, 32, 32)])
def test_conv_matches_oracle(dtype, l2, shape):
    import gated_delta_rule_21_gb300 as kda
    B, T, H, K, V = shape
    w_ = ki.custom_workload(B, T, H, K, V, dtype=dtype, prologue=True,
                            segments=[[7, 1, ("pad", 2), T - 12, ("pad", 2)]] * B)
    x = ki.make_inputs(w_, seed=9)
    seg = x["segment_ids"]
    q, k, v = kda.short_conv_silu(to_dev(x["q"]), to_dev(x["k"]), to_dev(x["v"]),
                                  to_dev(x["conv_w"]), segment_ids=to_dev(seg), l2norm_qk=l2)
    refs = oracle_prologue(x, x["conv_w"], seg.numpy(), l2, H, K, V, store_bf16=False)
    for got, ref, name in zip((q, k, v), refs, "qkv"):
        g = got.double().cpu().numpy()
        if dtype == "bf16":   # within one bf16 rounding of the exact value
            tol = 1.02 * 2.0 ** -8 * np.abs(ref) + 1e-6
        else:
            tol = 1e-5 * np.abs(ref) + 1e-6
        bad = np.abs(g - ref) > tol
        assert not bad.any(), f"{name}: {bad.sum()} elements off, max {np.abs(g - ref).max():.3e}"
    pad = torch.from_numpy((seg == 0).numpy())
    assert torch.all(q.cpu()[pad] == 0) and torch.all(v.cpu()[pad] == 0)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_conv_short_runs_several_channel_blocks(dtype):
    """Runs of 1-5 tokens, padding between and at the start, run starts on
    and next to the 24-token tile edges, 2048 channels per tensor (two
    1024-channel blocks) and a ragged last tile."""
    import gated_delta_rule_21_gb300 as kda
    B, T, H, K, V = 2, 203, 16, 128, 128
    rows = [[("pad", 1), 1, 2, 3, ("pad", 2), 1, 5, 9, 24, 1, 23, ("pad", 3), 2, 48, 1, 1, 30, 46],
            [22, 2, 1, 24, 25, ("pad", 1), 1, 3, 60, 4, 4, 50]]
    w_ = ki.custom_workload(B, T, H, K, V, dtype=dtype, prologue=True, segments=rows)
    x = ki.make_inputs(w_, seed=11)
    seg = x["segment_ids"]
    q, k, v = kda.short_conv_silu(to_dev(x["q"]), to_dev(x["k"]), to_dev(x["v"]),
                                  to_dev(x["conv_w"]), segment_ids=to_dev(seg), l2norm_qk=True)
    refs = oracle_prologue(x, x["conv_w"], seg.numpy(), True, H, K, V, store_bf16=False)
    for got, ref, name in zip((q, k, v), refs, "qkv"):
        g = got.double().cpu().numpy()
        tol = (1.02 * 2.0 ** -8 if dtype == "bf16" else 1e-5) * np.abs(ref) + 1e-6
        bad = np.abs(g - ref) > tol
        assert not bad.any(), f"{name}: {bad.sum()} elements off, max {np.abs(g - ref).max():.3e}"
    pad = torch.from_numpy((seg == 0).numpy())
    assert torch.all(k.cpu()[pad] == 0) and torch.all(v.cpu()[pad] == 0)


def test_prologue_then_chunk_fwd_packed_n25():
    """Prologue (conv + SiLU + L2 on q, k) followed by the chunked forward
    on the packed B=1 H=32 T=8192 K=V=128 shape with 25 segments, against
    the oracle's conv -> L2 -> bf16 storage -> recurrence."""
    import gated_delta_rule_21_gb300 as kda
    w = ki.WORKLOADS["packed_bf16_h32_t8192_25seg_conv"]
    x = ki.make_inputs(w, seed=0)
    seg = to_dev(x["segment_ids"])
    q, k, v = kda.short_conv_silu(to_dev(x["q"]), to_dev(x["k"]), to_dev(x["v"]),
                                  to_dev(x["conv_w"]), segment_ids=seg, l2norm_qk=True)
    o, fs = kda.chunk_fwd(q, k, v, to_dev(x["g"]), to_dev(x["beta"]), scale=x["scale"],
                          segment_ids=seg, output_final_state=True)
    torch.cuda.synchronize()
    qr, kr, vr = oracle_prologue(x, x["conv_w"], x["segment_ids"].numpy(), True,
                                 w.H, w.K, w.V, store_bf16=True)
    o_ref, fs_ref = oracle.kda_forward(qr, kr, vr, x["g"], x["beta"], x["scale"],
                                       segment_ids=x["segment_ids"])
    assert_parity(o, o_ref, True, "o")
    assert_parity(fs, fs_ref, True, "final_state")
