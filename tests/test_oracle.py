"""Pins of the fp64 oracle against what the pages and the mathematics fix.

The recurrence is page "feat(kda): integrate KDA attention with tokamax backend
and CP support", section "Delta Rule formulation"; the properties "zero-gate
accumulates" and "large-negative-gate decays" are its section "Test Coverage"
(category "Properties").  Each test names the mistake it would catch.
"""
import numpy as np
import pytest
import torch

import kda_inputs as ki
import oracle
from brute import matrix_form, transition_form

RNG = np.random.default_rng(1234)


def rand_case(B=1, T=6, H=2, K=3, V=4, seg=None, S0=False, gmin=-5.0, rng=RNG):
    q = rng.standard_normal((B, T, H, K))
    k = rng.standard_normal((B, T, H, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, V))
    g = rng.uniform(gmin, 0.0, (B, T, H, K))
    beta = rng.uniform(0.0, 1.0, (B, T, H))
    s0 = rng.standard_normal((B, H, K, V)) * 0.3 if S0 else None
    return q, k, v, g, beta, s0, seg


# --- 1. zero gate: pure delta rule accumulates --------------------------------

def test_zero_gate_orthonormal_keys_accumulate_exactly():
    """g = 0, keys = distinct basis vectors, beta = 1, S0 = 0: the state after
    t tokens is sum_i e_{p(i)} v_i^T exactly and o_t = scale sum_i (q_t .
    e_{p(i)}) v_i.  Catches a wrong residual sign, a missing beta, or g acting
    on the value axis."""
    K = V = 5
    T = 5
    perm = [3, 0, 4, 1, 2]
    q = RNG.standard_normal((1, T, 1, K))
    k = np.zeros((1, T, 1, K))
    for t in range(T):
        k[0, t, 0, perm[t]] = 1.0
    v = RNG.standard_normal((1, T, 1, V))
    g = np.zeros((1, T, 1, K))
    beta = np.ones((1, T, 1))
    scale = 0.7
    o, fs = oracle.kda_forward(q, k, v, g, beta, scale)
    S = np.zeros((K, V))
    for t in range(T):
        S[perm[t]] = v[0, t, 0]
        np.testing.assert_allclose(o[0, t, 0], scale * q[0, t, 0] @ S, rtol=0, atol=1e-15)
    np.testing.assert_array_equal(fs[0, 0], S)


def test_zero_gate_orthogonal_keys_fractional_beta():
    """g = 0 and mutually orthogonal keys: k_t^T S' = 0, so the state is
    sum_i beta_i k_i v_i^T.  Catches beta applied to the residual twice or
    not at all."""
    K, V, T = 4, 3, 4
    Qm, _ = np.linalg.qr(RNG.standard_normal((K, K)))
    k = Qm.T[None, :, None, :]          # rows orthonormal
    v = RNG.standard_normal((1, T, 1, V))
    beta = RNG.uniform(0.1, 0.9, (1, T, 1))
    q = RNG.standard_normal((1, T, 1, K))
    g = np.zeros((1, T, 1, K))
    o, fs = oracle.kda_forward(q, k, v, g, beta, 1.0)
    S = sum(beta[0, i, 0] * np.outer(k[0, i, 0], v[0, i, 0]) for i in range(T))
    np.testing.assert_allclose(fs[0, 0], S, rtol=0, atol=1e-14)


# --- 2. large negative gate decays ---------------------------------------------

def test_large_negative_gate_decays_to_single_token():
    """g = -1e4: exp underflows to 0, S' = 0 and o_t = scale beta_t (q_t .
    k_t) v_t; final_state = beta_T k_T v_T^T.  Catches the decay applied after
    the residual, or o read before the write."""
    q, k, v, _, beta, s0, _ = rand_case(T=7, S0=True)
    g = np.full_like(q, -1e4)
    scale = 0.5
    o, fs = oracle.kda_forward(q, k, v, g, beta, scale, initial_state=s0)
    exp_o = scale * beta[..., None] * np.sum(q * k, -1, keepdims=True) * v
    np.testing.assert_allclose(o, exp_o, rtol=1e-13, atol=1e-15)
    T = q.shape[1]
    for h in range(q.shape[2]):
        np.testing.assert_allclose(
            fs[0, h], beta[0, T - 1, h] * np.outer(k[0, T - 1, h], v[0, T - 1, h]),
            rtol=1e-13, atol=1e-15)


def test_gate_minus_five_decays_by_e5_per_token():
    """The kernel's contract edge g = -5 on every channel: with beta = 0 the
    state only decays, S_T = e^{-5T} S0.  Catches exp(g) vs exp(-g) and a
    gate applied per value column."""
    q, k, v, _, beta, s0, _ = rand_case(T=5, S0=True)
    g = np.full_like(q, -5.0)
    o, fs = oracle.kda_forward(q, k, v, g, np.zeros_like(beta), 1.0, initial_state=s0)
    np.testing.assert_allclose(fs, s0 * np.exp(-25.0), rtol=1e-13)
    for t in range(5):
        exp_o = np.einsum("hk,hkv->hv", q[0, t], s0[0] * np.exp(-5.0 * (t + 1)))
        np.testing.assert_allclose(o[0, t], exp_o, rtol=1e-12, atol=1e-300)


def test_per_channel_gate_scales_key_rows():
    """beta = 0, one token: S1 = diag(exp g) S0, so the gate multiplies key
    rows, not value columns (K != V to catch a transpose)."""
    q, k, v, g, beta, s0, _ = rand_case(T=1, K=3, V=5, S0=True)
    _, fs = oracle.kda_forward(q, k, v, g, np.zeros_like(beta), 1.0, initial_state=s0)
    for h in range(q.shape[2]):
        np.testing.assert_allclose(fs[0, h], np.exp(g[0, 0, h])[:, None] * s0[0, h],
                                   rtol=1e-14)


# --- 3. write then read ----------------------------------------------------------

@pytest.mark.parametrize("gmin", [0.0, -5.0])
def test_write_then_read_returns_v(gmin):
    """beta = 1 and unit k: k_t^T S_t = v_t for any gate, because the update
    removes exactly the old read-out along k_t.  With q = k and scale = 1 the
    output is v.  Catches a wrong update order or a dropped beta."""
    q, k, v, g, beta, s0, _ = rand_case(T=9, K=4, V=3, S0=True, gmin=gmin)
    beta = np.ones_like(beta)
    o, _ = oracle.kda_forward(k, k, v, g, beta, 1.0, initial_state=s0)
    np.testing.assert_allclose(o, v, rtol=0, atol=1e-12)


# --- 4. T = 1 closed form ----------------------------------------------------------

def test_single_token_closed_form():
    """S1 = D S0 + beta k (v - k^T D S0)^T with D = diag(exp g), o =
    scale S1^T q, written out by hand with explicit index sums."""
    q, k, v, g, beta, s0, _ = rand_case(T=1, H=1, K=2, V=2, S0=True)
    scale = 0.9
    o, fs = oracle.kda_forward(q, k, v, g, beta, scale, initial_state=s0)
    qq, kk, vv, gg, bb, S0 = q[0, 0, 0], k[0, 0, 0], v[0, 0, 0], g[0, 0, 0], beta[0, 0, 0], s0[0, 0]
    Sp = [[S0[i][j] * np.exp(gg[i]) for j in range(2)] for i in range(2)]
    res = [vv[j] - (kk[0] * Sp[0][j] + kk[1] * Sp[1][j]) for j in range(2)]
    S1 = [[Sp[i][j] + bb * kk[i] * res[j] for j in range(2)] for i in range(2)]
    oo = [scale * (qq[0] * S1[0][j] + qq[1] * S1[1][j]) for j in range(2)]
    np.testing.assert_allclose(fs[0, 0], np.array(S1), rtol=1e-14)
    np.testing.assert_allclose(o[0, 0, 0], np.array(oo), rtol=1e-14)


def test_two_tokens_hand_expanded():
    """T = 2, K = V = 1: scalars.  s1 = b1 k1 v1 (S0 = 0); s2 = e^{g2} s1 +
    b2 k2 (v2 - k2 e^{g2} s1); o = (q1 s1, q2 s2)."""
    q = np.array([0.3, -1.1]).reshape(1, 2, 1, 1)
    k = np.array([0.8, 0.6]).reshape(1, 2, 1, 1)
    v = np.array([2.0, -0.5]).reshape(1, 2, 1, 1)
    g = np.array([-0.25, -1.5]).reshape(1, 2, 1, 1)
    b = np.array([0.4, 0.9]).reshape(1, 2, 1)
    o, fs = oracle.kda_forward(q, k, v, g, b, 1.0)
    s1 = 0.4 * 0.8 * 2.0
    s2 = np.exp(-1.5) * s1 + 0.9 * 0.6 * (-0.5 - 0.6 * np.exp(-1.5) * s1)
    np.testing.assert_allclose(o.ravel(), [0.3 * s1, -1.1 * s2], rtol=1e-15)
    np.testing.assert_allclose(fs.ravel(), [s2], rtol=1e-15)


# --- 5. packed == separate ---------------------------------------------------------

def test_packed_equals_separate_runs_bitwise():
    """A packed row equals running each segment as its own sequence, the
    first from initial_state and the others from zero (bitwise in fp64)."""
    lens = [5, 1, 7, 3]
    T = sum(lens) + 2
    seg = ki.segment_ids_from_lengths(1, T, lens).numpy()
    q, k, v, g, beta, s0, _ = rand_case(T=T, S0=True)
    o, fs = oracle.kda_forward(q, k, v, g, beta, 0.8, initial_state=s0, segment_ids=seg)
    t = 0
    for i, n in enumerate(lens):
        sl = slice(t, t + n)
        oi, fi = oracle.kda_forward(q[:, sl], k[:, sl], v[:, sl], g[:, sl], beta[:, sl],
                                    0.8, initial_state=s0 if i == 0 else None)
        np.testing.assert_array_equal(o[:, sl], oi)
        t += n
    np.testing.assert_array_equal(fs, fi)          # state of the last run
    np.testing.assert_array_equal(o[:, t:], 0.0)   # trailing padding


def test_padding_ends_run_and_keeps_initial_state_for_first_run():
    """ids [0,0,1,1,0,1,1,2]: leading padding keeps S0 for the first run;
    padding between equal ids ends the run (the second run of id 1 starts
    from zero); padding rows give o = 0."""
    seg = np.array([[0, 0, 1, 1, 0, 1, 1, 2]], dtype=np.int32)
    q, k, v, g, beta, s0, _ = rand_case(T=8, S0=True)
    o, fs = oracle.kda_forward(q, k, v, g, beta, 1.0, initial_state=s0, segment_ids=seg)
    np.testing.assert_array_equal(o[:, [0, 1, 4]], 0.0)
    o1, _ = oracle.kda_forward(q[:, 2:4], k[:, 2:4], v[:, 2:4], g[:, 2:4], beta[:, 2:4], 1.0,
                               initial_state=s0)
    o2, _ = oracle.kda_forward(q[:, 5:7], k[:, 5:7], v[:, 5:7], g[:, 5:7], beta[:, 5:7], 1.0)
    o3, f3 = oracle.kda_forward(q[:, 7:], k[:, 7:], v[:, 7:], g[:, 7:], beta[:, 7:], 1.0)
    np.testing.assert_array_equal(o[:, 2:4], o1)
    np.testing.assert_array_equal(o[:, 5:7], o2)
    np.testing.assert_array_equal(o[:, 7:], o3)
    np.testing.assert_array_equal(fs, f3)


def test_all_padding_row_returns_initial_state():
    seg = np.zeros((1, 4), dtype=np.int32)
    q, k, v, g, beta, s0, _ = rand_case(T=4, S0=True)
    o, fs = oracle.kda_forward(q, k, v, g, beta, 1.0, initial_state=s0, segment_ids=seg)
    np.testing.assert_array_equal(o, 0.0)
    np.testing.assert_array_equal(fs, s0)


# --- 6. affinity in S0 ----------------------------------------------------------

def test_affine_in_initial_state():
    """o and final_state are affine in S0: f((A+B)/2) = (f(A)+f(B))/2."""
    q, k, v, g, beta, A, _ = rand_case(T=11, S0=True)
    Bm = RNG.standard_normal(A.shape)
    oA, fA = oracle.kda_forward(q, k, v, g, beta, 1.0, initial_state=A)
    oB, fB = oracle.kda_forward(q, k, v, g, beta, 1.0, initial_state=Bm)
    oM, fM = oracle.kda_forward(q, k, v, g, beta, 1.0, initial_state=(A + Bm) / 2)
    np.testing.assert_allclose(oM, (oA + oB) / 2, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(fM, (fA + fB) / 2, rtol=1e-12, atol=1e-13)


# --- 7. split-T hand-off -------------------------------------------------------------

@pytest.mark.parametrize("cut", [1, 6, 13])
def test_split_sequence_state_handoff(cut):
    """[0,cut) then [cut,T) with final -> initial state equals one pass
    (the single-device form of the context-parallel equivalence)."""
    q, k, v, g, beta, s0, _ = rand_case(T=14, S0=True)
    o, fs = oracle.kda_forward(q, k, v, g, beta, 0.6, initial_state=s0)
    a, sl = slice(0, cut), slice(cut, None)
    o1, f1 = oracle.kda_forward(q[:, a], k[:, a], v[:, a], g[:, a], beta[:, a], 0.6, initial_state=s0)
    o2, f2 = oracle.kda_forward(q[:, sl], k[:, sl], v[:, sl], g[:, sl], beta[:, sl], 0.6, initial_state=f1)
    np.testing.assert_array_equal(np.concatenate([o1, o2], 1), o)
    np.testing.assert_array_equal(f2, fs)


# --- 8. brute force on tiny shapes --------------------------------------------------

@pytest.mark.parametrize("shape", [(1, 4, 1, 2, 2), (2, 5, 3, 3, 2), (1, 9, 2, 4, 5)])
@pytest.mark.parametrize("with_seg", [False, True])
def test_matches_independent_transcriptions(shape, with_seg):
    B, T, H, K, V = shape
    seg = None
    if with_seg:
        seg = np.ones((B, T), dtype=np.int32)
        seg[:, T // 2:] = 2
        seg[:, -1] = 0
    q, k, v, g, beta, s0, _ = rand_case(B, T, H, K, V, S0=True)
    o, fs = oracle.kda_forward(q, k, v, g, beta, 0.75, initial_state=s0, segment_ids=seg)
    om, fm = matrix_form(q, k, v, g, beta, 0.75, s0, seg)
    ot, ft = transition_form(q, k, v, g, beta, 0.75, s0, seg)
    np.testing.assert_allclose(o, om, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(fs, fm, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(o, ot, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(fs, ft, rtol=1e-11, atol=1e-12)


# --- 9. independence and determinism ------------------------------------------------

def test_row_and_head_independence():
    q, k, v, g, beta, s0, _ = rand_case(B=2, T=6, H=3, S0=True)
    o, fs = oracle.kda_forward(q, k, v, g, beta, 1.0, initial_state=s0)
    q2 = q.copy(); v2 = v.copy()
    q2[1] += 1.0; v2[:, :, 2] -= 3.0
    o2, fs2 = oracle.kda_forward(q2, k, v2, g, beta, 1.0, initial_state=s0)
    np.testing.assert_array_equal(o2[0, :, :2], o[0, :, :2])
    np.testing.assert_array_equal(fs2[0, :2], fs[0, :2])
    assert not np.array_equal(o2[1], o[1])


def test_thread_count_does_not_change_result():
    q, k, v, g, beta, s0, _ = rand_case(B=2, T=20, H=5, K=8, V=6, S0=True)
    o1, f1 = oracle.kda_forward(q, k, v, g, beta, 1.0, initial_state=s0, threads=1)
    o7, f7 = oracle.kda_forward(q, k, v, g, beta, 1.0, initial_state=s0, threads=7)
    np.testing.assert_array_equal(o1, o7)
    np.testing.assert_array_equal(f1, f7)


def test_default_scale_is_inverse_sqrt_k():
    q, k, v, g, beta, _, _ = rand_case(T=3, K=4)
    o1, _ = oracle.kda_forward(q, k, v, g, beta, None)
    o2, _ = oracle.kda_forward(q, k, v, g, beta, 0.5)
    np.testing.assert_array_equal(o1, o2)


# --- short convolution + SiLU and L2 norm ------------------------------------------

def _torch_conv_silu(x, w):
    """Library reference: depthwise causal conv1d (left padding W-1) + SiLU."""
    xt = torch.from_numpy(x).permute(0, 2, 1)            # [B, C, T]
    W = w.shape[1]
    y = torch.nn.functional.conv1d(torch.nn.functional.pad(xt, (W - 1, 0)),
                                   torch.from_numpy(w)[:, None, :], groups=w.shape[0])
    return torch.nn.functional.silu(y).permute(0, 2, 1).numpy()


def test_conv_identity_tap_is_silu():
    x = RNG.standard_normal((1, 9, 6))
    w = np.zeros((6, 4)); w[:, 3] = 1.0
    y = oracle.short_conv_silu(x, w)
    ref = torch.nn.functional.silu(torch.from_numpy(x)).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-14, atol=1e-15)


def test_conv_matches_library_conv1d():
    x = RNG.standard_normal((2, 17, 5))
    w = RNG.standard_normal((5, 4))
    np.testing.assert_allclose(oracle.short_conv_silu(x, w), _torch_conv_silu(x, w),
                               rtol=1e-12, atol=1e-13)


def test_conv_segment_aware_equals_per_segment_library_conv():
    lens = [3, 1, 6, 5]
    T = sum(lens) + 2
    seg = ki.segment_ids_from_lengths(1, T, lens).numpy()
    x = RNG.standard_normal((1, T, 4))
    w = RNG.standard_normal((4, 4))
    y = oracle.short_conv_silu(x, w, seg)
    t = 0
    for n in lens:
        np.testing.assert_allclose(y[:, t:t + n], _torch_conv_silu(x[:, t:t + n], w),
                                   rtol=1e-12, atol=1e-13)
        t += n
    np.testing.assert_array_equal(y[:, t:], 0.0)


def test_l2norm_closed_form():
    x = np.array([[3.0, 4.0], [0.0, 0.0]])
    y = oracle.l2norm(x, 2, eps=1e-6)
    np.testing.assert_allclose(y[0], [3 / np.sqrt(25 + 1e-6), 4 / np.sqrt(25 + 1e-6)], rtol=1e-15)
    np.testing.assert_array_equal(y[1], [0.0, 0.0])
    z = oracle.l2norm(RNG.standard_normal((7, 3, 8)), 8, eps=0.0)
    np.testing.assert_allclose(np.linalg.norm(z.reshape(-1, 8), axis=-1), 1.0, rtol=1e-14)
