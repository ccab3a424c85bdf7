"""The chunked algebra the kernels implement equals the token oracle.

``chunk_model.chunk_forward`` (fp64) restates the kernels' chunk form: the
gate cumsum, the 16-row sub-block exponent factors, the strict (A_kk) and
inclusive (A_qk) diagonals, the UT transform, ragged chunk tails and run
resets.  If it agrees with the oracle to rounding, the algebra is right and
any GPU mismatch is an implementation bug.  The bf16-operand variant
estimates the error budget of the tensor-core kernel against the tolerances
(max-abs 2e-2, rel-L2 1e-2).
"""
import numpy as np
import pytest

import kda_inputs as ki
import oracle
from chunk_model import chunk_forward, naive_intra_products, intra_products, decay_factors

RNG = np.random.default_rng(7)


def case(T, H=2, K=16, V=8, gmin=-5.0, S0=True, seg=None, B=1):
    q = RNG.standard_normal((B, T, H, K)); q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k = RNG.standard_normal((B, T, H, K)); k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = RNG.standard_normal((B, T, H, V))
    g = RNG.uniform(gmin, 0.0, (B, T, H, K))
    beta = RNG.uniform(0, 1, (B, T, H))
    s0 = RNG.standard_normal((B, H, K, V)) * 0.1 if S0 else None
    return q, k, v, g, beta, s0, seg


def rel_l2(a, b):
    return np.linalg.norm(a - b) / np.linalg.norm(b)


@pytest.mark.parametrize("T", [1, 17, 64, 65, 150])
def test_chunk_algebra_equals_oracle(T):
    q, k, v, g, beta, s0, _ = case(T)
    o_ref, f_ref = oracle.kda_forward(q, k, v, g, beta, 0.25, initial_state=s0)
    o, f = chunk_forward(q, k, v, g, beta, 0.25, s0)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(f, f_ref, rtol=0, atol=1e-12)


def test_chunk_algebra_worst_case_gate():
    """g = -5 on every channel: the chunk-wide exponent span is 320, beyond
    fp32/bf16 range, so this fails unless the sub-block factoring is right."""
    q, k, v, g, beta, s0, _ = case(130)
    g[:] = -5.0
    o_ref, f_ref = oracle.kda_forward(q, k, v, g, beta, 1.0, initial_state=s0)
    o, f = chunk_forward(q, k, v, g, beta, 1.0, s0)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(f, f_ref, rtol=1e-9, atol=1e-15)


def test_sub_block_factoring_stays_finite_in_fp32():
    """In fp32 (the kernels' precision) with g = -5 the sub-block factors
    stay finite and match the oracle, while the chunk-wide factoring
    exp(G_r) exp(-G_j) overflows -- the reason for 16-row sub-blocks."""
    q, k, v, g, beta, s0, _ = case(128, K=32, V=16)
    g[:] = -5.0
    Kc = k[0, :64, 0].astype(np.float32)
    Gc = np.cumsum(g[0, :64, 0].astype(np.float32), axis=0)
    with np.errstate(over="ignore", invalid="ignore"):
        Akk_naive, _ = naive_intra_products(Kc, Kc, Gc)
    assert not np.all(np.isfinite(np.tril(Akk_naive)))
    Akk, Aqk = intra_products(Kc, Kc, decay_factors(Gc))
    assert np.all(np.isfinite(Akk)) and np.all(np.isfinite(Aqk))
    o_ref, f_ref = oracle.kda_forward(q, k, v, g, beta, 1.0, initial_state=s0)
    o, f = chunk_forward(q, k, v, g, beta, 1.0, s0, dtype=np.float32)
    assert o.dtype == np.float32
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=2e-6)
    np.testing.assert_allclose(f, f_ref, rtol=0, atol=2e-6)


def test_chunk_algebra_packed_runs():
    lens = [64, 1, 70, 33, 128]
    T = sum(lens) + 5
    seg = ki.segment_ids_from_lengths(2, T, [lens, [("pad", 3), 150, 40]]).numpy()
    q, k, v, g, beta, s0, _ = case(T, B=2)
    o_ref, f_ref = oracle.kda_forward(q, k, v, g, beta, 0.5, initial_state=s0, segment_ids=seg)
    o, f = chunk_forward(q, k, v, g, beta, 0.5, s0, seg)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(f, f_ref, rtol=0, atol=1e-12)


def test_bf16_operand_rounding_within_budget():
    """Rounding every tensor-core operand to bf16 (fp32 state and
    accumulators) on the pages' K = V = 128 shape keeps o and final_state
    within half the bf16 tolerances."""
    w = ki.custom_workload(B=1, T=256, H=1, K=128, V=128, init_state_std=0.1)
    x = ki.make_inputs(w, seed=3)
    args = [oracle._f64(x[n]) for n in ("q", "k", "v", "g", "beta")]
    s0 = oracle._f64(x["initial_state"])
    o_ref, f_ref = oracle.kda_forward(*args, x["scale"], initial_state=s0)
    o, f = chunk_forward(*args, x["scale"], s0, bf16_operands=True)
    assert np.abs(o - o_ref).max() < 1e-2 and rel_l2(o, o_ref) < 5e-3
    assert np.abs(f - f_ref).max() < 1e-2 and rel_l2(f, f_ref) < 5e-3
