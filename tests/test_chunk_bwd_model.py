"""The chunked backward algebra (tests/chunk_bwd_model.py) equals the
token-level backward oracle: every gradient, across chunk boundaries, ragged
chunk tails, run resets, padding and an initial state, for C = 16 and 64."""
import numpy as np
import pytest

import oracle
from chunk_bwd_model import chunk_backward
from test_oracle_bwd import NAMES, _case

CASES = {
    "plain_T150": dict(B=1, T=150, H=2, K=8, V=6, segments=None),
    "packed": dict(B=2, T=140, H=1, K=6, V=5,
                   segments=[[("pad", 3), 40, 1, ("pad", 2), 70, 24], [64, 64, 12]]),
}


@pytest.mark.parametrize("C", [16, 64])
@pytest.mark.parametrize("case", sorted(CASES))
def test_chunked_backward_equals_token_oracle(case, C):
    kw = dict(CASES[case])
    c = _case(kw.pop("B"), kw.pop("T"), kw.pop("H"), kw.pop("K"), kw.pop("V"), seed=13,
              segments=kw.pop("segments"))
    ref = oracle.kda_backward(c["q"], c["k"], c["v"], c["g"], c["beta"], c["scale"],
                              initial_state=c["s0"], segment_ids=c["seg"], d_o=c["d_o"],
                              d_final=c["d_f"])
    got = chunk_backward(c["q"], c["k"], c["v"], c["g"], c["beta"], c["scale"], S0=c["s0"],
                         seg=c["seg"], d_o=c["d_o"], d_final=c["d_f"], C=C)
    for name, a, b in zip(NAMES, got, ref):
        np.testing.assert_allclose(a, b, rtol=1e-8, atol=1e-10, err_msg=name)
