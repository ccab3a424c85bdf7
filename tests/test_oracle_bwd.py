"""Pins of the fp64 backward oracle (``oracle.kda_backward``), none of which
reuse its hand-derived adjoint:

* reverse-mode autodiff (torch.autograd, fp64) of a plain token-by-token
  transcription of the forward recurrence, on tiny packed shapes with
  padding, run resets, a repeated id after padding and an initial state;
* central finite differences of the C forward oracle along random
  directions, for every input;
* the packed-sequence identity: the gradients of a packed row equal those of
  its runs taken one at a time;
* zero upstream gradients give zero gradients; padding tokens get zero
  gradients; an all-padding row hands d_final straight to d_initial.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.filterwarnings("ignore")


def _case(B, T, H, K, V, seed, segments=None, with_s0=True):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, T, H, K))
    k = rng.standard_normal((B, T, H, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, V))
    g = -5.0 * rng.random((B, T, H, K))
    beta = rng.random((B, T, H))
    s0 = 0.3 * rng.standard_normal((B, H, K, V)) if with_s0 else None
    seg = None
    if segments is not None:
        seg = np.zeros((B, T), dtype=np.int32)
        for b, items in enumerate(segments):
            t, sid = 0, 0
            for it in items:
                if isinstance(it, tuple):
                    t += it[1]
                else:
                    sid += 1
                    seg[b, t:t + it] = sid
                    t += it
    d_o = rng.standard_normal((B, T, H, V))
    d_f = rng.standard_normal((B, H, K, V))
    return dict(q=q, k=k, v=v, g=g, beta=beta, s0=s0, seg=seg, d_o=d_o, d_f=d_f,
                scale=K ** -0.5)


def _torch_forward(q, k, v, g, beta, scale, s0, seg):
    """The recurrence written out once more, in torch fp64, for autograd."""
    B, T, H, K = q.shape
    V = v.shape[-1]
    outs, finals = [], []
    for b in range(B):
        ob, fb = [], []
        for h in range(H):
            S = s0[b, h] if s0 is not None else torch.zeros(K, V, dtype=torch.float64)
            seen, prev, oh = False, 0, []
            for t in range(T):
                s = int(seg[b, t]) if seg is not None else 1
                if s == 0:
                    oh.append(torch.zeros(V, dtype=torch.float64))
                    prev = 0
                    continue
                if s != prev:
                    if seen:
                        S = torch.zeros(K, V, dtype=torch.float64)
                    seen = True
                prev = s
                Sp = S * torch.exp(g[b, t, h])[:, None]
                r = v[b, t, h] - Sp.T @ k[b, t, h]
                S = Sp + beta[b, t, h] * torch.outer(k[b, t, h], r)
                oh.append(scale * (S.T @ q[b, t, h]))
            ob.append(torch.stack(oh))
            fb.append(S)
        outs.append(torch.stack(ob, dim=1))
        finals.append(torch.stack(fb))
    return torch.stack(outs), torch.stack(finals)


def _autograd(c):
    t = {n: torch.tensor(c[n], dtype=torch.float64, requires_grad=True)
         for n in ("q", "k", "v", "g", "beta")}
    s0 = (torch.tensor(c["s0"], dtype=torch.float64, requires_grad=True)
          if c["s0"] is not None else None)
    o, fs = _torch_forward(t["q"], t["k"], t["v"], t["g"], t["beta"], c["scale"], s0, c["seg"])
    L = (o * torch.tensor(c["d_o"])).sum() + (fs * torch.tensor(c["d_f"])).sum()
    L.backward()
    grads = [t[n].grad.numpy() for n in ("q", "k", "v", "g", "beta")]
    grads.append(s0.grad.numpy() if s0 is not None else None)
    return grads


def _oracle(c, **kw):
    return oracle.kda_backward(c["q"], c["k"], c["v"], c["g"], c["beta"], c["scale"],
                               initial_state=c["s0"], segment_ids=c["seg"], d_o=c["d_o"],
                               d_final=c["d_f"], **kw)


NAMES = ("dq", "dk", "dv", "dg", "dbeta", "d_initial")
SEGMENTS = {
    "plain": None,
    "packed": [[3, ("pad", 1), 5, 3], [("pad", 2), 4, 4, 2]],
    "len1_runs": [[1, 1, 2, ("pad", 2), 1, 5], [12]],
}


@pytest.mark.parametrize("segs", sorted(SEGMENTS))
@pytest.mark.parametrize("with_s0", [True, False])
def test_backward_matches_autograd(segs, with_s0):
    c = _case(2, 12, 2, 3, 4, seed=5, segments=SEGMENTS[segs], with_s0=with_s0)
    got = _oracle(c)
    ref = _autograd(c)
    for name, a, b in zip(NAMES, got, ref):
        if b is None:
            continue
        np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-12, err_msg=name)


def test_backward_matches_autograd_across_checkpoint_blocks():
    """T = 150 spans three 64-token replay blocks, with a run start at 64."""
    c = _case(1, 150, 1, 4, 3, seed=8, segments=[[64, 40, ("pad", 6), 40]])
    got = _oracle(c)
    ref = _autograd(c)
    for name, a, b in zip(NAMES, got, ref):
        np.testing.assert_allclose(a, b, rtol=1e-9, atol=1e-12, err_msg=name)


def _loss(c, **over):
    x = dict(c, **over)
    o, fs = oracle.kda_forward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"],
                               initial_state=x["s0"], segment_ids=x["seg"])
    return float((o * c["d_o"]).sum() + (fs * c["d_f"]).sum())


@pytest.mark.parametrize("segs", ["plain", "packed"])
def test_backward_matches_finite_differences(segs):
    c = _case(2, 12, 2, 4, 3, seed=11, segments=SEGMENTS[segs])
    grads = dict(zip(NAMES, _oracle(c)))
    rng = np.random.default_rng(3)
    eps = 1e-6
    for name, key in [("dq", "q"), ("dk", "k"), ("dv", "v"), ("dg", "g"), ("dbeta", "beta"),
                      ("d_initial", "s0")]:
        d = rng.standard_normal(c[key].shape)
        fd = (_loss(c, **{key: c[key] + eps * d}) - _loss(c, **{key: c[key] - eps * d})) / (2 * eps)
        an = float((grads[name] * d).sum())
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, fd, an)


def test_packed_gradients_equal_per_run_gradients():
    """Each run of a packed row is its own problem: its gradients equal those
    of the run taken alone (zero entering state, no d_final unless it is the
    row's last run), and the first run alone carries d_initial."""
    runs = [4, 6, 5]
    c = _case(1, 16, 2, 3, 3, seed=2, segments=[[runs[0], runs[1], ("pad", 1), runs[2]]])
    got = dict(zip(NAMES, _oracle(c)))
    starts = [0, 4, 11]
    for i, (t0, n) in enumerate(zip(starts, runs)):
        sl = slice(t0, t0 + n)
        one = {kk: (c[kk][:, sl] if kk in ("q", "k", "v", "g", "beta", "d_o") else c[kk])
               for kk in c}
        one["seg"] = None
        one["s0"] = c["s0"] if i == 0 else np.zeros_like(c["s0"])
        one["d_f"] = c["d_f"] if i == len(runs) - 1 else np.zeros_like(c["d_f"])
        alone = dict(zip(NAMES, _oracle(one)))
        for name in ("dq", "dk", "dv", "dg", "dbeta"):
            np.testing.assert_allclose(got[name][:, sl], alone[name], rtol=1e-12, atol=1e-14,
                                       err_msg=f"run {i} {name}")
        if i == 0:
            np.testing.assert_allclose(got["d_initial"], alone["d_initial"], rtol=1e-12,
                                       atol=1e-14)
    pad = c["seg"][0] == 0
    for name in ("dq", "dk", "dv", "dg", "dbeta"):
        assert np.all(got[name][:, pad] == 0), name


def test_zero_upstream_and_all_padding_row():
    c = _case(2, 10, 1, 3, 2, seed=4, segments=[[10], [("pad", 10)]])
    c0 = dict(c, d_o=np.zeros_like(c["d_o"]), d_f=np.zeros_like(c["d_f"]))
    for a in _oracle(c0):
        assert np.all(a == 0)
    got = dict(zip(NAMES, _oracle(c)))
    np.testing.assert_array_equal(got["d_initial"][1], c["d_f"][1])   # final = S0 there
    for name in ("dq", "dk", "dv", "dg", "dbeta"):
        assert np.all(got[name][1] == 0), name


def test_threads_do_not_change_the_result():
    c = _case(2, 40, 3, 4, 5, seed=9, segments=[[10, 30], [("pad", 3), 37]])
    a = _oracle(c, threads=1)
    b = _oracle(c, threads=4)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
