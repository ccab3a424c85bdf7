"""Independent transcriptions of the gated delta rule, used to pin the oracle.

These are written separately from ``oracle/kda_ref.c`` and evaluate the same
recurrence (page "feat(kda): integrate KDA attention with tokamax backend and
CP support", section "Delta Rule formulation") in two *different* orders, so a
dropped term, a wrong sign or a transposed operand in the oracle shows up as a
mismatch:

* :func:`matrix_form` -- token by token with numpy matrix algebra
  (``np.diag``, ``np.outer``, ``@``), one head at a time, tiny shapes only.
* :func:`transition_form` -- the same recurrence rewritten as an affine map
  per token, ``S_t = (I - beta_t k_t k_t^T) diag(exp g_t) S_{t-1} + beta_t k_t
  v_t^T``, which follows from substituting the residual into the update.
  The state after a run is the ordered product of the transitions applied to
  the start state plus the propagated offsets.
"""
from __future__ import annotations

import numpy as np


def _runs(seg_row, T):
    """List of (start, end) runs of equal non-zero ids, in order."""
    runs = []
    t = 0
    while t < T:
        s = 1 if seg_row is None else int(seg_row[t])
        if s == 0:
            t += 1
            continue
        e = t
        while e < T and (1 if seg_row is None else int(seg_row[e])) == s:
            e += 1
        runs.append((t, e))
        t = e
    return runs


def matrix_form(q, k, v, g, beta, scale, S0=None, seg=None):
    """Token-level numpy transcription.  Shapes as the oracle's (fp64)."""
    q, k, v, g, beta = (np.asarray(x, dtype=np.float64) for x in (q, k, v, g, beta))
    B, T, H, K = q.shape
    V = v.shape[-1]
    o = np.zeros((B, T, H, V))
    fs = np.zeros((B, H, K, V))
    for b in range(B):
        runs = _runs(None if seg is None else np.asarray(seg)[b], T)
        for h in range(H):
            S = np.zeros((K, V)) if S0 is None else np.array(S0[b, h], dtype=np.float64)
            for ri, (s, e) in enumerate(runs):
                if ri > 0:
                    S = np.zeros((K, V))
                for t in range(s, e):
                    Sp = np.diag(np.exp(g[b, t, h])) @ S
                    res = v[b, t, h] - k[b, t, h] @ Sp
                    S = Sp + beta[b, t, h] * np.outer(k[b, t, h], res)
                    o[b, t, h] = scale * (q[b, t, h] @ S)
            fs[b, h] = S
    return o, fs


def transition_form(q, k, v, g, beta, scale, S0=None, seg=None):
    """Affine-map transcription: S_t = A_t S_{t-1} + c_t per token."""
    q, k, v, g, beta = (np.asarray(x, dtype=np.float64) for x in (q, k, v, g, beta))
    B, T, H, K = q.shape
    V = v.shape[-1]
    o = np.zeros((B, T, H, V))
    fs = np.zeros((B, H, K, V))
    I = np.eye(K)
    for b in range(B):
        runs = _runs(None if seg is None else np.asarray(seg)[b], T)
        for h in range(H):
            start = np.zeros((K, V)) if S0 is None else np.array(S0[b, h], dtype=np.float64)
            S_end = start
            for ri, (s, e) in enumerate(runs):
                S_in = start if ri == 0 else np.zeros((K, V))
                # Accumulate the composite map P (K x K) and offset R (K x V)
                # so that the state after token t is P @ S_in + R.
                P = np.eye(K)
                R = np.zeros((K, V))
                for t in range(s, e):
                    kt = k[b, t, h]
                    A = (I - beta[b, t, h] * np.outer(kt, kt)) * np.exp(g[b, t, h])[None, :]
                    c = beta[b, t, h] * np.outer(kt, v[b, t, h])
                    P = A @ P
                    R = A @ R + c
                    o[b, t, h] = scale * ((P @ S_in + R).T @ q[b, t, h])
                S_end = P @ S_in + R
            fs[b, h] = S_end
    return o, fs
