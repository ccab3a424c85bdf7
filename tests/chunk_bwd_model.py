"""numpy fp64 model of the CHUNKED backward: the gradient of the chunk form
of tests/chunk_model.py, chunk by chunk in reverse.

Test code (not the oracle, not a GPU path): it fixes the algebra a
tensor-core backward would evaluate and checks it against the token-level
backward oracle on the CPU.  Per chunk of C rows with entering state S (rows
past the run end are zero), the forward is

    G = cumsum(g), Gam = e^G, gam = e^{G_C}, Kt = K*Gam, Qt = Q*Gam,
    Kh = K*e^{G_C - G}, Akk[r,j] = sum_c k_rc k_jc e^{G_rc - G_jc} (j < r),
    Aqk[r,j] = sum_c q_rc k_jc e^{G_rc - G_jc} (j <= r), L = diag(beta) Akk,
    T = (I + L)^-1, u = T diag(beta) V, w = T diag(beta) Kt,
    U = u - w S, O = scale (Qt S + Aqk U), S' = gam * S + Kh^T U,

and, given dO and dS' (the gradient of the state leaving the chunk),

    dU  = scale Aqk^T dO + Kh dS'
    dS  = scale Qt^T dO + gam * dS' - w^T dU          (the state chain, reversed)
    dQt = scale dO S^T,  dAqk = scale dO U^T (j <= r),  dKh = U dS'^T,
    dgam = rowsum(S * dS'),  dw = -dU S^T,  du = dU,
    [du | dw] = T [diag(beta) V | diag(beta) Kt]  ->  dT = [du|dw] Y^T, dY = T^T [du|dw],
    dL = -T^T dT T^T (j < r),  dbeta, dAkk = diag(beta) dL,
then through Akk, Aqk, Qt, Kt, Kh, gam to q, k, v, beta and G, and dg is the
reverse cumsum of dG within the chunk.  The state chain is the only serial
part: everything else is per chunk given S, dS' and dU.
"""
from __future__ import annotations

import numpy as np

from chunk_model import _runs


def _chunk_fwd_quantities(Qc, Kc, Vc, gc, bc):
    C = Qc.shape[0]
    G = np.cumsum(gc, axis=0)
    Gam = np.exp(G)
    GC = G[-1]
    gam = np.exp(GC)
    Kt, Qt = Kc * Gam, Qc * Gam
    Kh = Kc * np.exp(GC[None, :] - G)
    # e^{G_r - G_j} for j <= r, per channel: [r, j, c]
    D = np.exp(np.tril(np.ones((C, C)))[:, :, None] * (G[:, None, :] - G[None, :, :]))
    low = np.tril(np.ones((C, C)), -1)
    incl = np.tril(np.ones((C, C)))
    Akk = np.einsum("rc,jc,rjc->rj", Kc, Kc, D) * low
    Aqk = np.einsum("rc,jc,rjc->rj", Qc, Kc, D) * incl
    L = bc[:, None] * Akk
    T = np.linalg.inv(np.eye(C) + L)
    Y = np.concatenate([bc[:, None] * Vc, bc[:, None] * Kt], axis=1)
    X = T @ Y
    V = Vc.shape[1]
    return dict(G=G, Gam=Gam, GC=GC, gam=gam, Kt=Kt, Qt=Qt, Kh=Kh, D=D, low=low, incl=incl,
                Akk=Akk, Aqk=Aqk, T=T, Y=Y, u=X[:, :V], w=X[:, V:])


def chunk_backward(q, k, v, g, beta, scale, S0=None, seg=None, d_o=None, d_final=None, C=64):
    q, k, v, g, beta = (np.asarray(x, dtype=np.float64) for x in (q, k, v, g, beta))
    B, T, H, K = q.shape
    V = v.shape[-1]
    d_o = np.zeros((B, T, H, V)) if d_o is None else np.asarray(d_o, dtype=np.float64)
    dq = np.zeros((B, T, H, K)); dk = np.zeros((B, T, H, K)); dg = np.zeros((B, T, H, K))
    dv = np.zeros((B, T, H, V)); dbeta = np.zeros((B, T, H)); dS0 = np.zeros((B, H, K, V))
    for b in range(B):
        runs = _runs(None if seg is None else np.asarray(seg)[b], T)
        for h in range(H):
            # forward: the state entering every chunk of every run
            S = np.zeros((K, V)) if S0 is None else np.array(S0[b, h], dtype=np.float64)
            chunks = []
            for ri, (s, e) in enumerate(runs):
                if ri > 0:
                    S = np.zeros((K, V))
                for c0 in range(s, e, C):
                    n = min(C, e - c0)
                    Qc = np.zeros((C, K)); Kc = np.zeros((C, K)); Vc = np.zeros((C, V))
                    gc = np.zeros((C, K)); bc = np.zeros(C)
                    Qc[:n] = q[b, c0:c0 + n, h]; Kc[:n] = k[b, c0:c0 + n, h]
                    Vc[:n] = v[b, c0:c0 + n, h]; gc[:n] = g[b, c0:c0 + n, h]
                    bc[:n] = beta[b, c0:c0 + n, h]
                    F = _chunk_fwd_quantities(Qc, Kc, Vc, gc, bc)
                    U = F["u"] - F["w"] @ S
                    chunks.append((ri, c0, n, Qc, Kc, Vc, bc, F, S.copy(), U))
                    S = F["gam"][:, None] * S + F["Kh"].T @ U
            # backward, chunk by chunk from the end
            dS = np.zeros((K, V)) if d_final is None else np.array(d_final[b, h], dtype=np.float64)
            n_runs = len(runs)
            for idx in range(len(chunks) - 1, -1, -1):
                ri, c0, n, Qc, Kc, Vc, bc, F, S, U = chunks[idx]
                dO = np.zeros((C, V)); dO[:n] = d_o[b, c0:c0 + n, h]
                dSn = dS                                   # gradient of S'
                dU = scale * F["Aqk"].T @ dO + F["Kh"] @ dSn
                dS = scale * F["Qt"].T @ dO + F["gam"][:, None] * dSn - F["w"].T @ dU
                dQt = scale * dO @ S.T
                dAqk = scale * (dO @ U.T) * F["incl"]
                dKh = U @ dSn.T
                dgam = np.sum(S * dSn, axis=1)
                dw = -dU @ S.T
                dX = np.concatenate([dU, dw], axis=1)
                dT = dX @ F["Y"].T
                dY = F["T"].T @ dX
                dL = -(F["T"].T @ dT @ F["T"].T) * F["low"]
                dYv, dYk = dY[:, :V], dY[:, V:]
                dV = bc[:, None] * dYv
                db = np.sum(dYv * Vc, axis=1) + np.sum(dYk * F["Kt"], axis=1) \
                    + np.sum(dL * F["Akk"], axis=1)
                dAkk = bc[:, None] * dL
                dKt = bc[:, None] * dYk
                D = F["D"]
                # Akk[r,j] = sum_c k_rc k_jc D[r,j,c];  Aqk[r,j] = sum_c q_rc k_jc D[r,j,c]
                dQ = np.einsum("rj,jc,rjc->rc", dAqk, Kc, D)
                dK = (np.einsum("rj,jc,rjc->rc", dAkk, Kc, D)
                      + np.einsum("rj,rc,rjc->jc", dAkk, Kc, D)
                      + np.einsum("rj,rc,rjc->jc", dAqk, Qc, D))
                tk = np.einsum("rj,rc,jc,rjc->rjc", dAkk, Kc, Kc, D) \
                    + np.einsum("rj,rc,jc,rjc->rjc", dAqk, Qc, Kc, D)
                dG = tk.sum(axis=1) - tk.sum(axis=0)        # d/dG_r minus d/dG_j
                dQ += dQt * F["Gam"]; dG += dQt * F["Qt"]
                dK += dKt * F["Gam"]; dG += dKt * F["Kt"]
                eKh = np.exp(F["GC"][None, :] - F["G"])
                dK += dKh * eKh
                dG -= dKh * F["Kh"]
                dGC = np.sum(dKh * F["Kh"], axis=0) + dgam * F["gam"]
                dG[C - 1] += dGC
                dgc = np.cumsum(dG[::-1], axis=0)[::-1]     # G = cumsum(g)
                dq[b, c0:c0 + n, h] = dQ[:n]; dk[b, c0:c0 + n, h] = dK[:n]
                dv[b, c0:c0 + n, h] = dV[:n]; dg[b, c0:c0 + n, h] = dgc[:n]
                dbeta[b, c0:c0 + n, h] = db[:n]
                first_chunk_of_run = idx == 0 or chunks[idx - 1][0] != ri
                if first_chunk_of_run and ri > 0:
                    dS = np.zeros((K, V))                  # the reset stops the gradient
            if n_runs == 0:
                dS = np.zeros((K, V)) if d_final is None else np.array(d_final[b, h])
            dS0[b, h] = dS
    return dq, dk, dv, dg, dbeta, dS0
