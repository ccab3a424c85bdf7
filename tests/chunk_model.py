"""numpy model of the chunked algebra the CUDA kernels implement.

This is test code, not the oracle and not the GPU path.  It restates, in
float64 (optionally with bf16 rounding of the operands the tensor-core kernel
rounds), the chunk form of the gated delta rule (page "feat(kda): integrate
KDA attention with tokamax backend and CP support", section "Delta Rule
formulation") that the kernels evaluate, so that the algebra -- inclusive vs
strict diagonals, the sub-block exponent references, ragged chunk tails and
run resets -- is checked against the token oracle on the CPU before and
independently of any CUDA.

Per run and chunk of C rows (rows past the run end are zero: q = k = v = 0,
beta = 0, g = 0), with the state S0 entering the chunk:

    G       = inclusive cumsum of g over the chunk's rows (per key channel)
    A_kk[r,j] = beta_r * sum_c k_rc k_jc exp(G_rc - G_jc)   (j <  r)
    A_qk[r,j] =          sum_c q_rc k_jc exp(G_rc - G_jc)   (j <= r)
    T       = (I + A_kk)^-1
    u       = T diag(beta) V,      w = T diag(beta) (K * exp(G))
    U       = u - w S0
    O       = scale * ((Q * exp(G)) S0 + A_qk U)
    S1      = diag(exp(G_C)) S0 + (K * exp(G_C - G))^T U

The exponentials exp(G_r - G_j) are never formed from exp(G_r) * exp(-G_j)
over the whole chunk (the span reaches 64 * 5 = 320 > ln(FLT_MAX)); they are
factored per 16-row sub-block b with the reference P_b = G at the row before
the block (P_0 = 0) and the block end E_b = G at the block's last row:

    E1_r = exp(G_r - P_b)           in [e^-80, 1]
    E2_r = exp(E_b - G_r)           in [e^-75, 1]
    same block  (j <= r):  exp(G_r - G_j) = E1_r * (1 / E1_j)
    earlier block b' < b:  exp(G_r - G_j) = E1_r * exp(P_b - E_b') * E2_j
    exp(G_r)       = E1_r * exp(P_b)
    exp(G_C - G_r) = E2_r * exp(G_C - E_b)

and the per-channel factors exp(P_b - E_b'), exp(P_b), exp(G_C - E_b) are
products of the block decays exp(E_i - P_i), all <= 1.  The kernels use the
same factors.
"""
from __future__ import annotations

import numpy as np

C_DEFAULT = 64
SUB = 16


def _bf16(x):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float64)).to(
        torch.bfloat16).to(torch.float64).numpy()


def _runs(seg_row, T):
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


def decay_factors(Gc, sub=SUB):
    """Sub-block factors of one chunk.  Gc: [C, K] inclusive cumsum."""
    C, K = Gc.shape
    nb = C // sub
    dt = Gc.dtype
    P = np.zeros((nb, K), dt)      # reference before block b
    E = np.zeros((nb, K), dt)      # G at block b's last row
    for b in range(nb):
        P[b] = 0.0 if b == 0 else Gc[b * sub - 1]
        E[b] = Gc[b * sub + sub - 1]
    Dblk = np.exp(E - P)           # block decays, <= 1
    blk = np.arange(C) // sub
    E1 = np.exp(Gc - P[blk])
    E2 = np.exp(E[blk] - Gc)
    # prefix products: exp(P_b) = prod_{i<b} Dblk_i ; suffix exp(G_C - E_b)
    pre = np.ones((nb, K), dt)
    for b in range(1, nb):
        pre[b] = pre[b - 1] * Dblk[b - 1]
    suf = np.ones((nb, K), dt)
    for b in range(nb - 2, -1, -1):
        suf[b] = suf[b + 1] * Dblk[b + 1]
    # cross factor exp(P_b - E_b') for b' < b: prod_{i=b'+1}^{b-1} Dblk_i
    cross = np.ones((nb, nb, K), dt)
    for b in range(nb):
        for bp in range(b):
            f = np.ones(K, dt)
            for i in range(bp + 1, b):
                f = f * Dblk[i]
            cross[b, bp] = f
    gammaC = pre[nb - 1] * Dblk[nb - 1]
    return dict(E1=E1, E2=E2, Dblk=Dblk, pre=pre, suf=suf, cross=cross,
                gammaC=gammaC, blk=blk)


def intra_products(Qc, Kc, F, sub=SUB, rnd=lambda x: x):
    """A_raw_kk[r,j] = sum_c k_rc k_jc e^{G_rc-G_jc}, A_qk likewise, for
    j <= r, via the sub-block factors (no beta, no masks applied)."""
    C, K = Kc.shape
    E1, E2, blk, cross = F["E1"], F["E2"], F["blk"], F["cross"]
    Akk = np.zeros((C, C), Kc.dtype)
    Aqk = np.zeros((C, C), Kc.dtype)
    Xk = rnd(Kc * E1)
    Xq = rnd(Qc * E1)
    for r in range(C):
        b = blk[r]
        for j in range(r + 1):
            bp = blk[j]
            if bp == b:
                y = rnd(Kc[j] / E1[j])
            else:
                y = rnd(Kc[j] * E2[j] * cross[b, bp])
            Akk[r, j] = Xk[r] @ y
            Aqk[r, j] = Xq[r] @ y
    return Akk, Aqk


def naive_intra_products(Qc, Kc, Gc):
    """The factoring the sub-blocks avoid: exp(G_r) * exp(-G_j) over the
    whole chunk.  exp(-G_j) overflows once -G_j > ln(max float)."""
    Xk = Kc * np.exp(Gc)
    Y = Kc * np.exp(-Gc)
    return Xk @ Y.T, (Qc * np.exp(Gc)) @ Y.T


def chunk_forward(q, k, v, g, beta, scale, S0=None, seg=None, C=C_DEFAULT,
                  sub=SUB, bf16_operands=False, dtype=np.float64):
    """Chunked forward over the same layouts as the oracle, computed in
    ``dtype`` (float64, or float32 as the kernels do).  ``bf16_operands``
    rounds every tensor-core operand to bf16."""
    rnd = _bf16 if bf16_operands else (lambda x: x)
    if bf16_operands and dtype != np.float64:
        raise ValueError("bf16 emulation runs in float64")
    q, k, v, g, beta = (np.asarray(x, dtype=dtype) for x in (q, k, v, g, beta))
    B, T, H, K = q.shape
    V = v.shape[-1]
    o = np.zeros((B, T, H, V), dtype)
    fs = np.zeros((B, H, K, V), dtype)
    for b in range(B):
        runs = _runs(None if seg is None else np.asarray(seg)[b], T)
        for h in range(H):
            S = np.zeros((K, V), dtype) if S0 is None else np.array(S0[b, h], dtype=dtype)
            for ri, (s, e) in enumerate(runs):
                if ri > 0:
                    S = np.zeros((K, V), dtype)
                for c0 in range(s, e, C):
                    n = min(C, e - c0)
                    Qc = np.zeros((C, K), dtype); Kc = np.zeros((C, K), dtype)
                    Vc = np.zeros((C, V), dtype); gc = np.zeros((C, K), dtype)
                    bc = np.zeros(C, dtype)
                    Qc[:n] = q[b, c0:c0 + n, h]; Kc[:n] = k[b, c0:c0 + n, h]
                    Vc[:n] = v[b, c0:c0 + n, h]; gc[:n] = g[b, c0:c0 + n, h]
                    bc[:n] = beta[b, c0:c0 + n, h]
                    Gc = np.cumsum(gc, axis=0)
                    F = decay_factors(Gc, sub)
                    Akk, Aqk = intra_products(Qc, Kc, F, sub, rnd)
                    L = np.tril(bc[:, None] * Akk, -1)
                    Tm = np.linalg.inv(np.eye(C, dtype=dtype) + L)  # unit lower
                    blk = F["blk"]
                    Ktil = Kc * F["E1"] * F["pre"][blk]          # K * e^{G}
                    Qtil = Qc * F["E1"] * F["pre"][blk]          # Q * e^{G}
                    Khat = Kc * F["E2"] * F["suf"][blk]          # K * e^{G_C-G}
                    Tb = rnd(Tm)
                    u = Tb @ rnd(bc[:, None] * Vc)
                    w = Tb @ rnd(bc[:, None] * Ktil)
                    Sb = rnd(S)
                    U = u - rnd(w) @ Sb
                    Ub = rnd(U)
                    Oc = scale * (rnd(Qtil) @ Sb + rnd(np.tril(Aqk)) @ Ub)
                    S = F["gammaC"][:, None] * S + rnd(Khat).T @ Ub
                    o[b, c0:c0 + n, h] = Oc[:n]
            fs[b, h] = S
    return o, fs
