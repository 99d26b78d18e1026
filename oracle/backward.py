"""fp64 oracle for the backward pass of the gated delta rule -- TEST
INFRASTRUCTURE ONLY (same rules as the rest of ``oracle``).

Source: "Long-Context Aware Upcycling: A New Frontier for Hybrid LLM Scaling",
Appendix A.3, Eq. 16-19 (the recurrence), trained with the chunked kernel the
last paragraph of A.3 names.  The gradients are those of the recurrence
itself, so the oracle differentiates the token recurrence by hand, one token
at a time in reverse order, with nothing chunked:

forward (library orientation, S is dv x dk):
    S_t = alpha_t S_{t-1} + u_t k_t^T,   u_t = beta_t (v_t - alpha_t S_{t-1} k_t)
    o_t = S_t q_t / sqrt(dk)

reverse, with G = dL/dS_t accumulated from the end (G = dS_final, or 0):
    G     += dO_t q_t^T / sqrt(dk)                   (o_t reads S_t)
    dq_t   = S_t^T dO_t / sqrt(dk)
    dv_t   = beta_t G k_t
    dbeta_t = (v_t - alpha_t S_{t-1} k_t)^T G k_t
    dalpha_t = <G, S_{t-1}> - beta_t (S_{t-1} k_t)^T G k_t
    dk_t   = G^T u_t - alpha_t beta_t S_{t-1}^T G k_t
    G      = alpha_t G - alpha_t beta_t (G k_t) k_t^T  (dL/dS_{t-1}: G M_t^T, M_t symmetric)
and dS0 = G after the first token.

Each line is the derivative of one term of the forward line above it; the
tests pin them against central finite differences of the forward oracle and
against exact adjoint identities.  Inputs are widened exactly to fp64 like the
forward oracle's; layouts are the library's.
"""
from __future__ import annotations

import math

import numpy as np

from .layer_io import widen


def _bounds(T_total, cu_seqlens, B=None, T=None):
    if cu_seqlens is None:
        return [(n * T, (n + 1) * T) for n in range(B)]
    cu = [int(c) for c in np.asarray(widen(cu_seqlens)).astype(np.int64)]
    return list(zip(cu[:-1], cu[1:]))


def prefill_backward(q, k, v, alpha, beta, dout, S0=None, dS_final=None, cu_seqlens=None):
    """Gradients of L = <dout, out> + <dS_final, S_final> with respect to
    q, k, v, alpha, beta and S0, for the recurrence of Eq. 16-19 (Appendix
    A.3), differentiated token by token in reverse order (the lines of this
    module's header, each the derivative of one term of the forward line).

    q, k: [B, T, H, dk] or [T_total, H, dk]; v, dout likewise with dv;
    alpha, beta: [.., H]; S0, dS_final: [N, H, dv, dk] or None (zero).
    Returns dict dq, dk, dv [T_total, H, .], dalpha, dbeta [T_total, H],
    dS0 [N, H, dv, dk] (all fp64), plus out and S_final of the forward.
    """
    qa, ka, va, da = widen(q), widen(k), widen(v), widen(dout)
    H, dk = qa.shape[-2], qa.shape[-1]
    dv = va.shape[-1]
    if cu_seqlens is None:
        B, T = (qa.shape[0], qa.shape[1]) if qa.ndim == 4 else (1, qa.shape[0])
    else:
        B, T = None, None
    qa = qa.reshape(-1, H, dk)
    ka = ka.reshape(-1, H, dk)
    va = va.reshape(-1, H, dv)
    da = da.reshape(-1, H, dv)
    al = widen(alpha).reshape(-1, H)
    be = widen(beta).reshape(-1, H)
    T_total = qa.shape[0]
    bounds = _bounds(T_total, cu_seqlens, B, T)
    N = len(bounds)
    s = 1.0 / math.sqrt(dk)
    s0 = widen(S0) if S0 is not None else np.zeros((N, H, dv, dk))
    dsf = widen(dS_final) if dS_final is not None else np.zeros((N, H, dv, dk))
    res = dict(dq=np.zeros((T_total, H, dk)), dk=np.zeros((T_total, H, dk)),
               dv=np.zeros((T_total, H, dv)), dalpha=np.zeros((T_total, H)),
               dbeta=np.zeros((T_total, H)), dS0=np.zeros((N, H, dv, dk)),
               out=np.zeros((T_total, H, dv)), S_final=np.zeros((N, H, dv, dk)))
    for n, (a, b) in enumerate(bounds):
        for h in range(H):
            # forward, keeping every state S_{t-1} (small problems only)
            S = s0[n, h].copy()
            prev = []
            for t in range(a, b):
                kt, vt, at, bt = ka[t, h], va[t, h], al[t, h], be[t, h]
                prev.append(S.copy())
                u = bt * (vt - at * (S @ kt))
                S = at * S + np.outer(u, kt)
                res["out"][t, h] = s * (S @ qa[t, h])
            res["S_final"][n, h] = S
            # reverse
            G = dsf[n, h].copy()
            for i, t in enumerate(range(b - 1, a - 1, -1)):
                Sp = prev[len(prev) - 1 - i]
                kt, vt, qt, at, bt = ka[t, h], va[t, h], qa[t, h], al[t, h], be[t, h]
                dO = da[t, h]
                G += s * np.outer(dO, qt)
                res["dq"][t, h] = s * (S.T @ dO)
                kS = Sp @ kt
                Gk = G @ kt
                u = bt * (vt - at * kS)
                res["dv"][t, h] = bt * Gk
                res["dbeta"][t, h] = (vt - at * kS) @ Gk
                res["dalpha"][t, h] = np.sum(G * Sp) - bt * (kS @ Gk)
                res["dk"][t, h] = G.T @ u - at * bt * (Sp.T @ Gk)
                G = at * G - at * bt * np.outer(Gk, kt)
                S = Sp
            res["dS0"][n, h] = G
    return res
