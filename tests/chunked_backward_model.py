"""fp64 numpy model of the backward pass of the chunked (WY) form -- a
test-side design aid for the CUDA backward, NOT the oracle.  It is checked
against the token-by-token backward oracle (``oracle.backward``).

Per chunk (rows r, j < L), with start state S, G = cumsum(log alpha),
gamma = e^G, Gam[r, j] = e^{G_r - G_j}, d_r = e^{G_L - G_r}, s = 1/sqrt(dk):
  forward:  A = strict_lower(beta_r Gam KK^T), T = (I + A)^-1,
            W = T diag(beta gamma) K, U~ = T diag(beta) V, U = U~ - W S^T,
            Qh = s diag(gamma) Q, Ph = s lower(Gam QK^T),
            O = Qh S^T + Ph U,   S' = gamma_L S + U^T diag(d) K
  reverse, given dO and dS' (gradient of the chunk's end state):
     dU  = Ph^T dO + diag(d) K dS'^T
     dS  = gamma_L dS' + dO^T Qh - dU^T W             (to the previous chunk)
     dQh = dO S,  dPh = lower(dO U^T),  dW = -dU S,  dU~ = dU
     dK  = diag(d) U dS'          dd_r = u_r . (dS' k_r)       dgamma_L = <dS', S>
  and then through W, U~, T, A, Ph, Qh and the decays down to log alpha.
"""
import numpy as np


def _chunks(a, b, C):
    return [(t0, min(t0 + C, b)) for t0 in range(a, b, C)]


def chunk_forward_factors(Q, K, V, al, be, s):
    L = len(al)
    G = np.cumsum(np.log(al))
    g = np.exp(G)
    Gam = np.exp(np.minimum(G[:, None] - G[None, :], 0.0))
    KK = K @ K.T
    QK = Q @ K.T
    A = np.tril(be[:, None] * Gam * KK, -1)
    Tm = np.linalg.inv(np.eye(L) + A)
    Bw = (be * g)[:, None] * K
    Bu = be[:, None] * V
    return dict(G=G, g=g, Gam=Gam, KK=KK, QK=QK, Tm=Tm, Bw=Bw, Bu=Bu, W=Tm @ Bw, Ut=Tm @ Bu,
                Qh=s * g[:, None] * Q, Ph=s * np.tril(Gam * QK), d=np.exp(G[-1] - G))


def chunk_backward(f, Q, K, V, al, be, S, dO, dSp, s):
    """Local gradients of one chunk.  Returns (dS_start, dQ, dK, dV, dalpha, dbeta)."""
    U = f["Ut"] - f["W"] @ S.T
    d, g, Gam, Tm = f["d"], f["g"], f["Gam"], f["Tm"]
    dU = f["Ph"].T @ dO + (d[:, None] * K) @ dSp.T
    dS = g[-1] * dSp + dO.T @ f["Qh"] - dU.T @ f["W"]
    dQh = dO @ S
    dPh = np.tril(dO @ U.T)
    dW = -dU @ S
    dK = d[:, None] * (U @ dSp)
    dd = np.sum(U * (K @ dSp.T), axis=1)
    dgL = np.sum(dSp * S)
    # W = T Bw, U~ = T Bu
    dTm = dW @ f["Bw"].T + dU @ f["Bu"].T
    TdW = Tm.T @ dW
    TdU = Tm.T @ dU
    dK += (be * g)[:, None] * TdW
    kTdW = np.sum(K * TdW, axis=1)
    dbeta = g * kTdW + np.sum(V * TdU, axis=1)
    dgam = be * kTdW
    dV = be[:, None] * TdU
    # T = (I + A)^-1, A strictly lower
    dA = np.tril(-(Tm.T @ dTm @ Tm.T), -1)
    dbeta += np.sum(dA * Gam * f["KK"], axis=1)
    M = dA * Gam * be[:, None]
    dK += M @ K + M.T @ K
    dGam = dA * be[:, None] * f["KK"]
    # Ph = s lower(Gam QK^T)
    FG = dPh * Gam
    dQ = s * FG @ K
    dK += s * FG.T @ Q
    dGam += s * dPh * f["QK"]
    # Qh = s diag(gamma) Q
    dQ += s * g[:, None] * dQh
    dgam += s * np.sum(Q * dQh, axis=1)
    # decays: gamma_r = e^{G_r}; Gam_rj = e^{G_r - G_j}; d_r = e^{G_L - G_r}; gamma_L S
    dG = g * dgam
    X = dGam * Gam
    dG += X.sum(axis=1) - X.sum(axis=0)
    dG -= d * dd
    dG[-1] += np.sum(d * dd) + g[-1] * dgL
    dlog = np.cumsum(dG[::-1])[::-1]           # G = cumsum(log alpha)
    return dS, dQ, dK, dV, dlog / al, dbeta


def chunked_backward(q, k, v, alpha, beta, dout, S0, dSf, cu, C=64):
    q, k, v, dout = (np.asarray(x, np.float64) for x in (q, k, v, dout))
    alpha, beta = np.asarray(alpha, np.float64), np.asarray(beta, np.float64)
    Ttot, H, dk = q.shape
    dv = v.shape[-1]
    N = len(cu) - 1
    s = 1.0 / np.sqrt(dk)
    res = dict(dq=np.zeros((Ttot, H, dk)), dk=np.zeros((Ttot, H, dk)),
               dv=np.zeros((Ttot, H, dv)), dalpha=np.zeros((Ttot, H)),
               dbeta=np.zeros((Ttot, H)), dS0=np.zeros((N, H, dv, dk)))
    for n in range(N):
        for h in range(H):
            chunks = _chunks(cu[n], cu[n + 1], C)
            S = np.zeros((dv, dk)) if S0 is None else np.array(S0[n, h], np.float64)
            starts, facs = [], []
            for t0, t1 in chunks:       # forward: chunk-start states
                f = chunk_forward_factors(q[t0:t1, h], k[t0:t1, h], v[t0:t1, h],
                                          alpha[t0:t1, h], beta[t0:t1, h], s)
                starts.append(S)
                facs.append(f)
                U = f["Ut"] - f["W"] @ S.T
                S = f["g"][-1] * S + U.T @ (f["d"][:, None] * k[t0:t1, h])
            dS = np.zeros((dv, dk)) if dSf is None else np.array(dSf[n, h], np.float64)
            for c in range(len(chunks) - 1, -1, -1):
                t0, t1 = chunks[c]
                dS, dQ, dK, dV, dA_, dB_ = chunk_backward(
                    facs[c], q[t0:t1, h], k[t0:t1, h], v[t0:t1, h], alpha[t0:t1, h],
                    beta[t0:t1, h], starts[c], dout[t0:t1, h], dS, s)
                res["dq"][t0:t1, h] = dQ
                res["dk"][t0:t1, h] = dK
                res["dv"][t0:t1, h] = dV
                res["dalpha"][t0:t1, h] = dA_
                res["dbeta"][t0:t1, h] = dB_
            res["dS0"][n, h] = dS
    return res
