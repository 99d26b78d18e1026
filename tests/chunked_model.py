"""fp64 numpy model of the chunkwise-parallel (WY / UT transform) form of the
gated delta rule -- a test-side design aid, NOT the oracle and not used by
the GPU library.  It checks, against the token-by-token oracle, the chunk
algebra the CUDA kernels implement.

Chunked form (derived from the recurrence; the pages name it only as chunks
of C = 64 whose delta corrections are batched through the WY
representation, with the state carried sequentially across chunks --
Appendix A.3 of "Long-Context Aware Upcycling").  With the chunk's start
state S (dv x dk), G = cumsum(log alpha), gamma = exp(G),
Gam[r, j] = exp(G_r - G_j):
  A  = strict_lower(beta_r * Gam * K K^T),   T = (I + A)^{-1}
  W  = T diag(beta * gamma) K,               U~ = T diag(beta) V
  U  = U~ - W S^T
  O  = (diag(gamma) Q S^T + lower(Gam * Q K^T) U) / sqrt(dk)
  S' = gamma_L S + U^T diag(gamma_L / gamma) K
"""
import numpy as np


def chunked_prefill(q, k, v, alpha, beta, S0, cu, C=64):
    q, k, v = (np.asarray(x, np.float64) for x in (q, k, v))
    alpha, beta = np.asarray(alpha, np.float64), np.asarray(beta, np.float64)
    Ttot, H, dk = q.shape
    dv = v.shape[-1]
    N = len(cu) - 1
    out = np.zeros((Ttot, H, dv))
    Sf = np.zeros((N, H, dv, dk))
    for n in range(N):
        for h in range(H):
            S = np.zeros((dv, dk)) if S0 is None else np.array(S0[n, h], np.float64)
            for t0 in range(cu[n], cu[n + 1], C):
                t1 = min(t0 + C, cu[n + 1])
                Q, K, V = q[t0:t1, h], k[t0:t1, h], v[t0:t1, h]
                b = beta[t0:t1, h]
                G = np.cumsum(np.log(alpha[t0:t1, h]))
                g = np.exp(G)
                Gam = np.exp(G[:, None] - G[None, :])
                L = t1 - t0
                A = np.tril(b[:, None] * Gam * (K @ K.T), -1)
                Tm = np.linalg.inv(np.eye(L) + A)
                W = Tm @ ((b * g)[:, None] * K)
                Ut = Tm @ (b[:, None] * V)
                U = Ut - W @ S.T
                P = np.tril(Gam * (Q @ K.T))
                out[t0:t1, h] = (g[:, None] * (Q @ S.T) + P @ U) / np.sqrt(dk)
                S = g[-1] * S + U.T @ (np.exp(G[-1] - G)[:, None] * K)
            Sf[n, h] = S
    return out, Sf
