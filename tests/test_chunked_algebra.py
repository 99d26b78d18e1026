"""The chunked (WY / UT-transform) algebra the kernels implement agrees with
the token-by-token oracle to fp64 rounding, on ragged chunks and packed
sequences.  CPU only."""
import numpy as np
import pytest

import oracle
from chunked_model import chunked_prefill


@pytest.mark.parametrize("lens,C", [([200], 64), ([64, 1, 65, 127, 0, 3], 64), ([37, 80], 16)])
def test_chunked_form_matches_token_recurrence(lens, C):
    rng = np.random.default_rng(sum(lens) + C)
    T, H, dk, dv = sum(lens), 2, 16, 12
    q = rng.standard_normal((T, H, dk)).astype(np.float32)
    k = rng.standard_normal((T, H, dk))
    k = (k / np.linalg.norm(k, axis=-1, keepdims=True)).astype(np.float32)
    v = rng.standard_normal((T, H, dv)).astype(np.float32)
    alpha = np.exp(-np.logaddexp(0, rng.standard_normal((T, H)))).astype(np.float32)
    beta = (1 / (1 + np.exp(-rng.standard_normal((T, H))))).astype(np.float32)
    S0 = 0.5 * rng.standard_normal((len(lens), H, dv, dk))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    o_ref, s_ref, _ = oracle.prefill(q, k, v, alpha, beta, S0, cu_seqlens=cu)
    o, s = chunked_prefill(q, k, v, alpha, beta, S0, cu, C=C)
    assert np.abs(o - o_ref).max() <= 1e-12 * max(1.0, np.abs(o_ref).max())
    assert np.abs(s - s_ref).max() <= 1e-12 * max(1.0, np.abs(s_ref).max())


def test_chunked_backward_model_matches_backward_oracle():
    """The chunked backward the CUDA kernels implement (tests/chunked_backward_model.py)
    equals the token-by-token backward oracle on ragged, packed and empty
    sequences, chunk sizes 4, 8 and 64."""
    from chunked_backward_model import chunked_backward
    from oracle.backward import prefill_backward
    r = np.random.default_rng(11)
    for lens, C, dk, dv in [([10], 4, 6, 5), ([23, 1, 9, 0, 16], 8, 8, 8), ([130], 64, 16, 12)]:
        T, H = sum(lens), 2
        kk = r.standard_normal((T, H, dk))
        kk /= np.linalg.norm(kk, axis=-1, keepdims=True)
        x = dict(q=r.standard_normal((T, H, dk)), k=kk, v=r.standard_normal((T, H, dv)),
                 alpha=r.uniform(0.3, 1, (T, H)), beta=r.uniform(0, 1, (T, H)),
                 S0=r.standard_normal((len(lens), H, dv, dk)), dout=r.standard_normal((T, H, dv)),
                 dS=r.standard_normal((len(lens), H, dv, dk)))
        x = {k_: v_.astype(np.float32) for k_, v_ in x.items()}
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        o = prefill_backward(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["dout"], x["S0"],
                             x["dS"], cu)
        m = chunked_backward(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["dout"], x["S0"],
                             x["dS"], cu, C=C)
        for key in ("dq", "dk", "dv", "dalpha", "dbeta", "dS0"):
            assert np.max(np.abs(o[key] - m[key])) <= 1e-12 * np.max(np.abs(o[key])), (lens, key)


@pytest.mark.parametrize("T,P,C,dk,dv", [(300, 4, 16, 8, 8), (257, 5, 16, 8, 12), (96, 6, 16, 6, 6)])
def test_segment_scan_composes_to_the_full_chain(T, P, C, dk, dv):
    """The long-sequence prefill as a scan over segments: over a run of tokens
    the recurrence is affine in its start state, S_end = S_start A + B, with
    A = prod_t alpha_t (I - beta_t k_t k_t^T) (in token order, acting on the
    right of S) and B the end state from a zero start.  A pass from the start
    [I; 0] gives F = A + B on the first dk rows; composing the segments'
    (A, B) pairs reproduces the single chain's outputs and end state to fp64
    rounding.  Segments are whole chunks of C tokens, the last one ragged."""
    rng = np.random.default_rng(T * 7 + P)
    H = 2
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, dv))
    alpha = rng.uniform(0.9, 1.0, (T, H)).astype(np.float32)     # long memory: starts matter
    beta = rng.uniform(0.0, 1.0, (T, H)).astype(np.float32)
    q, k, v = (x.astype(np.float32) for x in (q, k, v))
    S0 = rng.standard_normal((1, H, dv, dk))
    o_ref, s_ref, _ = oracle.prefill(q, k, v, alpha, beta, S0,
                                     cu_seqlens=np.array([0, T], dtype=np.int64))
    seg = -(-(-(-T // C)) // P) * C                   # whole chunks per segment
    cu = np.array(sorted({min(j * seg, T) for j in range(P + 1)}), dtype=np.int64)
    n = len(cu) - 1
    assert n >= 2
    zero = np.zeros((n, H, dv, dk))
    start_b = zero.copy()
    start_b[0] = S0[0]
    ident = zero.copy()
    ident[:, :, :dk, :] = np.eye(dk)
    _, B, _ = oracle.prefill(q, k, v, alpha, beta, start_b, cu_seqlens=cu)
    _, F, _ = oracle.prefill(q, k, v, alpha, beta, ident, cu_seqlens=cu)
    # [segment, head, dk, dk]; for segment 0, whose B pass starts from S0, this
    # is (I - S0) A(0) instead, and the scan never uses it
    A = F[:, :, :dk, :] - B[:, :, :dk, :]
    # A is the product of the segment's per-token transitions (written out here)
    for j in range(1, n):
        for h in range(H):
            M = np.eye(dk)
            for t in range(cu[j], cu[j + 1]):
                kt = k[t, h].astype(np.float64)
                M = M @ (float(alpha[t, h]) * (np.eye(dk) - float(beta[t, h]) * np.outer(kt, kt)))
            assert np.abs(A[j, h] - M).max() <= 1e-12
    # the scan: every segment's true start from its predecessor's (A, B)
    starts = zero.copy()
    starts[0] = S0[0]
    starts[1] = B[0]
    for j in range(2, n):
        starts[j] = np.einsum("hij,hjk->hik", starts[j - 1], A[j - 1]) + B[j - 1]
    o, S_end, _ = oracle.prefill(q, k, v, alpha, beta, starts, cu_seqlens=cu)
    assert np.abs(o - o_ref).max() <= 1e-11 * np.abs(o_ref).max()
    assert np.abs(S_end[-1] - s_ref[0]).max() <= 1e-11 * np.abs(s_ref).max()
    # and the segment starts do matter on this input
    o_cut, _, _ = oracle.prefill(q, k, v, alpha, beta, start_b, cu_seqlens=cu)
    assert np.abs(o_cut - o_ref).max() > 1e-3 * np.abs(o_ref).max()
