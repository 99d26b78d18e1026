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
