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
