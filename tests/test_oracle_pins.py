"""Pins for the fp64 oracle against what the definition fixes exactly.

The oracle follows Eq. 16-19 of "Long-Context Aware Upcycling" (Appendix A.3)
in the paper's orientation; every check here comes from somewhere else: a
hand-worked example, closed forms, exact rational brute force of the
explicit-transition-matrix form S_t = alpha_t S_{t-1}(I - beta_t k_t k_t^T) +
beta_t v_t k_t^T, and invariants of the recurrence.  Each is chosen so that a
plausible slip in the oracle (dropped decay, wrong sign in Eq. 17, beta on the
wrong factor, output read from S_{t-1} instead of S_t, transposed state,
missing 1/sqrt(dk)) fails at least one of them.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng_master = np.random.default_rng(1234)


def _dense(T, H, dk, dv, rng, s0=True, dyadic=False):
    def draw(*shape):
        x = rng.standard_normal(shape)
        if dyadic:  # exactly representable in fp32 and closed under small sums
            x = np.round(x * 256) / 256
        return x.astype(np.float32)
    q, k, v = draw(T, H, dk), draw(T, H, dk), draw(T, H, dv)
    k = (k / np.linalg.norm(k, axis=-1, keepdims=True)).astype(np.float32) if not dyadic else k
    alpha = rng.uniform(0.05, 1.0, (T, H)).astype(np.float32)
    beta = rng.uniform(0.0, 1.0, (T, H)).astype(np.float32)
    S0 = rng.standard_normal((1, H, dv, dk)) if s0 else None
    return q, k, v, alpha, beta, S0


def test_hand_worked_example():
    """Three tokens worked by hand in exact fractions (tests/golden)."""
    g = json.load(open(os.path.join(GOLDEN, "hand_worked_2x2.json")))
    fr = lambda s: float(Fraction(s))
    toks = g["tokens"]
    T, dk, dv = len(toks), g["dk"], g["dv"]
    q = np.array([[[fr(x) for x in t["q"]]] for t in toks], np.float32)
    k = np.array([[[fr(x) for x in t["k"]]] for t in toks], np.float32)
    v = np.array([[[fr(x) for x in t["v"]]] for t in toks], np.float32)
    a = np.array([[fr(t["alpha"])] for t in toks], np.float32)
    b = np.array([[fr(t["beta"])] for t in toks], np.float32)
    S0 = np.array([[[[fr(x) for x in r] for r in g["S0"]]]])
    for t in range(1, T + 1):  # every prefix: S_t and o_t
        out, Sf, _ = oracle.prefill(q[:t], k[:t], v[:t], a[:t], b[:t], S0)
        want_S = np.array([[fr(x) for x in r] for r in toks[t - 1]["S"]])
        want_Sq = np.array([fr(x) for x in toks[t - 1]["Sq"]])
        assert np.array_equal(Sf[0, 0], want_S)
        np.testing.assert_allclose(out[t - 1, 0] * math.sqrt(dk), want_Sq, rtol=0, atol=1e-15)


def test_beta_zero_is_pure_decay():
    """beta = 0: S_t = (prod alpha) S0 and o_t = gamma_t S0 q_t / sqrt(dk)."""
    rng = np.random.default_rng(1)
    T, H, dk, dv = 40, 2, 16, 12
    q, k, v, alpha, beta, S0 = _dense(T, H, dk, dv, rng)
    beta[:] = 0
    out, Sf, _ = oracle.prefill(q, k, v, alpha, beta, S0)
    gamma = np.cumprod(alpha.astype(np.float64), axis=0)   # [T, H]
    for h in range(H):
        np.testing.assert_allclose(Sf[0, h], gamma[-1, h] * S0[0, h], rtol=1e-13, atol=0)
        want = gamma[:, h, None] * (q[:, h].astype(np.float64) @ S0[0, h].T) / math.sqrt(dk)
        np.testing.assert_allclose(out[:, h], want, rtol=1e-12, atol=1e-300)


def _hadamard(n):
    Hm = np.array([[1.0]])
    while Hm.shape[0] < n:
        Hm = np.block([[Hm, Hm], [Hm, -Hm]])
    return Hm


@pytest.mark.parametrize("dk", [16, 256])
def test_retrieval_with_orthonormal_keys(dk):
    """alpha = beta = 1 and orthonormal keys (normalised Hadamard rows, exact in
    fp32): every stored association is retrieved exactly, S_T k_j = v_j, and
    with q_t = k_t the output is v_t / sqrt(dk), whatever S0 was."""
    rng = np.random.default_rng(2)
    T, dv = min(dk, 24), 10
    perm = rng.permutation(dk)[:T]
    keys = (_hadamard(dk)[perm] / math.sqrt(dk)).astype(np.float32)  # entries +-2^-m
    k = keys[:, None, :]
    q = k.copy()
    v = rng.standard_normal((T, 1, dv)).astype(np.float32)
    ones = np.ones((T, 1), np.float32)
    S0 = rng.standard_normal((1, 1, dv, dk))
    out, Sf, _ = oracle.prefill(q, k, v, ones, ones, S0)
    retrieved = Sf[0, 0] @ keys.astype(np.float64).T          # [dv, T]
    np.testing.assert_allclose(retrieved.T, v[:, 0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(out[:, 0] * math.sqrt(dk), v[:, 0], rtol=0, atol=1e-12)


def test_single_token_closed_form():
    """T = 1 with explicit matrices: S_1 = alpha S0 (I - beta k k^T) + beta v k^T."""
    rng = np.random.default_rng(3)
    H, dk, dv = 3, 8, 6
    q, k, v, alpha, beta, S0 = _dense(1, H, dk, dv, rng)
    out, Sf, _ = oracle.prefill(q, k, v, alpha, beta, S0)
    for h in range(H):
        kk = k[0, h].astype(np.float64)
        a, b = float(alpha[0, h]), float(beta[0, h])
        S1 = a * S0[0, h] @ (np.eye(dk) - b * np.outer(kk, kk)) + b * np.outer(v[0, h], kk)
        np.testing.assert_allclose(Sf[0, h], S1, rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(out[0, h], S1 @ q[0, h].astype(np.float64) / math.sqrt(dk),
                                   rtol=1e-12, atol=1e-15)


def _frac_mat(x):
    return [[Fraction(float(e)) for e in row] for row in x]


def _mm(A, B):
    return [[sum(A[i][t] * B[t][j] for t in range(len(B))) for j in range(len(B[0]))]
            for i in range(len(A))]


@pytest.mark.parametrize("dk,dv,T", [(2, 3, 6), (3, 2, 5), (4, 4, 6)])
def test_bruteforce_transition_product_exact(dk, dv, T):
    """Exact rational brute force on tiny sizes of the composed form
    S_T = S0 M_1...M_T + sum_j beta_j v_j k_j^T M_{j+1}...M_T,
    M_t = alpha_t (I - beta_t k_t k_t^T), and o_t = S_t q_t / sqrt(dk), with
    dyadic inputs so every input is exact in fp32."""
    rng = np.random.default_rng(10 + dk)
    d = lambda *s: (np.round(rng.standard_normal(s) * 8) / 8).astype(np.float32)
    q, k, v = d(T, 1, dk), d(T, 1, dk), d(T, 1, dv)
    alpha = (rng.integers(1, 9, (T, 1)) / 8).astype(np.float32)
    beta = (rng.integers(0, 9, (T, 1)) / 8).astype(np.float32)
    S0 = np.round(rng.standard_normal((1, 1, dv, dk)) * 16) / 16
    out, Sf, _ = oracle.prefill(q, k, v, alpha, beta, S0)
    I = [[Fraction(int(i == j)) for j in range(dk)] for i in range(dk)]
    M = []
    for t in range(T):
        kt = [Fraction(float(x)) for x in k[t, 0]]
        a, b = Fraction(float(alpha[t, 0])), Fraction(float(beta[t, 0]))
        M.append([[a * (I[i][j] - b * kt[i] * kt[j]) for j in range(dk)] for i in range(dk)])
    S0f = _frac_mat(S0[0, 0])
    for t in range(1, T + 1):   # S_t from scratch for every prefix
        St = S0f
        for s in range(t):
            St = _mm(St, M[s])
        for j in range(t):
            kj = [Fraction(float(x)) for x in k[j, 0]]
            bj = Fraction(float(beta[j, 0]))
            term = [[bj * Fraction(float(v[j, 0, r])) * kj[c] for c in range(dk)] for r in range(dv)]
            for s in range(j + 1, t):
                term = _mm(term, M[s])
            St = [[St[r][c] + term[r][c] for c in range(dk)] for r in range(dv)]
        Sq = [sum(St[r][c] * Fraction(float(q[t - 1, 0, c])) for c in range(dk)) for r in range(dv)]
        want_o = np.array([float(x) for x in Sq]) / math.sqrt(dk)
        np.testing.assert_allclose(out[t - 1, 0], want_o, rtol=1e-12, atol=1e-13)
        if t == T:
            want_S = np.array([[float(x) for x in row] for row in St])
            np.testing.assert_allclose(Sf[0, 0], want_S, rtol=1e-12, atol=1e-13)


def test_linearity_in_values_and_initial_state():
    """For fixed q, k, alpha, beta the map (V, S0) -> (O, S_T) is linear."""
    rng = np.random.default_rng(4)
    T, H, dk, dv = 30, 2, 8, 8
    q, k, v1, alpha, beta, S1 = _dense(T, H, dk, dv, rng, dyadic=True)
    v2 = (np.round(rng.standard_normal(v1.shape) * 256) / 256).astype(np.float32)
    S2 = rng.standard_normal(S1.shape)
    v12 = (2 * v1.astype(np.float64) - 3 * v2).astype(np.float32)   # exact in fp32
    assert np.array_equal(v12.astype(np.float64), 2 * v1.astype(np.float64) - 3 * v2)
    o1, f1, _ = oracle.prefill(q, k, v1, alpha, beta, S1)
    o2, f2, _ = oracle.prefill(q, k, v2, alpha, beta, S2)
    o12, f12, _ = oracle.prefill(q, k, v12, alpha, beta, 2 * S1 - 3 * S2)
    np.testing.assert_allclose(o12, 2 * o1 - 3 * o2, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(f12, 2 * f1 - 3 * f2, rtol=1e-11, atol=1e-12)


def test_non_expansion_without_writes():
    """v = 0, |k| = 1, beta in [0, 1], alpha <= 1: I - beta k k^T has
    eigenvalues 1 - beta and 1, so the state norm never grows."""
    rng = np.random.default_rng(5)
    T, H, dk, dv = 25, 2, 12, 7
    q, k, v, alpha, beta, S0 = _dense(T, H, dk, dv, rng)
    v[:] = 0
    S = S0.copy()
    prev = np.linalg.norm(S, axis=(-2, -1))
    for t in range(T):
        _ = oracle.decode_step(q[t][None], k[t][None], v[t][None], alpha[t][None],
                               beta[t][None], S)
        now = np.linalg.norm(S, axis=(-2, -1))
        assert np.all(now <= prev * (1 + 1e-13))
        prev = now
    # and the decay is not the identity: with alpha < 1 the norm strictly drops
    assert np.all(prev < np.linalg.norm(S0, axis=(-2, -1)))


def test_split_resume_is_bitwise():
    """Oracle on T1 then T2 from S_final equals the oracle on T1 + T2."""
    rng = np.random.default_rng(6)
    T, H, dk, dv = 50, 2, 8, 6
    q, k, v, alpha, beta, S0 = _dense(T, H, dk, dv, rng)
    o, Sf, _ = oracle.prefill(q, k, v, alpha, beta, S0)
    o1, S1, _ = oracle.prefill(q[:17], k[:17], v[:17], alpha[:17], beta[:17], S0)
    o2, S2, _ = oracle.prefill(q[17:], k[17:], v[17:], alpha[17:], beta[17:], S1)
    assert np.array_equal(np.concatenate([o1, o2]), o) and np.array_equal(S2, Sf)


def test_varlen_equals_separate_runs():
    """Packing through cu_seqlens changes nothing: each sequence is an
    independent recurrence from its own S0 (including an empty one)."""
    rng = np.random.default_rng(7)
    lens = [5, 0, 13, 1]
    T, H, dk, dv = sum(lens), 2, 8, 4
    q, k, v, alpha, beta, _ = _dense(T, H, dk, dv, rng)
    S0 = rng.standard_normal((len(lens), H, dv, dk))
    cu = np.concatenate([[0], np.cumsum(lens)])
    o, Sf, _ = oracle.prefill(q, k, v, alpha, beta, S0, cu_seqlens=cu)
    for n in range(len(lens)):
        a, b = cu[n], cu[n + 1]
        on, sn, _ = oracle.prefill(q[a:b], k[a:b], v[a:b], alpha[a:b], beta[a:b], S0[n:n + 1])
        assert np.array_equal(o[a:b], on) and np.array_equal(Sf[n], sn[0])
    assert np.array_equal(Sf[1], S0[1])   # empty sequence: S_final = S0


def test_decode_step_equals_single_token_prefill():
    rng = np.random.default_rng(8)
    N, H, dk, dv = 3, 2, 8, 5
    q, k, v, alpha, beta, _ = _dense(N, H, dk, dv, rng)
    S = rng.standard_normal((N, H, dv, dk))
    cu = np.arange(N + 1)
    o_p, S_p, _ = oracle.prefill(q, k, v, alpha, beta, S, cu_seqlens=cu)
    S_d = S.copy()
    o_d = oracle.decode_step(q, k, v, alpha, beta, S_d)
    assert np.array_equal(o_d, o_p) and np.array_equal(S_d, S_p)


def test_bf16_inputs_widen_exactly():
    """bf16 inputs are read as the exact values the GPU reads."""
    import torch
    rng = np.random.default_rng(9)
    T, H, dk, dv = 9, 1, 8, 4
    q, k, v, alpha, beta, S0 = _dense(T, H, dk, dv, rng)
    qb, kb, vb = (torch.from_numpy(x).to(torch.bfloat16) for x in (q, k, v))
    o_b, s_b, _ = oracle.prefill(qb, kb, vb, alpha, beta, S0)
    o_f, s_f, _ = oracle.prefill(qb.float(), kb.float(), vb.float(), alpha, beta, S0)
    assert np.array_equal(o_b, o_f) and np.array_equal(s_b, s_f)


def test_threads_do_not_change_results():
    rng = np.random.default_rng(11)
    T, H, dk, dv = 20, 4, 8, 8
    q, k, v, alpha, beta, S0 = _dense(T, H, dk, dv, rng)
    o1, s1, used1 = oracle.prefill(q, k, v, alpha, beta, S0, nthreads=1)
    o4, s4, used4 = oracle.prefill(q, k, v, alpha, beta, S0, nthreads=4)
    assert used1 == 1 and np.array_equal(o1, o4) and np.array_equal(s1, s4)


def test_pages_geometry():
    """The head geometry the library targets is the pages' (Table 8 / card)."""
    g = json.load(open(os.path.join(GOLDEN, "table8_geometry.json")))
    d = g["hidden_size_d"]
    assert g["key_dim_dk_total"] == math.floor(0.75 * d)
    assert g["key_dim_dk_total"] // g["heads_H"] == g["head_dim_dh"] == 256
    assert round(g["key_dim_dk_total"] * d / 1e6, 2) == g["W_QK_params_millions_printed"]
    assert round(g["value_expansion"] * g["key_dim_dk_total"] * d / 1e6, 2) == \
        g["W_VGO_params_millions_printed"]
    assert g["model_card_gdn_head_dim"] == g["head_dim_dh"]
    assert g["chunk_size_C"] == 64
