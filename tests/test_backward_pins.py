"""Pins for the fp64 backward oracle (``oracle.backward``).

The gradients are checked against things outside the backward's own code:
  * central finite differences of the (separately pinned) C forward oracle,
    on dyadic inputs so that every perturbed value is exact in fp32, with
    Richardson extrapolation (error O(h^4));
  * exact adjoint identities: (out, S_final) is linear in (v, S0), so
    <dv, v> + <dS0, S0> = <dout, out> + <dS_final, S_final>; out is linear in
    q and S_final does not depend on it, so <dq, q> = <dout, out>;
  * closed forms at beta = 0 (pure decay);
  * packing invariance (a sequence's gradients do not depend on its batch).
A dropped term in any gradient line, a wrong sign, S_t used where S_{t-1} is
meant, or a missing decay in the carried G fails at least one of them.
"""
import math

import numpy as np
import pytest

import oracle
from oracle.backward import prefill_backward

rng = np.random.default_rng(2024)


def dyadic(shape, scale=1.0, lo=None, hi=None, bits=12):
    if lo is not None:
        x = rng.uniform(lo, hi, shape)
    else:
        x = rng.standard_normal(shape) * scale
    return (np.round(x * 2 ** bits) / 2 ** bits).astype(np.float32)


def case(lens, H=2, dk=3, dv=3):
    T = sum(lens)
    return dict(q=dyadic((T, H, dk)), k=dyadic((T, H, dk), 0.6), v=dyadic((T, H, dv)),
                alpha=dyadic((T, H), lo=0.3, hi=1.0), beta=dyadic((T, H), lo=0.1, hi=0.9),
                S0=dyadic((len(lens), H, dv, dk)), dout=dyadic((T, H, dv)),
                dS_final=dyadic((len(lens), H, dv, dk)),
                cu=np.concatenate([[0], np.cumsum(lens)]).astype(np.int32))


def loss(x):
    out, sf, _ = oracle.prefill(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["S0"], x["cu"])
    return float(np.sum(out * x["dout"].astype(np.float64))
                 + np.sum(sf * x["dS_final"].astype(np.float64)))


def fd(x, name, idx, h):
    def at(delta):
        y = dict(x)
        y[name] = x[name].copy()
        y[name][idx] = np.float32(np.float64(x[name][idx]) + delta)
        assert np.float64(y[name][idx]) == np.float64(x[name][idx]) + delta   # exact in fp32
        return loss(y)
    d1 = (at(h) - at(-h)) / (2 * h)
    d2 = (at(h / 2) - at(-h / 2)) / h
    return (4 * d2 - d1) / 3


@pytest.mark.parametrize("name,gname", [("q", "dq"), ("k", "dk"), ("v", "dv"),
                                        ("alpha", "dalpha"), ("beta", "dbeta"),
                                        ("S0", "dS0")])
def test_gradients_match_finite_differences(name, gname):
    x = case([4, 3])
    g = prefill_backward(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["dout"], x["S0"],
                         x["dS_final"], x["cu"])
    h = 2.0 ** -8
    worst = 0.0
    for idx in np.ndindex(x[name].shape):
        num = fd(x, name, idx, h)
        worst = max(worst, abs(num - g[gname][idx]))
    assert worst < 1e-7, worst


def _big(lens, H=2, dk=16, dv=24, seed=0):
    r = np.random.default_rng(seed)
    T = sum(lens)
    kk = r.standard_normal((T, H, dk))
    kk /= np.linalg.norm(kk, axis=-1, keepdims=True)
    return dict(q=r.standard_normal((T, H, dk)).astype(np.float32), k=kk.astype(np.float32),
                v=r.standard_normal((T, H, dv)).astype(np.float32),
                alpha=r.uniform(0.2, 1.0, (T, H)).astype(np.float32),
                beta=r.uniform(0.0, 1.0, (T, H)).astype(np.float32),
                S0=r.standard_normal((len(lens), H, dv, dk)).astype(np.float32),
                dout=r.standard_normal((T, H, dv)).astype(np.float32),
                dS_final=r.standard_normal((len(lens), H, dv, dk)).astype(np.float32),
                cu=np.concatenate([[0], np.cumsum(lens)]).astype(np.int32))


def test_adjoint_identities():
    x = _big([40, 1, 17])
    g = prefill_backward(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["dout"], x["S0"],
                         x["dS_final"], x["cu"])
    out, sf, _ = oracle.prefill(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["S0"], x["cu"])
    f64 = lambda a: np.asarray(a, np.float64)
    lhs_out = np.sum(f64(x["dout"]) * out)
    rhs = lhs_out + np.sum(f64(x["dS_final"]) * sf)
    lin = np.sum(g["dv"] * f64(x["v"])) + np.sum(g["dS0"] * f64(x["S0"]))
    assert abs(lin - rhs) <= 1e-11 * (abs(rhs) + 1)
    assert abs(np.sum(g["dq"] * f64(x["q"])) - lhs_out) <= 1e-11 * (abs(lhs_out) + 1)
    # the forward the backward recomputes is the forward oracle's
    assert np.max(np.abs(g["out"] - out)) < 1e-12 and np.max(np.abs(g["S_final"] - sf)) < 1e-12


def test_beta_zero_closed_forms():
    """beta = 0: S_t = gamma_t S0 with gamma_t = prod alpha, so
    dS0 = sum_t s gamma_t dO_t q_t^T + gamma_T dS_T, dv = dk = 0,
    dq_t = s gamma_t S0^T dO_t, and
    dalpha_t = (1/alpha_t) [sum_{t' >= t} s gamma_t' dO_t'.(S0 q_t') + gamma_T <dS_T, S0>]."""
    x = _big([9], H=1, dk=8, dv=5, seed=3)
    x["beta"][:] = 0
    g = prefill_backward(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["dout"], x["S0"],
                         x["dS_final"], x["cu"])
    f = lambda a: np.asarray(a, np.float64)
    al, q, dO, S0, dST = f(x["alpha"])[:, 0], f(x["q"])[:, 0], f(x["dout"])[:, 0], \
        f(x["S0"])[0, 0], f(x["dS_final"])[0, 0]
    s = 1 / math.sqrt(8)
    gam = np.cumprod(al)
    want_dS0 = sum(s * gam[t] * np.outer(dO[t], q[t]) for t in range(9)) + gam[-1] * dST
    np.testing.assert_allclose(g["dS0"][0, 0], want_dS0, rtol=1e-12, atol=1e-12)
    assert np.all(g["dv"] == 0) and np.all(g["dk"] == 0)
    for t in range(9):
        np.testing.assert_allclose(g["dq"][t, 0], s * gam[t] * S0.T @ dO[t], rtol=1e-12,
                                   atol=1e-12)
        tail = sum(s * gam[u] * dO[u] @ (S0 @ q[u]) for u in range(t, 9)) \
            + gam[-1] * np.sum(dST * S0)
        np.testing.assert_allclose(g["dalpha"][t, 0], tail / al[t], rtol=1e-11, atol=1e-12)


def test_packing_invariance_bitwise():
    lens = [5, 0, 7, 1]
    x = _big(lens, H=2, dk=4, dv=6, seed=5)
    g = prefill_backward(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["dout"], x["S0"],
                         x["dS_final"], x["cu"])
    cu = x["cu"]
    for n in range(len(lens)):
        sl = slice(cu[n], cu[n + 1])
        one = prefill_backward(x["q"][sl], x["k"][sl], x["v"][sl], x["alpha"][sl],
                               x["beta"][sl], x["dout"][sl], x["S0"][n:n + 1],
                               x["dS_final"][n:n + 1], np.array([0, lens[n]], np.int32))
        for key in ("dq", "dk", "dv", "dalpha", "dbeta"):
            assert np.array_equal(one[key], g[key][sl]), (n, key)
        assert np.array_equal(one["dS0"][0], g["dS0"][n])
