"""Pins for the fp64 oracle of the layer's pre- and post-recurrence steps
(short convolution + SiLU, q/k L2 normalisation, decay and write-strength
gates; gated RMSNorm of the read-out), "Long-Context Aware Upcycling",
Appendix A.3 (Table 8's paragraph and Eq. 20).

Each check comes from outside the oracle's own formulas: library routines
(numpy.convolve, torch's normalize / rms_norm / silu), exact closed forms at
special inputs, identities (silu(z) - silu(-z) = z), and split / segment
invariants.  A dropped tap, a reversed kernel, a wrong history order, a head
index mix-up or a missing epsilon fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import layer_io as lio

rng = np.random.default_rng(4321)


def _rand(*shape):
    return rng.standard_normal(shape).astype(np.float32)


def test_conv_matches_numpy_convolve_and_silu_identity():
    """y(w) - y(-w) = the pre-activation (silu(z) - silu(-z) = z), and the
    pre-activation is numpy's full convolution with the reversed kernel."""
    T, C = 37, 5
    x, w = _rand(T, C), _rand(C, 4)
    y_pos, _ = lio.short_conv_silu(x, w)
    y_neg, _ = lio.short_conv_silu(x, -w)
    for c in range(C):
        want = np.convolve(x[:, c].astype(np.float64), w[c, ::-1].astype(np.float64))[:T]
        np.testing.assert_allclose(y_pos[:, c] - y_neg[:, c], want, rtol=1e-13, atol=1e-13)


def test_silu_special_values():
    assert lio.silu(np.float64(0.0)) == 0.0
    assert abs(lio.silu(np.float64(40.0)) - 40.0) < 1e-15 * 40 + 40 * math.exp(-40)
    z = np.linspace(-5, 5, 11)
    np.testing.assert_allclose(lio.silu(z), F.silu(torch.tensor(z)).numpy(), rtol=1e-15,
                               atol=1e-15)


def test_conv_history_order_and_taps():
    """Tap j multiplies x[t - 3 + j]; the history is the three previous inputs,
    oldest first: with a one-hot kernel the pre-activation reads them back."""
    N, C = 2, 3
    hist = _rand(N, 3, C)
    x = _rand(8, C)
    cu = np.array([0, 5, 8])
    for j in range(4):
        w = np.zeros((C, 4), np.float32)
        w[:, j] = 1.0
        yp, _ = lio.short_conv_silu(x, w, cu, hist)
        yn, _ = lio.short_conv_silu(x, -w, cu, hist)
        pre = yp - yn
        for n, (a, b) in enumerate([(0, 5), (5, 8)]):
            ext = np.concatenate([hist[n], x[a:b]])          # oldest first
            for t in range(b - a):
                np.testing.assert_allclose(pre[a + t], ext[t + j].astype(np.float64),
                                           rtol=1e-14, atol=1e-15)


def test_conv_split_resume_and_segmentation_exact():
    """Running T1 then T2 with the carried state equals T1 + T2 in one go, and a
    packed batch equals its sequences run alone (fp64, bit for bit)."""
    C = 6
    x, w, h0 = _rand(50, C), _rand(C, 4), _rand(1, 3, C)
    full, fs = lio.short_conv_silu(x, w, None, h0)
    for cut in (0, 1, 2, 3, 17, 50):
        a, sa = lio.short_conv_silu(x[:cut], w, None, h0)
        b, sb = lio.short_conv_silu(x[cut:], w, None, sa)
        assert np.array_equal(np.concatenate([a, b]), full) and np.array_equal(sb, fs)
    lens = [7, 0, 1, 2, 30]
    cu = np.concatenate([[0], np.cumsum(lens)])
    X = _rand(int(cu[-1]), C)
    H0 = _rand(len(lens), 3, C)
    packed, pst = lio.short_conv_silu(X, w, cu, H0)
    for n, L in enumerate(lens):
        alone, st = lio.short_conv_silu(X[cu[n]:cu[n + 1]], w, None, H0[n:n + 1])
        assert np.array_equal(packed[cu[n]:cu[n + 1]], alone) and np.array_equal(pst[n], st[0])
    assert np.array_equal(pst[1], H0[1].astype(np.float64))     # empty: state passes through


def test_l2_normalize_matches_torch_and_eps():
    x = rng.standard_normal((9, 4, 256))
    np.testing.assert_allclose(lio.l2_normalize(x, eps=0.0),
                               F.normalize(torch.tensor(x), dim=-1).numpy(), rtol=1e-14, atol=0)
    # eps enters under the root: a vector of norm 1e-3 keeps norm 1e-3/sqrt(1e-6 + 1e-6)
    tiny = np.zeros(256)
    tiny[3] = 1e-3
    assert abs(np.linalg.norm(lio.l2_normalize(tiny)) - 1e-3 / math.sqrt(2e-6)) < 1e-12


def test_gates_closed_forms_per_head():
    """softplus(0) = ln 2, so with a_raw + dt_bias = 0 the decay is
    2^(-exp(A_log)): A_log = ln m gives alpha = 2^-m exactly; sigmoid(ln 3) = 3/4."""
    H = 4
    A_log = np.log(np.array([1.0, 2.0, 3.0, 4.0])).astype(np.float32)
    dt_bias = np.array([0.5, -1.0, 2.0, 0.0], np.float32)
    a_raw = np.tile(-dt_bias, (3, 1))
    b_raw = np.tile(np.log(np.array([3.0, 1.0, 1 / 3, 1e9])), (3, 1)).astype(np.float32)
    alpha, beta = lio.gates(a_raw, b_raw, A_log, dt_bias)
    m = np.exp(A_log.astype(np.float64))
    np.testing.assert_allclose(alpha, np.tile(2.0 ** -m, (3, 1)), rtol=1e-14)
    np.testing.assert_allclose(beta[0], [0.75, 0.5, 0.25, 1.0], rtol=1e-7)
    # far below the bias the decay tends to 1; far above, alpha ~ exp(-exp(A_log)(a + dt))
    alpha2, _ = lio.gates(np.full((1, H), -60.0), b_raw[:1], A_log, np.zeros(H))
    assert np.all(np.abs(alpha2 - 1.0) < 1e-20 + 5 * np.exp(-60.0))
    alpha3, _ = lio.gates(np.full((1, H), 30.0), b_raw[:1], np.zeros(H), np.zeros(H))
    np.testing.assert_allclose(alpha3, math.exp(-30.0), rtol=1e-12)


def test_prepare_splits_channels_and_normalises():
    """q | k | v channel blocks land in the right outputs; q, k rows have unit
    norm up to eps; v is the plain conv + SiLU output."""
    H, dk, dv, T = 2, 4, 8, 5
    C = H * (2 * dk + dv)
    x, w = _rand(T, C), _rand(C, 4)
    r = lio.prepare(x, w, _rand(T, H), _rand(T, H), _rand(H), _rand(H), H, dk, dv)
    yp, _ = lio.short_conv_silu(x, w)
    np.testing.assert_array_equal(r["v"].reshape(T, -1), yp[:, 2 * H * dk:])
    for name, off in (("q", 0), ("k", H * dk)):
        raw = yp[:, off:off + H * dk].reshape(T, H, dk)
        cos = np.sum(r[name] * raw, -1) / np.linalg.norm(raw, axis=-1)
        np.testing.assert_allclose(cos, np.linalg.norm(r[name], axis=-1), rtol=1e-12)
        assert np.all(np.abs(np.linalg.norm(r[name], axis=-1) - 1) < 1e-5)


def test_decode_steps_equal_prefill():
    H, dk, dv, N, steps = 2, 4, 8, 3, 6
    C = H * (2 * dk + dv)
    w, A_log, dtb = _rand(C, 4), _rand(H), _rand(H)
    x, a, b = _rand(steps, N, C), _rand(steps, N, H), _rand(steps, N, H)
    h0 = _rand(N, 3, C)
    st = h0.astype(np.float64).copy()
    outs = [lio.prepare_decode_step(x[t], w, a[t], b[t], A_log, dtb, st, H, dk, dv)
            for t in range(steps)]
    # the same tokens as N sequences of length `steps`, packed
    xp = x.transpose(1, 0, 2).reshape(N * steps, C)
    ap = a.transpose(1, 0, 2).reshape(N * steps, H)
    bp = b.transpose(1, 0, 2).reshape(N * steps, H)
    cu = np.arange(N + 1) * steps
    r = lio.prepare(xp, w, ap, bp, A_log, dtb, H, dk, dv, cu, h0)
    for name in ("q", "k", "v", "alpha", "beta"):
        dec = np.stack([o[name] for o in outs], axis=1).reshape(r[name].shape)
        assert np.array_equal(dec, r[name]), name
    assert np.array_equal(st, r["conv_state"])


def test_output_norm_gate_matches_torch_rms_norm():
    dv = 256
    o = rng.standard_normal((7, 3, dv))
    g = rng.standard_normal((7, 3, dv))
    w = rng.standard_normal(dv)
    eps = 1e-5
    ref = F.rms_norm(torch.tensor(o), (dv,), weight=torch.tensor(w), eps=eps).numpy()
    np.testing.assert_allclose(lio.output_norm_gate(o, g, w, eps, "silu"),
                               ref * F.silu(torch.tensor(g)).numpy(), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lio.output_norm_gate(o, g, w, eps, "sigmoid"),
                               ref * torch.sigmoid(torch.tensor(g)).numpy(), rtol=1e-12,
                               atol=1e-13)


def test_output_norm_gate_invariants():
    """eps = 0: scale invariance in o, and unit RMS when w = 1 and the gate is
    saturated (sigmoid(50) = 1 to fp64); eps > 0 shrinks small rows."""
    dv = 512
    o = rng.standard_normal((4, dv))
    ones = np.ones(dv)
    big = np.full((4, dv), 50.0)
    y = lio.output_norm_gate(o, big, ones, 0.0, "sigmoid")
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, -1)), 1.0, rtol=1e-14)
    np.testing.assert_allclose(lio.output_norm_gate(1e-3 * o, big, ones, 0.0, "sigmoid"), y,
                               rtol=1e-12)
    small = lio.output_norm_gate(1e-3 * o, big, ones, 1e-6, "sigmoid")
    ms = np.mean((1e-3 * o) ** 2, -1)
    np.testing.assert_allclose(np.sqrt(np.mean(small * small, -1)), np.sqrt(ms / (ms + 1e-6)),
                               rtol=1e-12)


def test_bf16_inputs_widen_exactly():
    x = torch.randn(64, dtype=torch.float32).to(torch.bfloat16)
    assert np.array_equal(lio.widen(x), x.float().double().numpy())
