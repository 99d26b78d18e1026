"""Full-size checks of the rows beyond the core path, in the launch
configurations the benchmark times.

* gdn_prefill_backward on the 8K workload (B=4, T=8192, H=6, d=256, bf16):
  the token oracle cannot hold 8192 states a head, so the check uses the
  exact adjoint identities of the recurrence, which hold at any size --
  (out, S_final) is linear in (v, S0), so <dv, v> + <dS0, S0> = <dout, out> +
  <dS_final, S_final>; out is linear in q and S_final does not depend on it,
  so <dq, q> = <dout, out> -- evaluated in fp64 on the GPU's own forward and
  backward results (bf16 rounding of dq, dv bounds the error well inside 2e-2).
* gdn_decode_layer_step on 256 sequences x 6 heads against the oracle's
  prepare, token recurrence and gated RMSNorm, one step.
"""
import numpy as np
import pytest
import torch

import gdn_inputs
import oracle
from oracle import layer_io as lio

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _dot(a, b):
    return float((a.double() * b.double()).sum())


def test_backward_adjoint_identities_at_8k(gdn_lib):
    case = gdn_inputs.prefill_8k()
    x = gdn_inputs.make_prefill(case, device=DEV)
    g = torch.Generator(device=DEV)
    g.manual_seed(101)
    dout = torch.randn(x["v"].shape, generator=g, device=DEV).to(x["v"].dtype)
    dsf = torch.randn(x["S0"].shape, generator=g, device=DEV) * 0.1
    out, sf = gdn_lib.prefill(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["S0"])
    gr = gdn_lib.prefill_backward(x["q"], x["k"], x["v"], x["alpha"], x["beta"], dout, x["S0"],
                                  dsf)
    assert gdn_lib.device_status() == 0
    lhs_out = _dot(dout, out)
    rhs = lhs_out + _dot(dsf, sf)
    lin = _dot(gr["dv"], x["v"]) + _dot(gr["dS0"], x["S0"])
    scale = abs(lhs_out) + abs(_dot(dsf, sf))
    assert abs(lin - rhs) <= 2e-2 * scale, (lin, rhs)
    assert abs(_dot(gr["dq"], x["q"]) - lhs_out) <= 2e-2 * abs(lhs_out), (_dot(gr["dq"], x["q"]), lhs_out)
    for k in ("dq", "dk", "dv", "dalpha", "dbeta", "dS0"):
        assert torch.isfinite(gr[k].float()).all(), k


def test_decode_layer_step_at_full_size(gdn_lib):
    lc = gdn_inputs.layer_decode_256()
    x = gdn_inputs.make_layer(lc, device="cpu")
    N, H, dv = len(lc.lengths), lc.H, lc.dv
    gen = torch.Generator().manual_seed(102)
    S0 = torch.randn((N, H, dv, 256), generator=gen) * 0.02
    st, S = x["conv_state"].clone().to(DEV), S0.clone().to(DEV)
    gate = x["g"].reshape(N, H, dv)
    y = gdn_lib.decode_layer_step(x["qkv"].to(DEV), x["conv_w"].to(DEV), x["a_raw"].to(DEV),
                                  x["b_raw"].to(DEV), x["A_log"].to(DEV), x["dt_bias"].to(DEV),
                                  st, S, gate.to(DEV), x["norm_w"].to(DEV), 1e-5, "silu")
    assert gdn_lib.device_status() == 0
    st_ref = lio.widen(x["conv_state"]).copy()
    p = lio.prepare_decode_step(x["qkv"], x["conv_w"], x["a_raw"], x["b_raw"], x["A_log"],
                                x["dt_bias"], st_ref, H, 256, dv)
    S_ref = S0.double().numpy().copy()
    f32 = lambda z: np.ascontiguousarray(z, np.float32)
    o = oracle.decode_step(f32(p["q"]), f32(p["k"]), f32(p["v"]), f32(p["alpha"]),
                           f32(p["beta"]), S_ref)
    y_ref = lio.output_norm_gate(o, gate, x["norm_w"], 1e-5, "silu")
    got = y.double().cpu().numpy()
    err = np.linalg.norm(got - y_ref, axis=-1) / np.linalg.norm(y_ref, axis=-1)
    assert err.max() <= 2e-2, err.max()
    Sg = S.cpu().numpy()
    es = np.linalg.norm((Sg - S_ref).reshape(N * H, -1), axis=1) / \
        np.linalg.norm(S_ref.reshape(N * H, -1), axis=1)
    assert es.max() <= 1e-4, es.max()
    assert np.array_equal(st.double().cpu().numpy(), st_ref)
