"""GPU parity of the layer steps around the recurrence (gdn_prepare,
gdn_prepare_decode_step, gdn_output_norm_gate) against the fp64 oracle in
``oracle.layer_io``, through the C ABI.

Tolerances (relative Frobenius error per output tensor, derived from the
arithmetic): fp32 I/O computes and stores in fp32, a few ulp per element, so
1e-5.  bf16 I/O reads exact bf16 inputs, computes in fp32 and rounds each
output once to nearest bf16 (relative error <= 2^-9 per element), so
3e-3 (2^-9 = 1.95e-3 plus the fp32 arithmetic).  alpha and beta are fp32
outputs either way: 1e-5.  The convolution state out is a copy of inputs:
exact.  Segmentation (packed vs alone) and decode-vs-prefill are bit for bit.
"""
import numpy as np
import pytest
import torch

import gdn_inputs
import oracle
from gdn_inputs import LayerCase
from oracle import layer_io as lio

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
TOL = {torch.float32: 1e-5, torch.bfloat16: 3e-3}


def rel(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / nb) if nb > 0 else float(np.linalg.norm(a))


def _f64(t):
    return t.detach().double().cpu().numpy()


def run_prepare(gdn, x, case, state_out=True):
    N = len(case.lengths)
    so = (torch.full((N, 3, case.channels), float("nan"), dtype=case.io_dtype, device=DEV)
          if state_out else None)
    r = gdn.prepare(x["qkv"], x["conv_w"], x["a_raw"], x["b_raw"], x["A_log"], x["dt_bias"],
                    case.H, case.dk, case.dv, cu_seqlens=x["cu_seqlens"],
                    conv_state_in=x["conv_state"], conv_state_out=so)
    assert gdn.device_status() == 0
    r["conv_state"] = so
    return r


def oracle_prepare(x, case):
    qkv = x["qkv"].reshape(-1, case.channels)
    cu = x["cu_seqlens"]
    if cu is None:   # a dense batch: B sequences of equal length
        cu = np.arange(len(case.lengths) + 1) * case.lengths[0]
    return lio.prepare(qkv, x["conv_w"], x["a_raw"].reshape(-1, case.H),
                       x["b_raw"].reshape(-1, case.H), x["A_log"], x["dt_bias"], case.H,
                       case.dk, case.dv, cu, x["conv_state"])


def check_prepare(gdn, case):
    x = gdn_inputs.make_layer(case, device="cpu")
    xd = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    got = run_prepare(gdn, xd, case)
    want = oracle_prepare(x, case)
    T = case.total_tokens
    tol = TOL[case.io_dtype]
    for name, width in (("q", case.dk), ("k", case.dk), ("v", case.dv)):
        g = _f64(got[name]).reshape(T, case.H, width)
        for h in range(case.H):
            assert rel(g[:, h], want[name][:, h]) <= tol, (case.name, name, h)
    for name in ("alpha", "beta"):
        assert rel(_f64(got[name]).reshape(T, case.H), want[name]) <= 1e-5, (case.name, name)
    assert np.array_equal(_f64(got["conv_state"]), want["conv_state"]), case.name
    return got


@pytest.mark.parametrize("io", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("dv", [256, 512])
def test_prepare_dense(gdn_lib, io, dv):
    """Two sequences of 200 tokens: three full tiles of 64 and a ragged one,
    with a carried convolution state."""
    check_prepare(gdn_lib, LayerCase("prepare dense", [200, 200], H=2, dv=dv, io_dtype=io,
                                     seed=81))


@pytest.mark.parametrize("carry", [True, False])
def test_prepare_varlen_short_and_empty(gdn_lib, carry):
    """Sequences shorter than the kernel width, empty ones (also first and
    last), and boundaries inside a 64-token tile."""
    lens = [0, 1, 2, 3, 70, 0, 130, 5, 0]
    check_prepare(gdn_lib, LayerCase("prepare varlen", lens, H=2, io_dtype=torch.bfloat16,
                                     seed=82, varlen=True, carry_state=carry))


def test_prepare_segmentation_bitwise(gdn_lib):
    lens = [70, 1, 130, 64]
    case = LayerCase("prepare seg", lens, H=2, dv=512, io_dtype=torch.bfloat16, seed=83,
                     varlen=True)
    x = gdn_inputs.make_layer(case, device=DEV)
    packed = run_prepare(gdn_lib, x, case)
    cu = np.concatenate([[0], np.cumsum(lens)])
    for n, L in enumerate(lens):
        sl = slice(int(cu[n]), int(cu[n + 1]))
        one = LayerCase("one", [L], H=2, dv=512, io_dtype=torch.bfloat16, varlen=True)
        xo = dict(x, qkv=x["qkv"][sl].contiguous(), a_raw=x["a_raw"][sl].contiguous(),
                  b_raw=x["b_raw"][sl].contiguous(), conv_state=x["conv_state"][n:n + 1].contiguous(),
                  cu_seqlens=torch.tensor([0, L], dtype=torch.int32, device=DEV))
        alone = run_prepare(gdn_lib, xo, one)
        for name in ("q", "k", "v", "alpha", "beta"):
            assert torch.equal(alone[name], packed[name][sl]), (n, name)
        assert torch.equal(alone["conv_state"][0], packed["conv_state"][n])


def test_prepare_decode_steps(gdn_lib):
    """Four decode steps of five sequences, the state carried in place,
    match the oracle step by step."""
    H, dv, N, steps = 2, 256, 5, 4
    case = LayerCase("prepare decode", [1] * (N * steps), H=H, dv=dv, io_dtype=torch.bfloat16,
                     seed=84, varlen=True)
    x = gdn_inputs.make_layer(case, device="cpu")
    C = case.channels
    qkv = x["qkv"].reshape(steps, N, C)
    a = x["a_raw"].reshape(steps, N, H)
    b = x["b_raw"].reshape(steps, N, H)
    state0 = x["conv_state"][:N].clone()
    st_gpu = state0.to(DEV)
    st_ref = lio.widen(state0).copy()
    for t in range(steps):
        got = gdn_lib.prepare_decode_step(qkv[t].to(DEV), x["conv_w"].to(DEV), a[t].to(DEV),
                                          b[t].to(DEV), x["A_log"].to(DEV),
                                          x["dt_bias"].to(DEV), st_gpu, H, 256, dv)
        want = lio.prepare_decode_step(qkv[t], x["conv_w"], a[t], b[t], x["A_log"],
                                       x["dt_bias"], st_ref, H, 256, dv)
        for name in ("q", "k", "v"):
            assert rel(_f64(got[name]), want[name]) <= TOL[torch.bfloat16], (t, name)
        for name in ("alpha", "beta"):
            assert rel(_f64(got[name]), want[name]) <= 1e-5
        assert np.array_equal(_f64(st_gpu), st_ref)
    assert gdn_lib.device_status() == 0


def test_prepare_decode_equals_one_token_prepare(gdn_lib):
    H, dv, N = 2, 512, 7
    case = LayerCase("dec vs prep", [1] * N, H=H, dv=dv, io_dtype=torch.bfloat16, seed=85,
                     varlen=True)
    x = gdn_inputs.make_layer(case, device=DEV)
    st = x["conv_state"].clone()
    dec = gdn_lib.prepare_decode_step(x["qkv"], x["conv_w"], x["a_raw"], x["b_raw"], x["A_log"],
                                      x["dt_bias"], st, H, 256, dv)
    pre = run_prepare(gdn_lib, x, case)
    for name in ("q", "k", "v", "alpha", "beta"):
        assert torch.equal(dec[name], pre[name]), name
    assert torch.equal(st, pre["conv_state"])


def test_prepare_then_prefill_matches_oracle_pipeline(gdn_lib):
    """Raw projections -> gdn_prepare -> gdn_prefill against the oracle's
    prepare and token recurrence (q, k, v handed to the recurrence oracle in
    fp32, rounded on the oracle side)."""
    lens = [130, 1, 64]
    case = LayerCase("pipeline", lens, H=2, io_dtype=torch.bfloat16, seed=86, varlen=True)
    x = gdn_inputs.make_layer(case, device="cpu")
    xd = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    p = run_prepare(gdn_lib, xd, case, state_out=False)
    out, Sf = gdn_lib.prefill(p["q"], p["k"], p["v"], p["alpha"], p["beta"], None,
                              xd["cu_seqlens"])
    assert gdn_lib.device_status() == 0
    w = oracle_prepare(x, case)
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32))
    o_ref, s_ref, _ = oracle.prefill(f32(w["q"]), f32(w["k"]), f32(w["v"]), f32(w["alpha"]),
                                     f32(w["beta"]), None, x["cu_seqlens"])
    o = _f64(out)
    cu = np.concatenate([[0], np.cumsum(lens)])
    for n in range(len(lens)):
        for h in range(case.H):
            a, b = cu[n], cu[n + 1]
            assert rel(o[a:b, h], o_ref[a:b, h]) <= 2e-2
            assert rel(_f64(Sf[n, h]), s_ref[n, h]) <= 2e-2


@pytest.mark.parametrize("io", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("dv", [256, 512])
@pytest.mark.parametrize("act", ["silu", "sigmoid"])
def test_output_norm_gate(gdn_lib, io, dv, act):
    case = LayerCase("norm gate", [300], H=3, dv=dv, io_dtype=io, seed=87)
    x = gdn_inputs.make_layer(case, device="cpu")
    g = torch.Generator().manual_seed(88)
    o = (torch.randn((300, 3, dv), generator=g) * 0.05).to(io)
    o[7, 1] = 0          # an all-zero row: y = 0 exactly (eps > 0)
    eps = 1e-5
    y = gdn_lib.output_norm_gate(o.to(DEV), x["g"].reshape(300, 3, dv).to(DEV),
                                 x["norm_w"].to(DEV), eps, act)
    assert gdn_lib.device_status() == 0
    want = lio.output_norm_gate(o, x["g"].reshape(300, 3, dv), x["norm_w"], eps, act)
    got = _f64(y)
    for h in range(3):
        assert rel(got[:, h], want[:, h]) <= TOL[io], h
    assert np.all(got[7, 1] == 0)


def test_output_norm_gate_in_place(gdn_lib):
    case = LayerCase("norm gate", [129], H=6, dv=256, io_dtype=torch.bfloat16, seed=89)
    x = gdn_inputs.make_layer(case, device=DEV)
    o = torch.randn((129, 6, 256), device=DEV).to(torch.bfloat16)
    y = gdn_lib.output_norm_gate(o, x["g"].reshape(129, 6, 256), x["norm_w"])
    gdn_lib.output_norm_gate(o, x["g"].reshape(129, 6, 256), x["norm_w"], y=o)
    assert gdn_lib.device_status() == 0
    assert torch.equal(o, y)


def test_layer_steps_at_full_size(gdn_lib):
    """The 8K workload (B=4, T=8192, H=6, d=256, bf16) in the launch
    configuration the benchmark times: every output of gdn_prepare and of
    gdn_output_norm_gate against the oracle."""
    case = gdn_inputs.layer_8k()
    x = gdn_inputs.make_layer(case, device="cpu")
    xd = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    got = run_prepare(gdn_lib, xd, case)
    want = oracle_prepare(x, case)
    T = case.total_tokens
    for name, width in (("q", case.dk), ("k", case.dk), ("v", case.dv)):
        assert rel(_f64(got[name]).reshape(T, case.H, width), want[name]) <= 3e-3, name
    for name in ("alpha", "beta"):
        assert rel(_f64(got[name]).reshape(T, case.H), want[name]) <= 1e-5, name
    assert np.array_equal(_f64(got["conv_state"]), want["conv_state"])
    gen = torch.Generator().manual_seed(90)
    o = (torch.randn(x["g"].shape, generator=gen) * 0.05).to(torch.bfloat16)
    y = gdn_lib.output_norm_gate(o.to(DEV), xd["g"], xd["norm_w"], 1e-5, "silu")
    assert gdn_lib.device_status() == 0
    yr = lio.output_norm_gate(o, x["g"], x["norm_w"], 1e-5, "silu")
    assert rel(_f64(y), yr) <= 3e-3


@pytest.mark.parametrize("io", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("dv,act", [(256, "silu"), (512, "sigmoid")])
def test_decode_layer_step_matches_oracle_composition(gdn_lib, io, dv, act):
    """The fused decode step (one cluster launch) against the oracle's prepare,
    token recurrence and gated RMSNorm, over four steps with the convolution
    and recurrent states carried in place."""
    H, N, steps = 2, 5, 4
    case = LayerCase("fused decode", [1] * (N * steps), H=H, dv=dv, io_dtype=io, seed=97,
                     varlen=True)
    x = gdn_inputs.make_layer(case, device="cpu")
    C = case.channels
    qkv = x["qkv"].reshape(steps, N, C)
    a = x["a_raw"].reshape(steps, N, H)
    b = x["b_raw"].reshape(steps, N, H)
    gate = x["g"].reshape(steps, N, H, dv)
    gen = torch.Generator().manual_seed(98)
    S0 = torch.randn((N, H, dv, 256), generator=gen) * 0.02
    st_gpu, S_gpu = x["conv_state"][:N].clone().to(DEV), S0.clone().to(DEV)
    st_ref, S_ref = lio.widen(x["conv_state"][:N]).copy(), S0.double().numpy().copy()
    tol = 1e-4 if io == torch.float32 else 2e-2
    dev = {k: x[k].to(DEV) for k in ("conv_w", "A_log", "dt_bias", "norm_w")}
    for t in range(steps):
        y = gdn_lib.decode_layer_step(qkv[t].to(DEV), dev["conv_w"], a[t].to(DEV), b[t].to(DEV),
                                      dev["A_log"], dev["dt_bias"], st_gpu, S_gpu,
                                      gate[t].to(DEV), dev["norm_w"], 1e-5, act)
        p = lio.prepare_decode_step(qkv[t], x["conv_w"], a[t], b[t], x["A_log"], x["dt_bias"],
                                    st_ref, H, 256, dv)
        f32 = lambda z: np.ascontiguousarray(z, np.float32)
        o = oracle.decode_step(f32(p["q"]), f32(p["k"]), f32(p["v"]), f32(p["alpha"]),
                               f32(p["beta"]), S_ref)
        y_ref = lio.output_norm_gate(o, gate[t], x["norm_w"], 1e-5, act)
        got = _f64(y)
        for n in range(N):
            for h in range(H):
                assert rel(got[n, h], y_ref[n, h]) <= tol, (t, n, h)
        assert np.array_equal(_f64(st_gpu), st_ref)
    assert gdn_lib.device_status() == 0
    Sg = S_gpu.cpu().numpy()
    for n in range(N):
        for h in range(H):
            assert rel(Sg[n, h], S_ref[n, h]) <= 1e-4
