"""gdn_prefill_layer (the pre-recurrence steps as their own pass, Eq. 20's
gated RMSNorm inside the prefill: its per-chunk workers in the fused form, its
state units as 2-CTA clusters in the split form; for sequences in the
segmented form the convolution inside the per-chunk prep) through the C ABI:

* against the fp64 oracle's composition layer_io.prepare -> oracle.prefill ->
  layer_io.output_norm_gate, within the bf16 tolerance 2e-2 per (sequence,
  head) on y and S_final; the convolution state out is a copy of inputs, so
  exact;
* against the library's own three calls (gdn_prepare -> gdn_prefill ->
  gdn_output_norm_gate): q, k, v, alpha and beta are the same values, so
  S_final and the convolution state are equal bit for bit, and y differs only
  in the order of the norm's sum of squares (a bf16 rounding step at most);
* in both launch forms of the prefill;
* packing never changes a sequence's result, also for a 64K-token sequence
  that the length rule cuts into segments.
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
TOL = 2e-2


def rel(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / nb) if nb > 0 else float(np.linalg.norm(a))


def _inputs(case, s0_seed, device="cpu"):
    x = gdn_inputs.make_layer(case, device="cpu")
    gen = torch.Generator().manual_seed(s0_seed)
    x["S0"] = torch.randn((len(case.lengths), case.H, case.dv, case.dk), generator=gen) * 0.02
    return {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}


def _layer(gdn, xd, case, act="silu", eps=1e-5):
    N = len(case.lengths)
    so = torch.full((N, 3, case.channels), float("nan"), dtype=case.io_dtype, device=DEV)
    y, sf = gdn.prefill_layer(xd["qkv"], xd["conv_w"], xd["a_raw"], xd["b_raw"], xd["A_log"],
                              xd["dt_bias"], xd["g"], xd["norm_w"], case.H, S0=xd["S0"],
                              cu_seqlens=xd["cu_seqlens"], conv_state_in=xd["conv_state"],
                              conv_state_out=so, eps=eps, act=act)
    assert gdn.device_status() == 0
    return y, sf, so


def _three_calls(gdn, xd, case, act="silu", eps=1e-5):
    N = len(case.lengths)
    so = torch.full((N, 3, case.channels), float("nan"), dtype=case.io_dtype, device=DEV)
    p = gdn.prepare(xd["qkv"], xd["conv_w"], xd["a_raw"], xd["b_raw"], xd["A_log"],
                    xd["dt_bias"], case.H, cu_seqlens=xd["cu_seqlens"],
                    conv_state_in=xd["conv_state"], conv_state_out=so)
    o, sf = gdn.prefill(p["q"], p["k"], p["v"], p["alpha"], p["beta"], xd["S0"],
                        xd["cu_seqlens"])
    y = gdn.output_norm_gate(o, xd["g"], xd["norm_w"], eps, act)
    assert gdn.device_status() == 0
    return y, sf, so


def _oracle_units(x, case, units, act="silu", eps=1e-5):
    """The oracle composition for the sampled (sequence, head) units:
    prepare over each sampled sequence (its own history), the token
    recurrence per head, the gated RMSNorm."""
    C, H = case.channels, case.H
    qkv = x["qkv"].reshape(-1, C)
    a, b = x["a_raw"].reshape(-1, H), x["b_raw"].reshape(-1, H)
    g = x["g"].reshape(-1, H, case.dv)
    cu = np.concatenate([[0], np.cumsum(case.lengths)]).astype(np.int64)
    res = {}
    for n in sorted({n for n, _ in units}):
        s, e = int(cu[n]), int(cu[n + 1])
        st = None if x["conv_state"] is None else x["conv_state"][n:n + 1]
        p = lio.prepare(qkv[s:e], x["conv_w"], a[s:e], b[s:e], x["A_log"], x["dt_bias"], H,
                        case.dk, case.dv, np.array([0, e - s]), st)
        hs = [h for m, h in units if m == n]
        f32 = lambda t: np.ascontiguousarray(t[:, hs], dtype=np.float32)
        o, sf, _ = oracle.prefill(f32(p["q"]), f32(p["k"]), f32(p["v"]), f32(p["alpha"]),
                                  f32(p["beta"]), x["S0"][n:n + 1, hs])
        y = lio.output_norm_gate(o, g[s:e][:, hs], x["norm_w"], eps, act)
        for j, h in enumerate(hs):
            res[(n, h)] = (y[:, j], sf[0, j], p["conv_state"][0])
    return res


def _check_oracle(y, sf, so, x, case, units, act="silu"):
    H, dv = case.H, case.dv
    cu = np.concatenate([[0], np.cumsum(case.lengths)])
    yg = y.float().cpu().numpy().reshape(-1, H, dv)
    ref = _oracle_units(x, case, units, act)
    for (n, h), (yr, sr, cr) in ref.items():
        s, e = cu[n], cu[n + 1]
        if e > s:
            assert rel(yg[s:e, h], yr) <= TOL, (n, h)
        assert rel(sf[n, h].cpu().numpy(), sr) <= TOL, (n, h)
        assert np.array_equal(so[n].float().cpu().numpy(), cr), n


@pytest.mark.parametrize("case,act", [
    (LayerCase("layer dense", [200, 200], H=2, seed=131), "silu"),
    (LayerCase("layer varlen", [70, 0, 129, 5, 300, 1], H=2, seed=132, varlen=True), "sigmoid"),
    (LayerCase("layer varlen no history", [64, 65, 2], H=2, seed=133, varlen=True,
               carry_state=False), "silu"),
], ids=lambda c: c.name.replace(" ", "-") if isinstance(c, LayerCase) else c)
def test_layer_matches_oracle_composition(gdn_lib, case, act):
    x = _inputs(case, 134)
    xd = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    y, sf, so = _layer(gdn_lib, xd, case, act)
    units = [(n, h) for n in range(len(case.lengths)) for h in range(case.H)]
    _check_oracle(y, sf, so, x, case, units, act)
    # the three separate calls: equal inputs to the recurrence
    y3, sf3, so3 = _three_calls(gdn_lib, xd, case, act)
    assert torch.equal(sf, sf3) and torch.equal(so, so3)
    assert rel(y.float().cpu().numpy(), y3.float().cpu().numpy()) <= 4e-3


def test_layer_packed_is_bitwise(gdn_lib):
    lens = [300, 0, 129, 1, 64]
    case = LayerCase("layer packed", lens, H=2, seed=135, varlen=True)
    xd = _inputs(case, 136, DEV)
    y, sf, so = _layer(gdn_lib, xd, case)
    cu = [0] + list(np.cumsum(lens))
    C = case.channels
    for n, L in enumerate(lens):
        a, b = cu[n], cu[n + 1]
        one = LayerCase("one", [L], H=2, seed=0, varlen=True)
        xn = {"qkv": xd["qkv"][a:b].contiguous(), "conv_w": xd["conv_w"],
              "a_raw": xd["a_raw"][a:b].contiguous(), "b_raw": xd["b_raw"][a:b].contiguous(),
              "A_log": xd["A_log"], "dt_bias": xd["dt_bias"], "g": xd["g"][a:b].contiguous(),
              "norm_w": xd["norm_w"], "S0": xd["S0"][n:n + 1].contiguous(),
              "conv_state": xd["conv_state"][n:n + 1].contiguous(),
              "cu_seqlens": torch.tensor([0, L], dtype=torch.int32, device=DEV)}
        y1, s1, so1 = _layer(gdn_lib, xn, one)
        assert torch.equal(y[a:b], y1) and torch.equal(sf[n], s1[0]), n
        assert torch.equal(so[n], so1[0]), n
    assert so.shape == (len(lens), 3, C)


def test_layer_at_full_size_8k(gdn_lib):
    """The 8K workload's layer (B=4, T=8192, H=6, bf16): against the three
    calls at every token and head, and the oracle composition on sampled
    (sequence, head) units."""
    case = gdn_inputs.layer_8k()
    x = _inputs(case, 137)
    xd = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    y, sf, so = _layer(gdn_lib, xd, case)
    y3, sf3, so3 = _three_calls(gdn_lib, xd, case)
    assert torch.equal(sf, sf3) and torch.equal(so, so3)
    assert rel(y.float().cpu().numpy(), y3.float().cpu().numpy()) <= 4e-3
    # dense [4, 8192]: as a packing of four sequences for the oracle
    xo = dict(x)
    xo["qkv"] = x["qkv"].reshape(-1, case.channels)
    _check_oracle(y.reshape(-1, case.H, case.dv), sf, so, xo, case, [(0, 0), (3, 5)])


def _last_form(gdn_lib):
    import ctypes
    f = gdn_lib.load().gdn_testing_last_prefill_form
    f.restype = ctypes.c_int32
    return int(f())


@pytest.mark.parametrize("n_seq,form", [(3, 1), (61, 0)])
def test_layer_readout_in_both_launch_forms(gdn_lib, n_seq, form):
    """Few heads: the prefill's fused form, whose per-chunk workers apply
    Eq. 20 behind the chains.  61 sequences x 1 head (122 state units) leave
    too few SMs for the workers: the split form, whose units finish their
    rows as 2-CTA clusters.  Both against the three separate calls."""
    rng = np.random.default_rng(140 + n_seq)
    lens = [int(t) for t in rng.integers(1, 400, size=n_seq)]
    case = LayerCase("layer form", lens, H=1 if n_seq > 3 else 2, seed=141, varlen=True)
    xd = _inputs(case, 142, DEV)
    y, sf, so = _layer(gdn_lib, xd, case)
    assert _last_form(gdn_lib) == form
    y3, sf3, so3 = _three_calls(gdn_lib, xd, case)
    assert torch.equal(sf, sf3) and torch.equal(so, so3)
    assert rel(y.float().cpu().numpy(), y3.float().cpu().numpy()) <= 4e-3


def test_layer_long_sequence(gdn_lib):
    """A 64K-token sequence packed between two short ones: the layer cuts it
    by gdn_prefill's rule (the same bits as the three calls for S_final and
    the convolution state), and packing changes nothing."""
    lens = [1000, 65536, 37]
    case = LayerCase("layer long", lens, H=1, seed=138, varlen=True)
    xd = _inputs(case, 139, DEV)
    y, sf, so = _layer(gdn_lib, xd, case)
    y3, sf3, so3 = _three_calls(gdn_lib, xd, case)
    assert torch.equal(sf, sf3) and torch.equal(so, so3)
    assert rel(y.float().cpu().numpy(), y3.float().cpu().numpy()) <= 4e-3
    a, b = 1000, 1000 + 65536
    one = LayerCase("one", [65536], H=1, seed=0, varlen=True)
    xn = {"qkv": xd["qkv"][a:b].contiguous(), "conv_w": xd["conv_w"],
          "a_raw": xd["a_raw"][a:b].contiguous(), "b_raw": xd["b_raw"][a:b].contiguous(),
          "A_log": xd["A_log"], "dt_bias": xd["dt_bias"], "g": xd["g"][a:b].contiguous(),
          "norm_w": xd["norm_w"], "S0": xd["S0"][1:2].contiguous(),
          "conv_state": xd["conv_state"][1:2].contiguous(),
          "cu_seqlens": torch.tensor([0, 65536], dtype=torch.int32, device=DEV)}
    y1, s1, so1 = _layer(gdn_lib, xn, one)
    assert torch.equal(y[a:b], y1) and torch.equal(sf[1], s1[0]) and torch.equal(so[1], so1[0])
