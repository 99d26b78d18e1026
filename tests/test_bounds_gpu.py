"""Bounds checks with guard bands (compute-sanitizer is not available): every
output and in-place state sits inside a larger buffer whose leading and
trailing 4 KiB hold a canary pattern; after each entry point runs, the
canaries must be untouched."""
import pytest
import torch

import gdn_inputs
from gdn_inputs import LayerCase, PrefillCase

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
GUARD_BYTES = 4096


class Guarded:
    """A contiguous tensor of `shape` in the middle of a canary-filled buffer."""

    def __init__(self, shape, dtype, init=None):
        es = torch.tensor([], dtype=dtype).element_size()
        self.g = GUARD_BYTES // es
        n = 1
        for d in shape:
            n *= d
        self.n = n
        self.base = torch.empty(n + 2 * self.g, dtype=dtype, device=DEV)
        self.base.view(torch.uint8).fill_(0xA5)
        self.t = self.base[self.g:self.g + n].view(shape)
        if init is not None:
            self.t.copy_(init)

    def intact(self):
        b = self.base.view(torch.uint8)
        gb = self.g * self.base.element_size()
        return bool((b[:gb] == 0xA5).all()) and bool((b[b.numel() - gb:] == 0xA5).all())


def test_prefill_outputs_stay_in_bounds(gdn_lib):
    for case in (PrefillCase("fused", [130, 1, 64], H=2, seed=41, varlen=True),
                 PrefillCase("split", [40] * 70, H=2, seed=42, varlen=True),
                 PrefillCase("fp32", [100], H=2, io_dtype=torch.float32, seed=43),
                 PrefillCase("dv512", [70, 3], H=1, dv=512, seed=44, varlen=True)):
        x = gdn_inputs.make_prefill(case, device=DEV)
        out = Guarded(x["v"].shape, x["v"].dtype)
        sf = Guarded(x["S0"].shape, torch.float32)
        gdn_lib.prefill(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["S0"],
                        x["cu_seqlens"], out=out.t, S_final=sf.t)
        assert gdn_lib.device_status() == 0
        assert out.intact() and sf.intact(), case.name


def test_decode_and_fused_decode_stay_in_bounds(gdn_lib):
    for dv in (256, 512):
        d = gdn_inputs.make_decode(gdn_inputs.DecodeCase("b", N=3, steps=1, H=2, dv=dv, seed=45),
                                   device=DEV)
        S = Guarded(d["S"].shape, torch.float32, d["S"])
        out = Guarded(d["v"].shape[1:], d["v"].dtype)
        gdn_lib.decode_step(d["q"][0], d["k"][0], d["v"][0], d["alpha"][0], d["beta"][0], S.t,
                            out=out.t)
        assert gdn_lib.device_status() == 0
        assert S.intact() and out.intact()
        lc = LayerCase("b", [1] * 3, H=2, dv=dv, seed=46, varlen=True)
        lx = gdn_inputs.make_layer(lc, device=DEV)
        st = Guarded(lx["conv_state"].shape, lx["conv_state"].dtype, lx["conv_state"])
        S2 = Guarded((3, 2, dv, 256), torch.float32, torch.zeros((3, 2, dv, 256)))
        y = Guarded((3, 2, dv), lx["g"].dtype)
        gdn_lib.decode_layer_step(lx["qkv"], lx["conv_w"], lx["a_raw"], lx["b_raw"], lx["A_log"],
                                  lx["dt_bias"], st.t, S2.t, lx["g"].reshape(3, 2, dv),
                                  lx["norm_w"], y=y.t)
        out2 = {k: Guarded(v.shape, v.dtype) for k, v in (
            ("q", torch.empty((3, 2, 256), dtype=lx["qkv"].dtype)),
            ("k", torch.empty((3, 2, 256), dtype=lx["qkv"].dtype)),
            ("v", torch.empty((3, 2, dv), dtype=lx["qkv"].dtype)),
            ("alpha", torch.empty((3, 2))), ("beta", torch.empty((3, 2))))}
        gdn_lib.prepare_decode_step(lx["qkv"], lx["conv_w"], lx["a_raw"], lx["b_raw"],
                                    lx["A_log"], lx["dt_bias"], st.t, 2, dv=dv,
                                    out={k: g.t for k, g in out2.items()})
        assert gdn_lib.device_status() == 0
        assert st.intact() and S2.intact() and y.intact()
        assert all(g.intact() for g in out2.values())


def test_norm_gate_stays_in_bounds(gdn_lib):
    for io, dv in ((torch.bfloat16, 256), (torch.float32, 512)):
        o = torch.randn((33, 3, dv), device=DEV).to(io)
        g = torch.randn((33, 3, dv), device=DEV).to(io)
        y = Guarded(o.shape, io)
        gdn_lib.output_norm_gate(o, g, torch.ones(dv, device=DEV), y=y.t)
        assert gdn_lib.device_status() == 0
        assert y.intact()


def test_backward_outputs_stay_in_bounds(gdn_lib):
    case = PrefillCase("bwd", [70, 1], H=2, seed=47, varlen=True)
    x = gdn_inputs.make_prefill(case, device=DEV)
    dout = torch.randn(x["v"].shape, device=DEV).to(x["v"].dtype)
    g = gdn_lib.prefill_backward(x["q"], x["k"], x["v"], x["alpha"], x["beta"], dout, x["S0"],
                                 None, x["cu_seqlens"])
    assert gdn_lib.device_status() == 0
    # the binding allocates its outputs; re-run through the C ABI into guarded ones
    import ctypes
    outs = {k: Guarded(v.shape, v.dtype) for k, v in g.items() if v is not None}
    f = gdn_lib.load().gdn_prefill_backward
    p = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None
    rc = f(p(x["q"]), p(x["k"]), p(x["v"]), p(x["alpha"]), p(x["beta"]), p(x["S0"]),
           p(x["cu_seqlens"]), p(dout), None, p(outs["dq"].t), p(outs["dk"].t), p(outs["dv"].t),
           p(outs["dalpha"].t), p(outs["dbeta"].t), p(outs["dS0"].t), 2, 71, 2, 256, 256, 1,
           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0 and gdn_lib.device_status() == 0
    for k, gt in outs.items():
        assert gt.intact(), k
        assert torch.equal(gt.t, g[k]), k


def test_prepare_outputs_stay_in_bounds(gdn_lib):
    import ctypes
    lc = LayerCase("prep", [70, 0, 3], H=2, seed=48, varlen=True)
    lx = gdn_inputs.make_layer(lc, device=DEV)
    T, C = lc.total_tokens, lc.channels
    io = lx["qkv"].dtype
    outs = dict(q=Guarded((T, 2, 256), io), k=Guarded((T, 2, 256), io), v=Guarded((T, 2, 256), io),
                alpha=Guarded((T, 2), torch.float32), beta=Guarded((T, 2), torch.float32),
                st=Guarded((3, 3, C), io))
    p = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None
    rc = gdn_lib.load().gdn_prepare(
        p(lx["qkv"]), p(lx["conv_w"]), p(lx["a_raw"]), p(lx["b_raw"]), p(lx["A_log"]),
        p(lx["dt_bias"]), p(lx["cu_seqlens"]), p(lx["conv_state"]), p(outs["st"].t),
        p(outs["q"].t), p(outs["k"].t), p(outs["v"].t), p(outs["alpha"].t), p(outs["beta"].t),
        3, T, 2, 256, 256, 1, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0 and gdn_lib.device_status() == 0
    assert all(g.intact() for g in outs.values())
