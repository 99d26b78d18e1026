"""GPU parity at dv = 512, the value expansion dv = 2 dk of Table 8 of "Long-Context
Aware Upcycling" (the configurations use dv = dk = 256): prefill and decode through the
C ABI against the fp64 oracle, same tolerances as at dv = 256."""
import numpy as np
import pytest
import torch

import gdn_inputs
import oracle
from gdn_inputs import PrefillCase
from test_parity_gpu import DEV, TOL, check_case, rel, run_gpu, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("io", [torch.float32, torch.bfloat16])
def test_prefill_dv512_dense(gdn_lib, io):
    """Two sequences of 200 tokens: three full chunks and a ragged one."""
    check_case(gdn_lib, PrefillCase("dv512 dense", [200, 200], H=2, dv=512, io_dtype=io,
                                    seed=71))


def test_prefill_dv512_varlen_and_segmentation(gdn_lib):
    """Packed sequences of unequal length match the oracle, and each one equals
    its own standalone run bit for bit."""
    lens = [70, 1, 130]
    case = PrefillCase("dv512 varlen", lens, H=2, dv=512, io_dtype=torch.bfloat16, seed=72,
                       varlen=True)
    check_case(gdn_lib, case)
    x = to_dev(gdn_inputs.make_prefill(case, device="cpu"))
    out, Sf = run_gpu(gdn_lib, x)
    cu = np.concatenate([[0], np.cumsum(lens)])
    for n, L in enumerate(lens):
        sl = {k: x[k][:, cu[n]:cu[n + 1]].contiguous() for k in ("q", "k", "v", "alpha", "beta")}
        o1, s1 = gdn_lib.prefill(sl["q"], sl["k"], sl["v"], sl["alpha"], sl["beta"],
                                 x["S0"][n:n + 1].contiguous())
        assert gdn_lib.device_status() == 0
        assert torch.equal(o1[0], out[0, cu[n]:cu[n + 1]]) and torch.equal(s1[0], Sf[n])


@pytest.mark.parametrize("io", [torch.float32, torch.bfloat16])
def test_decode_dv512(gdn_lib, io):
    case = gdn_inputs.DecodeCase("decode dv512", N=3, steps=8, H=2, dv=512, io_dtype=io, seed=73)
    d = gdn_inputs.make_decode(case, device="cpu")
    S = d["S"].to(DEV)
    S_ref = d["S"].double().numpy().copy()
    outs, refs = [], []
    for t in range(case.steps):
        args = [d[name][t].to(DEV) for name in ("q", "k", "v", "alpha", "beta")]
        outs.append(gdn_lib.decode_step(*args, S).float().cpu().numpy())
        refs.append(oracle.decode_step(d["q"][t], d["k"][t], d["v"][t], d["alpha"][t],
                                       d["beta"][t], S_ref))
    assert gdn_lib.device_status() == 0
    outs, refs = np.stack(outs), np.stack(refs)
    S = S.cpu().numpy()
    for n in range(case.N):
        for h in range(case.H):
            assert rel(outs[:, n, h], refs[:, n, h]) <= TOL[io]
            assert rel(S[n, h], S_ref[n, h]) <= 1e-4


def test_decode_dv512_equals_single_token_prefill(gdn_lib):
    case = gdn_inputs.DecodeCase("decode vs prefill dv512", N=2, steps=1, H=2, dv=512,
                                 io_dtype=torch.float32, seed=74)
    d = gdn_inputs.make_decode(case, device="cpu")
    a = {name: d[name][0].to(DEV) for name in ("q", "k", "v", "alpha", "beta")}
    S = d["S"].to(DEV)
    o_p, s_p = gdn_lib.prefill(a["q"][:, None].contiguous(), a["k"][:, None].contiguous(),
                               a["v"][:, None].contiguous(), a["alpha"][:, None].contiguous(),
                               a["beta"][:, None].contiguous(), S)
    o_d = gdn_lib.decode_step(a["q"], a["k"], a["v"], a["alpha"], a["beta"], S)
    assert rel(o_d.cpu().numpy(), o_p[:, 0].cpu().numpy()) <= 1e-5
    assert rel(S.cpu().numpy(), s_p.cpu().numpy()) <= 1e-5


def _last_form(gdn_lib):
    import ctypes
    f = gdn_lib.load().gdn_testing_last_prefill_form
    f.restype = ctypes.c_int32
    return int(f())


def test_prefill_dv512_split_form(gdn_lib):
    """40 sequences x 1 head x 4 slices of S leave too few SMs for the fused
    form: the split form runs at dv = 512 and matches the oracle."""
    rng = np.random.default_rng(75)
    lens = [int(t) for t in rng.integers(1, 150, size=40)]
    check_case(gdn_lib, PrefillCase("dv512 split", lens, H=1, dv=512, io_dtype=torch.bfloat16,
                                    seed=75, varlen=True))
    assert _last_form(gdn_lib) == 0


def test_prefill_dv512_fused_matches_split_bitwise(gdn_lib):
    """At dv = 512 the fused launch and the split one (what gdn_prefill_scan
    runs with one segment) agree bit for bit."""
    lens = [700, 64, 1, 900]
    H, dv = 2, 512
    case = PrefillCase("dv512 fused vs split", lens, H=H, dv=dv, io_dtype=torch.bfloat16, seed=76,
                       varlen=True)
    x = to_dev(gdn_inputs.make_prefill(case, device="cpu"))
    out, Sf = run_gpu(gdn_lib, x)
    assert _last_form(gdn_lib) == 1
    out1, Sf1 = gdn_lib.prefill_scan(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["S0"],
                                     x["cu_seqlens"], segments=1)
    assert gdn_lib.device_status() == 0
    assert _last_form(gdn_lib) == 0
    assert torch.equal(out, out1) and torch.equal(Sf, Sf1)
