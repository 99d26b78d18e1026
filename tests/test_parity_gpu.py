"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on
the same seeded inputs.

Tolerances: max over (sequence, head) of the relative Frobenius error
||X_gpu - X_ref||_F / ||X_ref||_F, for X = the outputs and the final state:
<= 1e-4 with fp32 q/k/v/out, <= 2e-2 with bf16 q/k/v/out (fp32 state and
accumulation either way).  Segmentation through cu_seqlens is checked
bit for bit.
"""
import numpy as np
import pytest
import torch

import gdn_inputs
import oracle
from gdn_inputs import PrefillCase

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}
DEV = torch.device("cuda:0")


def rel(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / nb) if nb > 0 else float(np.linalg.norm(a))


def to_dev(x):
    return {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}


def run_gpu(gdn, x):
    out, S_final = gdn.prefill(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["S0"],
                               x["cu_seqlens"])
    assert gdn.device_status() == 0
    return out, S_final


def per_unit_errors(case, out, S_final, o_ref, s_ref, units=None):
    """Max relative errors over (sequence, head) units."""
    out = out.float().cpu().numpy().reshape(-1, case.H, case.dv)
    o_ref = o_ref.reshape(-1, case.H, case.dv)
    S_final = S_final.cpu().numpy()
    cu = np.concatenate([[0], np.cumsum(case.lengths)])
    eo = es = 0.0
    for n in range(len(case.lengths)):
        for h in range(case.H):
            if units is not None and (n, h) not in units:
                continue
            a, b = cu[n], cu[n + 1]
            if b > a:
                eo = max(eo, rel(out[a:b, h], o_ref[a:b, h]))
            es = max(es, rel(S_final[n, h], s_ref[n, h]))
    return eo, es


def check_case(gdn, case):
    x = gdn_inputs.make_prefill(case, device="cpu")
    xd = to_dev(x)
    out, S_final = run_gpu(gdn, xd)
    o_ref, s_ref, _ = oracle.prefill(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["S0"],
                                     x["cu_seqlens"])
    eo, es = per_unit_errors(case, out, S_final, o_ref, s_ref)
    tol = TOL[case.io_dtype]
    assert eo <= tol and es <= tol, (case.name, eo, es)
    return eo, es


# ----------------------------------------------------------------- prefill
def test_prefill_small_fp32_config(gdn_lib):
    """B=1, T=512, H=6, d=256, fp32 throughout, S0 = 0, seed 0 (tolerance 1e-4)."""
    check_case(gdn_lib, gdn_inputs.prefill_small_fp32())


@pytest.mark.parametrize("io", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("T", [1, 63, 64, 65, 127, 200])
def test_prefill_ragged_lengths(gdn_lib, io, T):
    check_case(gdn_lib, PrefillCase(f"ragged T={T}", [T, T], H=2, io_dtype=io, seed=T))


@pytest.mark.parametrize("io", [torch.float32, torch.bfloat16])
def test_prefill_varlen_small(gdn_lib, io):
    lens = [5, 0, 64, 130, 1, 77]
    check_case(gdn_lib, PrefillCase("varlen small", lens, H=3, io_dtype=io, seed=21, varlen=True))


def test_prefill_zero_state_pointer(gdn_lib):
    check_case(gdn_lib, PrefillCase("S0 NULL", [150], H=2, io_dtype=torch.bfloat16,
                                    s0_std=None, seed=5))


def test_prefill_without_final_state(gdn_lib):
    case = PrefillCase("no S_final", [70], H=1, io_dtype=torch.float32, seed=6)
    x = to_dev(gdn_inputs.make_prefill(case, device="cpu"))
    out, S_final = gdn_lib.prefill(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["S0"],
                                   return_final=False)
    assert S_final is None
    ref, _ = gdn_lib.prefill(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["S0"])
    assert torch.equal(out, ref)


def test_varlen_segmentation_is_bitwise(gdn_lib):
    """(i) each packed sequence equals its standalone run bit for bit;
    (ii) perturbing one sequence's tokens and S0 leaves every other sequence's
    outputs and final state bitwise unchanged; (iii) an empty sequence
    returns S_final = S0 exactly."""
    lens = [100, 0, 64, 1, 257]
    case = PrefillCase("seg", lens, H=2, io_dtype=torch.bfloat16, seed=31, varlen=True)
    x = to_dev(gdn_inputs.make_prefill(case, device="cpu"))
    out, Sf = run_gpu(gdn_lib, x)
    cu = [0] + list(np.cumsum(lens))
    for n, L in enumerate(lens):
        a, b = cu[n], cu[n + 1]
        sl = lambda t: t[:, a:b].contiguous()
        o1, s1 = gdn_lib.prefill(sl(x["q"]), sl(x["k"]), sl(x["v"]), sl(x["alpha"]),
                                 sl(x["beta"]), x["S0"][n:n + 1].contiguous())
        assert torch.equal(out[:, a:b], o1) and torch.equal(Sf[n], s1[0]), n
    assert torch.equal(Sf[1], x["S0"][1])
    # perturb sequence 3 (the single-token one) and its S0
    y = {k: (v.clone() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    a, b = cu[3], cu[4]
    y["v"][:, a:b] += 1.0
    y["k"][:, a:b] *= -1.0
    y["S0"][3] += 0.5
    out2, Sf2 = run_gpu(gdn_lib, y)
    for n in range(len(lens)):
        if n == 3:
            continue
        assert torch.equal(out2[:, cu[n]:cu[n + 1]], out[:, cu[n]:cu[n + 1]])
        assert torch.equal(Sf2[n], Sf[n])


@pytest.mark.parametrize("io", [torch.float32, torch.bfloat16])
def test_resume_from_final_state(gdn_lib, io):
    """prefill(T1) then prefill(T2, S0 = S_final) equals prefill(T1 + T2):
    bitwise at a chunk-aligned split, within tolerance of the oracle at a
    ragged one."""
    case = PrefillCase("resume", [320], H=2, io_dtype=io, seed=41)
    x = to_dev(gdn_inputs.make_prefill(case, device="cpu"))
    full_o, full_s = run_gpu(gdn_lib, x)
    for split in (128, 77):
        part = lambda t, a, b: t[:, a:b].contiguous()
        o1, s1 = gdn_lib.prefill(part(x["q"], 0, split), part(x["k"], 0, split),
                                 part(x["v"], 0, split), part(x["alpha"], 0, split),
                                 part(x["beta"], 0, split), x["S0"])
        o2, s2 = gdn_lib.prefill(part(x["q"], split, 320), part(x["k"], split, 320),
                                 part(x["v"], split, 320), part(x["alpha"], split, 320),
                                 part(x["beta"], split, 320), s1)
        if split % 64 == 0:
            assert torch.equal(torch.cat([o1, o2], 1), full_o) and torch.equal(s2, full_s)
        else:
            assert rel(s2.cpu().numpy(), full_s.cpu().numpy()) <= TOL[io]
            assert rel(torch.cat([o1, o2], 1).float().cpu().numpy(),
                       full_o.float().cpu().numpy()) <= TOL[io]


def test_malformed_cu_seqlens_sets_status(gdn_lib):
    """A non-monotone cu_seqlens is caught on the device: the status word says
    so and the call leaves every sequence with zero chunks (S_final = S0)."""
    case = PrefillCase("bad cu", [10, 20], H=1, io_dtype=torch.float32, seed=7, varlen=True)
    x = to_dev(gdn_inputs.make_prefill(case, device="cpu"))
    bad = torch.tensor([0, 25, 30], dtype=torch.int32, device=DEV)
    bad[1] = 31   # 31 > 30: decreasing
    _, Sf = gdn_lib.prefill(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["S0"], bad)
    assert gdn_lib.device_status() == 6
    assert torch.equal(Sf, x["S0"])
    assert gdn_lib.device_status() == 0


# ------------------------------------------------------------------ decode
@pytest.mark.parametrize("io", [torch.float32, torch.bfloat16])
def test_decode_steps_against_oracle(gdn_lib, io):
    case = gdn_inputs.DecodeCase("decode small", N=5, steps=12, H=3, io_dtype=io, seed=2)
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
            assert rel(S[n, h], S_ref[n, h]) <= 1e-4   # fp32 state either way


def test_decode_equals_single_token_prefill(gdn_lib):
    case = gdn_inputs.DecodeCase("decode vs prefill", N=3, steps=1, H=2,
                                 io_dtype=torch.float32, seed=9)
    d = gdn_inputs.make_decode(case, device="cpu")
    args = {name: d[name][0].to(DEV) for name in ("q", "k", "v", "alpha", "beta")}
    S = d["S"].to(DEV)
    o_p, s_p = gdn_lib.prefill(args["q"][:, None].contiguous(), args["k"][:, None].contiguous(),
                               args["v"][:, None].contiguous(),
                               args["alpha"][:, None].contiguous(),
                               args["beta"][:, None].contiguous(), S)
    o_d = gdn_lib.decode_step(args["q"], args["k"], args["v"], args["alpha"], args["beta"], S)
    assert rel(o_d.cpu().numpy(), o_p[:, 0].cpu().numpy()) <= 1e-5
    assert rel(S.cpu().numpy(), s_p.cpu().numpy()) <= 1e-5


def _last_form(gdn_lib):
    import ctypes
    f = gdn_lib.load().gdn_testing_last_prefill_form
    f.restype = ctypes.c_int32
    return int(f())


@pytest.mark.parametrize("lens,varlen", [([4160], False), ([700, 64, 1, 2000], True)])
def test_prefill_fused_against_oracle(gdn_lib, lens, varlen):
    """Few sequences x heads: the tensor-core prefill runs as one cooperative
    launch in which per-chunk workers hand each chunk's operands to the state
    pass through ready flags (chunk positions in order, sequences of unequal
    length included); the result matches the oracle."""
    check_case(gdn_lib, PrefillCase("fused", lens, H=2, io_dtype=torch.bfloat16, seed=61,
                                    varlen=varlen))
    assert _last_form(gdn_lib) == 1


@pytest.mark.parametrize("lens,varlen", [([4160], False), ([700, 64, 1, 2000], True)])
def test_prefill_fused_matches_split_bitwise(gdn_lib, lens, varlen):
    """The fused launch and the split one (per-chunk kernel, then state-pass
    kernel: what gdn_prefill_scan runs with one segment, every sequence left
    whole) do the same arithmetic in the same order, so they agree bit for
    bit."""
    H = 2
    case = PrefillCase("fused vs split", lens, H=H, io_dtype=torch.bfloat16, seed=62, varlen=varlen)
    x = to_dev(gdn_inputs.make_prefill(case, device="cpu"))
    out, Sf = run_gpu(gdn_lib, x)
    assert _last_form(gdn_lib) == 1
    out1, Sf1 = gdn_lib.prefill_scan(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["S0"],
                                     x["cu_seqlens"], segments=1)
    assert gdn_lib.device_status() == 0
    assert _last_form(gdn_lib) == 0
    assert torch.equal(out.reshape(out1.shape), out1) and torch.equal(Sf, Sf1)


def test_prefill_many_units_split_form(gdn_lib):
    """70 sequences x 1 head leave too few SMs for the fused form's workers:
    the split form runs (persistent per-chunk kernel over every item), and
    matches the oracle."""
    rng = np.random.default_rng(5)
    lens = [int(t) for t in rng.integers(1, 200, size=70)]
    check_case(gdn_lib, PrefillCase("split", lens, H=1, io_dtype=torch.bfloat16, seed=63,
                                    varlen=True))
    assert _last_form(gdn_lib) == 0
