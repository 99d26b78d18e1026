"""GPU parity of gdn_prefill_backward (the chunked backward, CUDA cores, fp32
arithmetic) against the fp64 token-by-token backward oracle, through the C
ABI.  Tolerances, relative Frobenius error per (sequence, head) of every
gradient: 1e-4 with fp32 I/O and 2e-2 with bf16 I/O (the forward's bounds:
same inputs, fp32 arithmetic, bf16 rounding of dq, dk, dv).  Packing is
checked bit for bit."""
import numpy as np
import pytest
import torch

import gdn_inputs
from gdn_inputs import PrefillCase
from oracle.backward import prefill_backward as oracle_backward

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}


def rel(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / nb) if nb > 0 else float(np.linalg.norm(a))


def grad_inputs(case, seed):
    x = gdn_inputs.make_prefill(case, device="cpu")
    g = torch.Generator().manual_seed(seed)
    x["dout"] = torch.randn(x["v"].shape, generator=g).to(case.io_dtype)
    N = len(case.lengths)
    x["dS_final"] = torch.randn((N, case.H, case.dv, case.dk), generator=g) * 0.1
    return x


def run(gdn, x, with_dsf=True):
    d = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    g = gdn.prefill_backward(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["dout"], d["S0"],
                             d["dS_final"] if with_dsf else None, d["cu_seqlens"])
    assert gdn.device_status() == 0
    return {k: (v.double().cpu().numpy() if v is not None else None) for k, v in g.items()}


def check(gdn, case, seed, with_dsf=True):
    x = grad_inputs(case, seed)
    got = run(gdn, x, with_dsf)
    cu = x["cu_seqlens"]
    if cu is None:
        cu = torch.arange(len(case.lengths) + 1, dtype=torch.int32) * case.lengths[0]
    want = oracle_backward(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["dout"], x["S0"],
                           x["dS_final"] if with_dsf else None, cu)
    H, dk, dv = case.H, case.dk, case.dv
    bounds = np.concatenate([[0], np.cumsum(case.lengths)])
    tol = TOL[case.io_dtype]
    worst = {}
    for key, w in (("dq", dk), ("dk", dk), ("dv", dv), ("dalpha", None), ("dbeta", None)):
        gk = got[key].reshape((-1, H, w) if w else (-1, H))
        for n in range(len(case.lengths)):
            a, b = bounds[n], bounds[n + 1]
            if b == a:
                continue
            for h in range(H):
                e = rel(gk[a:b, h], want[key][a:b, h])
                worst[key] = max(worst.get(key, 0.0), e)
                assert e <= tol, (case.name, key, n, h, e)
    for n in range(len(case.lengths)):
        for h in range(H):
            e = rel(got["dS0"][n, h], want["dS0"][n, h])
            worst["dS0"] = max(worst.get("dS0", 0.0), e)
            assert e <= tol, (case.name, "dS0", n, h, e)
    return worst


@pytest.mark.parametrize("io", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("T", [1, 64, 65, 200])
def test_backward_ragged_lengths(gdn_lib, io, T):
    check(gdn_lib, PrefillCase("bwd dense", [T], H=2, io_dtype=io, seed=91 + T), seed=7)


def test_backward_dense_batch_no_state_gradient(gdn_lib):
    check(gdn_lib, PrefillCase("bwd B=2", [130, 130], H=2, io_dtype=torch.float32, s0_std=None,
                               seed=92), seed=8, with_dsf=False)


def test_backward_varlen_with_empty_sequences(gdn_lib):
    check(gdn_lib, PrefillCase("bwd varlen", [0, 70, 1, 0, 129, 64], H=2,
                               io_dtype=torch.bfloat16, seed=93, varlen=True), seed=9)


def test_backward_repeatable_bitwise(gdn_lib):
    """Repeated calls on the same inputs give the same bits, whatever the
    workspace held before (caller workspaces filled with 0x00 and 0xFF
    bytes in turn).  The packing has chunks of 1 and 64 rows and a sequence
    of 129 tokens, whose one-row chunk starts the reverse pass: the pass's
    first MMA must see every warp's rows of the state-gradient operand."""
    lens = [0, 70, 1, 0, 129, 64]
    case = PrefillCase("bwd repeat", lens, H=2, io_dtype=torch.bfloat16, seed=93, varlen=True)
    x = grad_inputs(case, 9)
    d = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    need = gdn_lib.prefill_backward_workspace_size(len(lens), sum(lens), 2, varlen=True)
    first = None
    for i in range(8):
        buf = torch.full((need + 1024,), 0xFF if i % 2 else 0, dtype=torch.uint8, device=DEV)
        off = (-buf.data_ptr()) % 1024
        g = gdn_lib.prefill_backward(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["dout"],
                                     d["S0"], d["dS_final"], d["cu_seqlens"],
                                     workspace=buf[off:off + need])
        assert gdn_lib.device_status() == 0
        g = {k: v.clone() for k, v in g.items()}
        if first is None:
            first = g
        for key in ("dq", "dk", "dv", "dalpha", "dbeta", "dS0"):
            assert torch.equal(g[key], first[key]), (i, key)


def test_backward_dv512(gdn_lib):
    check(gdn_lib, PrefillCase("bwd dv512", [100, 3], H=1, dv=512, io_dtype=torch.float32,
                               seed=94, varlen=True), seed=10)


def test_backward_six_heads_config_shape(gdn_lib):
    """The small fp32 configuration's geometry (H = 6, d = 256) over 2.5 chunks."""
    check(gdn_lib, PrefillCase("bwd H=6", [160], io_dtype=torch.float32, s0_std=None, seed=95),
          seed=11)


def test_backward_packing_bitwise(gdn_lib):
    lens = [70, 1, 130]
    case = PrefillCase("bwd pack", lens, H=2, io_dtype=torch.bfloat16, seed=96, varlen=True)
    x = grad_inputs(case, 12)
    packed = run(gdn_lib, x)
    cu = np.concatenate([[0], np.cumsum(lens)])
    for n, L in enumerate(lens):
        sl = slice(int(cu[n]), int(cu[n + 1]))
        one = {k: x[k][:, sl].contiguous() for k in ("q", "k", "v", "alpha", "beta", "dout")}
        one["S0"] = x["S0"][n:n + 1].contiguous()
        one["dS_final"] = x["dS_final"][n:n + 1].contiguous()
        one["cu_seqlens"] = None
        alone = run(gdn_lib, one)
        for key in ("dq", "dk", "dv", "dalpha", "dbeta"):
            assert np.array_equal(alone[key][0], packed[key][0, sl]), (n, key)
        assert np.array_equal(alone["dS0"][0], packed["dS0"][n])


def test_backward_split_form_forward_rerun(gdn_lib):
    """70 sequences x 2 heads (140 state units) leave too few SMs for the fused
    launch, so the backward's tensor-core forward re-run (which stores the
    chunk-start states) takes the split form; gradients still match."""
    import ctypes
    rng = np.random.default_rng(97)
    lens = [int(t) for t in rng.integers(1, 150, size=70)]
    check(gdn_lib, PrefillCase("bwd split", lens, H=2, io_dtype=torch.bfloat16, seed=98,
                               varlen=True), seed=13)
    f = gdn_lib.load().gdn_testing_last_prefill_form
    f.restype = ctypes.c_int32
    assert int(f()) == 0
