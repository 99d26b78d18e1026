"""Caller-owned scratch: the ``*_ws`` entry points against the fp64 oracle and
against their pool-allocating twins (bit for bit: same kernels, same scratch
layout), and gdn_release_scratch handing the library's pool back.

The library's pool keeps freed scratch mapped between calls (remapping it
after every synchronisation would cost about as much as a call); these tests
check that a caller can see and release what it holds, and that a call given
a workspace never touches the pool."""
import numpy as np
import pytest
import torch

import gdn_inputs
import oracle
from gdn_inputs import PrefillCase

from test_parity_gpu import TOL, per_unit_errors, to_dev

pytestmark = pytest.mark.gpu


def _workspace(nbytes):
    # torch's caching allocator hands out 512-byte aligned blocks; the
    # backward and the scan ask for 1024: over-allocate and offset
    buf = torch.empty(nbytes + 1024, dtype=torch.uint8, device="cuda")
    off = (-buf.data_ptr()) % 1024
    return buf[off:off + nbytes]


@pytest.mark.parametrize("case", [
    PrefillCase("ws dense bf16", [200, 200], H=3, io_dtype=torch.bfloat16, seed=61),
    PrefillCase("ws varlen bf16", [70, 0, 129, 5], H=2, io_dtype=torch.bfloat16, seed=62,
                varlen=True),
    PrefillCase("ws dense fp32", [130], H=2, io_dtype=torch.float32, seed=63),
    PrefillCase("ws varlen fp32", [64, 1, 100], H=2, io_dtype=torch.float32, seed=64,
                varlen=True),
], ids=lambda c: c.name.replace(" ", "-"))
def test_prefill_ws_matches_oracle_and_pool_form(gdn_lib, case):
    x = gdn_inputs.make_prefill(case, device="cpu")
    xd = to_dev(x)
    N, T_total = len(case.lengths), sum(case.lengths)
    need = gdn_lib.prefill_workspace_size(N, T_total if case.varlen else case.lengths[0], case.H,
                                          io_dtype=case.io_dtype, varlen=case.varlen)
    ws = _workspace(need)
    out, S_final = gdn_lib.prefill(xd["q"], xd["k"], xd["v"], xd["alpha"], xd["beta"], xd["S0"],
                                   xd["cu_seqlens"], workspace=ws)
    assert gdn_lib.device_status() == 0
    o_ref, s_ref, _ = oracle.prefill(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["S0"],
                                     x["cu_seqlens"])
    eo, es = per_unit_errors(case, out, S_final, o_ref, s_ref)
    assert eo <= TOL[case.io_dtype] and es <= TOL[case.io_dtype], (eo, es)
    out2, S2 = gdn_lib.prefill(xd["q"], xd["k"], xd["v"], xd["alpha"], xd["beta"], xd["S0"],
                               xd["cu_seqlens"])
    assert torch.equal(out, out2) and torch.equal(S_final, S2)


def test_prefill_ws_segmented_form_matches_pool_form(gdn_lib):
    """A 64K-token sequence (cut into segments by gdn_prefill) with its scratch
    in a caller workspace of gdn_prefill_workspace_size bytes: the same bits
    as the pool form."""
    case = PrefillCase("ws long", [65536], H=1, io_dtype=torch.bfloat16, seed=70)
    xd = to_dev(gdn_inputs.make_prefill(case, device="cpu"))
    args = (xd["q"], xd["k"], xd["v"], xd["alpha"], xd["beta"], xd["S0"])
    ws = _workspace(gdn_lib.prefill_workspace_size(1, 65536, 1))
    a = gdn_lib.prefill(*args, workspace=ws)
    b = gdn_lib.prefill(*args)
    assert gdn_lib.device_status() == 0
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_prefill_ws_rejects_a_small_workspace_without_launching(gdn_lib):
    case = PrefillCase("ws small", [256], H=2, io_dtype=torch.bfloat16, seed=65)
    xd = to_dev(gdn_inputs.make_prefill(case, device="cpu"))
    need = gdn_lib.prefill_workspace_size(1, 256, 2)
    ws = _workspace(need - 256)
    before = gdn_lib.kernel_launches()
    with pytest.raises(gdn_lib.GDNError) as e:
        gdn_lib.prefill(xd["q"], xd["k"], xd["v"], xd["alpha"], xd["beta"], xd["S0"],
                        workspace=ws)
    assert e.value.code == 1 and gdn_lib.kernel_launches() == before


@pytest.mark.parametrize("io", [torch.bfloat16, torch.float32])
def test_scan_ws_matches_scan(gdn_lib, io):
    case = PrefillCase("ws scan", [1000, 0, 1000], H=2, io_dtype=io, seed=66, varlen=True)
    xd = to_dev(gdn_inputs.make_prefill(case, device="cpu"))
    need = gdn_lib.prefill_scan_workspace_size(3, 2000, 2, io_dtype=io, varlen=True, segments=3)
    ws = _workspace(need)
    a = gdn_lib.prefill_scan(xd["q"], xd["k"], xd["v"], xd["alpha"], xd["beta"], xd["S0"],
                             xd["cu_seqlens"], segments=3, workspace=ws)
    b = gdn_lib.prefill_scan(xd["q"], xd["k"], xd["v"], xd["alpha"], xd["beta"], xd["S0"],
                             xd["cu_seqlens"], segments=3)
    assert gdn_lib.device_status() == 0
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("lens,H,varlen", [([8192], 1, False), ([0, 70, 1, 0, 129, 64], 2, True)])
def test_prefill_ws_contents_do_not_matter(gdn_lib, lens, H, varlen):
    """Every byte the call reads from its workspace it wrote first: workspaces
    filled with 0x00, 0xFF and 0x7F bytes give the same bits (one sequence
    over 128 chunks in the fused form; a packing with empty sequences and
    one-row chunks)."""
    case = PrefillCase("ws fill", lens, H=H, io_dtype=torch.bfloat16, seed=64, varlen=varlen)
    xd = to_dev(gdn_inputs.make_prefill(case, device="cpu"))
    need = gdn_lib.prefill_workspace_size(len(lens), sum(lens) if varlen else lens[0], H,
                                          varlen=varlen)
    got = []
    for fill in (0x00, 0xFF, 0x7F):
        ws = _workspace(need)
        ws.fill_(fill)
        out, Sf = gdn_lib.prefill(xd["q"], xd["k"], xd["v"], xd["alpha"], xd["beta"], xd["S0"],
                                  xd["cu_seqlens"], workspace=ws)
        assert gdn_lib.device_status() == 0
        got.append((out.clone(), Sf.clone()))
    for out, Sf in got[1:]:
        assert torch.equal(out, got[0][0]) and torch.equal(Sf, got[0][1])


@pytest.mark.parametrize("io", [torch.bfloat16, torch.float32])
def test_backward_ws_matches_backward(gdn_lib, io):
    case = PrefillCase("ws bwd", [70, 129], H=2, io_dtype=io, seed=67, varlen=True)
    x = gdn_inputs.make_prefill(case, device="cpu")
    xd = to_dev(x)
    g = torch.Generator().manual_seed(68)
    dout = torch.randn(x["v"].shape, generator=g).to(io).cuda()
    dsf = (torch.randn(x["S0"].shape, generator=g) * 0.1).cuda()
    need = gdn_lib.prefill_backward_workspace_size(2, 199, 2, io_dtype=io, varlen=True)
    ws = _workspace(need)
    a = gdn_lib.prefill_backward(xd["q"], xd["k"], xd["v"], xd["alpha"], xd["beta"], dout,
                                 xd["S0"], dsf, xd["cu_seqlens"], workspace=ws)
    b = gdn_lib.prefill_backward(xd["q"], xd["k"], xd["v"], xd["alpha"], xd["beta"], dout,
                                 xd["S0"], dsf, xd["cu_seqlens"])
    assert gdn_lib.device_status() == 0
    for key in ("dq", "dk", "dv", "dalpha", "dbeta", "dS0"):
        assert torch.equal(a[key], b[key]), key


def test_release_scratch_returns_the_pool_and_ws_calls_leave_it_alone(gdn_lib):
    case = PrefillCase("ws release", [2048, 2048], H=6, io_dtype=torch.bfloat16, seed=69)
    xd = to_dev(gdn_inputs.make_prefill(case, device="cpu"))
    args = (xd["q"], xd["k"], xd["v"], xd["alpha"], xd["beta"], xd["S0"])
    gdn_lib.prefill(*args)                               # scratch from the pool
    torch.cuda.synchronize()
    need = gdn_lib.prefill_workspace_size(2, 2048, 6)
    assert gdn_lib.scratch_reserved() >= need            # the pool kept it mapped
    gdn_lib.release_scratch()
    assert gdn_lib.scratch_reserved() == 0
    ws = _workspace(need)
    gdn_lib.prefill(*args, workspace=ws)                 # allocates nothing
    torch.cuda.synchronize()
    assert gdn_lib.scratch_reserved() == 0
    assert gdn_lib.device_status() == 0
