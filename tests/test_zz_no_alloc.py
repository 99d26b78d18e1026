"""gdn_prefill_noalloc: the prefill for callers that must not allocate device
memory while they run (serving loops with a memory footprint fixed at
start-up, processes whose device memory belongs to another allocator, static
memory budgets).  It keeps its scratch in one static device array instead of
asking cudaMallocAsync for it.  Here it is called through the C ABI twice in
a row, on different inputs (the array keeps the previous call's contents),
and each result is compared with gdn_prefill's on the same inputs: the same
launch form and the same bits at bf16 (the fused cooperative form), within
the parity tests' tolerance at fp32.  A problem larger than the array is
rejected before anything runs.

This file is named to be collected last, and it passes both on its own in a
fresh process and after the rest of the suite."""
import ctypes

import numpy as np
import pytest
import torch

import gdn_inputs
from gdn_inputs import PrefillCase

pytestmark = pytest.mark.gpu
TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}
GDN_ERR_SCRATCH_LIMIT = 7


def _entry(lib):
    f = lib.gdn_prefill_noalloc
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    f.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i64, i32, i32, i32, i32, vp]
    f.restype = ctypes.c_int
    return f


def _ptr(t):
    return t.data_ptr() if t is not None else None


def _call(f, x, out, S_final, io):
    q = x["q"]
    cu = x["cu_seqlens"]
    if cu is None:
        N, seqlen = q.shape[0], q.shape[1]
    else:
        N, seqlen = cu.numel() - 1, q.shape[1]
    code = 1 if io == torch.bfloat16 else 0
    return f(_ptr(q), _ptr(x["k"]), _ptr(x["v"]), _ptr(x["alpha"]), _ptr(x["beta"]),
             _ptr(x["S0"]), _ptr(cu), _ptr(out), _ptr(S_final), N, seqlen, q.shape[2], 256, 256,
             code, torch.cuda.current_stream().cuda_stream)


def _last_form(gdn_lib):
    """The tensor-core prefill's last launch form (1: fused cooperative)."""
    f = gdn_lib.load().gdn_testing_last_prefill_form
    f.restype = ctypes.c_int32
    return int(f())


def _rel(a, b):
    a, b = a.double().cpu(), b.double().cpu()
    return float(torch.linalg.norm(a - b) / torch.linalg.norm(b))


@pytest.mark.parametrize("io", [torch.bfloat16, torch.float32])
def test_noalloc_matches_prefill_on_two_calls(gdn_lib, io):
    f = _entry(gdn_lib.load())
    cases = [PrefillCase("noalloc dense", [300, 300], H=6, io_dtype=io, seed=51),
             PrefillCase("noalloc varlen", [70, 0, 129, 5], H=6, io_dtype=io, seed=52,
                         varlen=True)]
    for case in cases:   # two calls in a row, different shapes and inputs
        x = {k: (v.cuda() if isinstance(v, torch.Tensor) else v)
             for k, v in gdn_inputs.make_prefill(case, device="cpu").items()}
        out = torch.full_like(x["v"], float("nan"))
        S_final = torch.full((len(case.lengths), case.H, 256, 256), float("nan"), device="cuda")
        assert _call(f, x, out, S_final, io) == 0
        assert gdn_lib.device_status() == 0
        form = _last_form(gdn_lib)
        ref_out, ref_S = gdn_lib.prefill(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["S0"],
                                         x["cu_seqlens"])
        assert gdn_lib.device_status() == 0
        if io == torch.bfloat16:
            assert form == 1 and _last_form(gdn_lib) == 1, case.name
            assert torch.equal(out, ref_out) and torch.equal(S_final, ref_S), case.name
        assert _rel(out.float(), ref_out.float()) <= TOL[io], case.name
        assert _rel(S_final, ref_S) <= TOL[io], case.name


def test_noalloc_rejects_problems_beyond_its_buffer(gdn_lib):
    f = _entry(gdn_lib.load())
    case = PrefillCase("too large", [8192], H=6, io_dtype=torch.bfloat16, seed=53)
    x = {k: (v.cuda() if isinstance(v, torch.Tensor) else v)
         for k, v in gdn_inputs.make_prefill(case, device="cpu").items()}
    out = torch.zeros_like(x["v"])
    before = gdn_lib.kernel_launches()
    assert _call(f, x, out, None, torch.bfloat16) == GDN_ERR_SCRATCH_LIMIT
    assert gdn_lib.kernel_launches() == before      # nothing was launched
    assert bool((out == 0).all())
