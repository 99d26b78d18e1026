"""The segmented form of the prefill (a sequence cut into segments that run
as independent chains, composed by a scan over their affine maps) against the
fp64 oracle, through the C ABI: gdn_prefill_scan with the segment count fixed
by the caller (dense and packed, bf16 and fp32, sequences shorter than one
segment and empty ones), and gdn_prefill taking the form by itself for a
sequence of 1024 chunks or more.  Tolerances as for the plain prefill: 2e-2
per (sequence, head) with bf16 I/O, 1e-4 with fp32 I/O.  Packing never changes
a result: every sequence equals its standalone run bit for bit."""
import numpy as np
import pytest
import torch

import gdn_inputs
import oracle
from gdn_inputs import PrefillCase
from test_parity_gpu import DEV, TOL, per_unit_errors, to_dev

pytestmark = pytest.mark.gpu


def _scan(gdn, xd, segments):
    out, sf = gdn.prefill_scan(xd["q"], xd["k"], xd["v"], xd["alpha"], xd["beta"], xd["S0"],
                               xd["cu_seqlens"], segments=segments)
    assert gdn.device_status() == 0
    return out, sf


def _oracle(x):
    o_ref, s_ref, _ = oracle.prefill(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["S0"],
                                     x["cu_seqlens"])
    return o_ref, s_ref


def _slice_seq(x, a, b, n):
    """Sequence n (tokens [a, b) of a packed batch) as a dense batch of one."""
    sl = lambda t: t[:, a:b].contiguous()
    S0 = x["S0"][n:n + 1].contiguous() if x["S0"] is not None else None
    return sl(x["q"]), sl(x["k"]), sl(x["v"]), sl(x["alpha"]), sl(x["beta"]), S0


@pytest.mark.parametrize("lens,H,dv,segments,s0", [
    ([700, 700], 2, 256, 3, 0.02),      # ragged last segment, two sequences
    ([1000], 1, 512, 4, 0.02),          # dv = 512: identity in the first dk rows
    ([640], 2, 256, 10, None),          # one chunk a segment, zero S0
])
def test_prefill_scan_matches_oracle(gdn_lib, lens, H, dv, segments, s0):
    case = PrefillCase("scan", lens, H=H, dv=dv, io_dtype=torch.bfloat16, s0_std=s0, seed=111)
    x = gdn_inputs.make_prefill(case, device="cpu")
    xd = to_dev(x)
    out, sf = _scan(gdn_lib, xd, segments)
    o_ref, s_ref = _oracle(x)
    eo, es = per_unit_errors(case, out, sf, o_ref, s_ref)
    assert eo <= 2e-2 and es <= 2e-2, (eo, es)


@pytest.mark.parametrize("io", [torch.bfloat16, torch.float32])
def test_prefill_scan_varlen_matches_oracle(gdn_lib, io):
    """Packed: sequences cut into 3 (1000 tokens: 16 chunks -> 6 + 6 + 4),
    one of 3 chunks (one chunk a segment), one of exactly one chunk and one
    of one token (never cut: a single chunk), an empty one (S_final = S0)."""
    lens = [1000, 0, 130, 64, 1, 700]
    case = PrefillCase("scan varlen", lens, H=2, io_dtype=io, seed=115, varlen=True)
    x = gdn_inputs.make_prefill(case, device="cpu")
    xd = to_dev(x)
    out, sf = _scan(gdn_lib, xd, 3)
    o_ref, s_ref = _oracle(x)
    eo, es = per_unit_errors(case, out, sf, o_ref, s_ref)
    assert eo <= TOL[io] and es <= TOL[io], (eo, es)
    assert torch.equal(sf[1], xd["S0"][1])
    # packing changes nothing: each sequence alone, cut the same way
    cu = [0] + list(np.cumsum(lens))
    for n in range(len(lens)):
        a, b = cu[n], cu[n + 1]
        q, k, v, al, be, S0 = _slice_seq(xd, a, b, n)
        o1, s1 = gdn_lib.prefill_scan(q, k, v, al, be, S0, segments=3)
        assert torch.equal(out[:, a:b], o1) and torch.equal(sf[n], s1[0]), n


@pytest.mark.parametrize("io", [torch.bfloat16, torch.float32])
def test_prefill_scan_one_segment_is_prefill(gdn_lib, io):
    case = PrefillCase("scan1", [300, 20, 129], H=2, io_dtype=io, seed=112, varlen=True)
    xd = to_dev(gdn_inputs.make_prefill(case, device="cpu"))
    out, sf = _scan(gdn_lib, xd, 1)
    o2, s2 = gdn_lib.prefill(xd["q"], xd["k"], xd["v"], xd["alpha"], xd["beta"], xd["S0"],
                             xd["cu_seqlens"])
    assert torch.equal(out, o2) and torch.equal(sf, s2)


@pytest.mark.parametrize("io,dv", [(torch.bfloat16, 256), (torch.bfloat16, 512),
                                   (torch.float32, 256)])
def test_prefill_scan_with_long_memory(gdn_lib, io, dv):
    """Weak decay (alpha in [0.995, 1)): a segment's start state still
    carries ~30 % of its weight to the segment's end, so the scan's
    start(j-1) A(j-1) term (A from the identity-start chains) decides the
    result; with the workloads' strong decay it is below fp32 resolution."""
    case = PrefillCase("scan long memory", [768], H=2, dv=dv, io_dtype=io, seed=113)
    x = gdn_inputs.make_prefill(case, device="cpu")
    g = torch.Generator().manual_seed(114)
    x["alpha"] = (1.0 - 0.005 * torch.rand(x["alpha"].shape, generator=g)).contiguous()
    xd = to_dev(x)
    out, sf = _scan(gdn_lib, xd, 4)
    o_ref, s_ref = _oracle(x)
    eo, es = per_unit_errors(case, out, sf, o_ref, s_ref)
    assert eo <= TOL[io] and es <= TOL[io], (eo, es)
    # the segment starts matter here: the oracle with every segment (4 x 192
    # tokens) restarted from zero is far off the true result
    cu = torch.tensor([0, 192, 384, 576, 768], dtype=torch.int32)
    o_cut, _, _ = oracle.prefill(x["q"][0], x["k"][0], x["v"][0], x["alpha"][0], x["beta"][0],
                                 None, cu)
    gap = np.linalg.norm(o_cut - o_ref[0]) / np.linalg.norm(o_ref[0])
    assert gap > 10 * max(eo, 1e-3), (gap, eo)


# ------------------------------------------------- the length rule inside gdn_prefill
LONG = 65536   # 1024 chunks: the shortest length cut by gdn_prefill is 65,473 tokens


@pytest.mark.parametrize("io", [torch.bfloat16, torch.float32])
def test_prefill_cuts_a_long_sequence_by_itself(gdn_lib, io):
    """One 64K-token sequence (1024 chunks -> 7 segments of 147 chunks):
    gdn_prefill equals gdn_prefill_scan with 7 segments bit for bit, agrees
    with the uncut chain (segments = 1) and matches the oracle within the
    tolerance of the I/O type.  (With the workloads' decay, alpha around 0.5,
    a start state's weight falls below fp32 resolution within a few hundred
    tokens, so cut and uncut chains come out alike to the bit; the tests with
    long memory above are the ones where the scan's A terms count.)"""
    case = PrefillCase("long", [LONG], H=1, io_dtype=io, seed=116, s0_std=0.02)
    x = gdn_inputs.make_prefill(case, device="cpu")
    xd = to_dev(x)
    args = (xd["q"], xd["k"], xd["v"], xd["alpha"], xd["beta"], xd["S0"])
    out, sf = gdn_lib.prefill(*args)
    assert gdn_lib.device_status() == 0
    o7, s7 = gdn_lib.prefill_scan(*args, segments=7)
    assert torch.equal(out, o7) and torch.equal(sf, s7)
    o1, s1 = gdn_lib.prefill_scan(*args, segments=1)
    d = (out.float() - o1.float()).norm() / o1.float().norm()
    assert float(d) <= TOL[io] and float((sf - s1).norm() / s1.norm()) <= TOL[io]
    o_ref, s_ref = _oracle(x)
    eo, es = per_unit_errors(case, out, sf, o_ref, s_ref)
    assert eo <= TOL[io] and es <= TOL[io], (eo, es)


def test_prefill_long_sequence_packed_is_bitwise(gdn_lib):
    """A packed batch holding a 64K-token sequence takes the segmented form
    for the whole batch: the long sequence is cut exactly as when alone, and
    the short ones (and an empty one) run the plain kernels with the bits of
    their standalone runs."""
    lens = [3000, LONG, 0, 5000, 65472]   # 65,472 tokens: 1023 chunks, never cut
    case = PrefillCase("long packed", lens, H=1, io_dtype=torch.bfloat16, seed=117, varlen=True)
    xd = to_dev(gdn_inputs.make_prefill(case, device="cpu"))
    out, sf = gdn_lib.prefill(xd["q"], xd["k"], xd["v"], xd["alpha"], xd["beta"], xd["S0"],
                              xd["cu_seqlens"])
    assert gdn_lib.device_status() == 0
    cu = [0] + list(np.cumsum(lens))
    for n in range(len(lens)):
        a, b = cu[n], cu[n + 1]
        o1, s1 = gdn_lib.prefill(*_slice_seq(xd, a, b, n))
        assert torch.equal(out[:, a:b], o1) and torch.equal(sf[n], s1[0]), n
    assert torch.equal(sf[2], xd["S0"][2])
