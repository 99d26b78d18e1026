"""gdn_prefill_scan (a long sequence cut into segments that run as
independent chains, composed by a scan over their affine maps) against the
fp64 oracle, through the C ABI: the bf16 tolerance 2e-2 per (sequence, head)
on out and S_final; segments = 1 is gdn_prefill itself, bit for bit."""
import numpy as np
import pytest
import torch

import gdn_inputs
import oracle
from gdn_inputs import PrefillCase
from test_parity_gpu import DEV, per_unit_errors

pytestmark = pytest.mark.gpu


def _run(gdn, case, segments):
    x = gdn_inputs.make_prefill(case, device="cpu")
    xd = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    out, sf = gdn.prefill_scan(xd["q"], xd["k"], xd["v"], xd["alpha"], xd["beta"], xd["S0"],
                               segments=segments)
    assert gdn.device_status() == 0
    return x, xd, out, sf


@pytest.mark.parametrize("lens,H,dv,segments,s0", [
    ([700, 700], 2, 256, 3, 0.02),      # ragged last segment, two sequences
    ([1000], 1, 512, 4, 0.02),          # dv = 512: identity in the first dk rows
    ([640], 2, 256, 10, None),          # one chunk a segment, zero S0
])
def test_prefill_scan_matches_oracle(gdn_lib, lens, H, dv, segments, s0):
    case = PrefillCase("scan", lens, H=H, dv=dv, io_dtype=torch.bfloat16, s0_std=s0, seed=111)
    x, xd, out, sf = _run(gdn_lib, case, segments)
    o_ref, s_ref, _ = oracle.prefill(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["S0"])
    eo, es = per_unit_errors(case, out, sf, o_ref, s_ref)
    assert eo <= 2e-2 and es <= 2e-2, (eo, es)
    # and it agrees with the single-chain prefill to the same order
    o2, s2 = gdn_lib.prefill(xd["q"], xd["k"], xd["v"], xd["alpha"], xd["beta"], xd["S0"])
    assert gdn_lib.device_status() == 0
    d = (out.float() - o2.float()).norm() / o2.float().norm()
    assert float(d) <= 2e-2


def test_prefill_scan_one_segment_is_prefill(gdn_lib):
    case = PrefillCase("scan1", [300], H=2, io_dtype=torch.bfloat16, seed=112)
    x, xd, out, sf = _run(gdn_lib, case, 1)
    o2, s2 = gdn_lib.prefill(xd["q"], xd["k"], xd["v"], xd["alpha"], xd["beta"], xd["S0"])
    assert torch.equal(out, o2) and torch.equal(sf, s2)


@pytest.mark.parametrize("dv", [256, 512])
def test_prefill_scan_with_long_memory(gdn_lib, dv):
    """Weak decay (alpha in [0.995, 1)): a segment's start state still
    carries ~30 % of its weight to the segment's end, so the scan's
    start(j-1) A(j-1) term (A from the identity-start pass) decides the
    result; with the workloads' strong decay it is below fp32 resolution."""
    case = PrefillCase("scan long memory", [768], H=2, dv=dv, io_dtype=torch.bfloat16,
                       seed=113)
    x = gdn_inputs.make_prefill(case, device="cpu")
    g = torch.Generator().manual_seed(114)
    x["alpha"] = (1.0 - 0.005 * torch.rand(x["alpha"].shape, generator=g)).contiguous()
    xd = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    out, sf = gdn_lib.prefill_scan(xd["q"], xd["k"], xd["v"], xd["alpha"], xd["beta"], xd["S0"],
                                   segments=4)
    assert gdn_lib.device_status() == 0
    o_ref, s_ref, _ = oracle.prefill(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["S0"])
    eo, es = per_unit_errors(case, out, sf, o_ref, s_ref)
    assert eo <= 2e-2 and es <= 2e-2, (eo, es)
    # the segment starts matter here: the oracle with every segment (4 x 192
    # tokens) restarted from zero is far off the true result
    cu = torch.tensor([0, 192, 384, 576, 768], dtype=torch.int32)
    o_cut, _, _ = oracle.prefill(x["q"][0], x["k"][0], x["v"][0], x["alpha"][0], x["beta"][0],
                                 None, cu)
    gap = np.linalg.norm(o_cut - o_ref[0]) / np.linalg.norm(o_ref[0])
    assert gap > 10 * max(eo, 1e-3), (gap, eo)
