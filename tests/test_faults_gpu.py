"""Fault tests without a GPU fault: the library's bounded waits (an mbarrier
try-wait, a ready-flag poll) run on something that never completes, give up
after a short limit, record GDN_ERR_TIMEOUT in the device status word, and
leave the context usable -- a prefill right after still matches the oracle."""
import ctypes

import pytest
import torch

import gdn_inputs
from test_parity_gpu import check_case

pytestmark = pytest.mark.gpu
GDN_ERR_TIMEOUT = 5


def _wait(gdn, which, limit_ns):
    f = gdn.load().gdn_testing_bounded_wait
    f.argtypes = [ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p]
    f.restype = ctypes.c_int
    return f(which, limit_ns, torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("which", [0, 1])
def test_bounded_wait_times_out_and_context_survives(gdn_lib, which):
    assert gdn_lib.device_status() == 0
    assert _wait(gdn_lib, which, 20_000_000) == 0          # 20 ms
    assert gdn_lib.device_status() == GDN_ERR_TIMEOUT        # recorded ...
    assert gdn_lib.device_status() == 0                      # ... and cleared by the read
    check_case(gdn_lib, gdn_inputs.PrefillCase("after timeout", [100, 30], H=2, seed=33,
                                               varlen=True))
