"""Pins the tensor-core building blocks (tcgen05.mma with bf16 operands in
128-byte-swizzled shared-memory images, matrix descriptors, TMA tensor copies,
TMEM read-back) against a plain fp32 matmul of the same bf16 inputs, for every
operand-major combination the kernels use."""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu


def _fn(lib):
    f = lib.gdn_testing_umma_gemm
    vp, i32, u32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint32
    f.argtypes = [vp, vp, vp, i32, i32, i32, i32, u32, u32, u32, u32, i32, vp]
    f.restype = ctypes.c_int
    return f


def _run(f, A, B, a_mn, b_mn, a_desc, b_desc, tma=0):
    N, K = B.shape
    D = torch.full((128, N), float("nan"), device="cuda")
    rc = f(A.data_ptr(), B.data_ptr(), D.data_ptr(), N, K, a_mn, b_mn, a_desc[0], a_desc[1],
           b_desc[0], b_desc[1], tma, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return rc, D


def _desc(mn, R, K):
    """Convention the kernels use: K-major -> (LBO unused = 16, SBO = 1024 per
    8-row group); MN-major -> (LBO = bytes between 64-element MN blocks,
    SBO = 1024 per 8-row K group)."""
    return (K * 128, 1024) if mn else (16, 1024)


@pytest.mark.parametrize("N,K", [(64, 64), (64, 256), (256, 64), (128, 128), (256, 256)])
def test_umma_operand_majors(gdn_lib, N, K):
    f = _fn(gdn_lib.load())
    g = torch.Generator(device="cuda").manual_seed(N * 1000 + K)
    A = torch.randn(128, K, device="cuda", generator=g).to(torch.bfloat16)
    B = torch.randn(N, K, device="cuda", generator=g).to(torch.bfloat16)
    ref = A.float() @ B.float().T
    report = []
    for a_mn in (0, 1):
        for b_mn in (0, 1):
            rc, D = _run(f, A, B, a_mn, b_mn, _desc(a_mn, 128, K), _desc(b_mn, N, K))
            err = float((D - ref).abs().max() / ref.abs().max()) if rc == 0 else float("inf")
            report.append((a_mn, b_mn, rc, err))
            # the swapped LBO/SBO reading of the MN-major descriptor, for diagnosis
            if a_mn or b_mn:
                swap = lambda mn, R: (1024, K * 128) if mn else (16, 1024)
                rc2, D2 = _run(f, A, B, a_mn, b_mn, swap(a_mn, 128), swap(b_mn, N))
                err2 = float((D2 - ref).abs().max() / ref.abs().max()) if rc2 == 0 else None
                report.append((a_mn, b_mn, "swapped", rc2, err2))
    print(f"N={N} K={K}:", report)
    assert gdn_lib.device_status() == 0
    for row in report:
        if row[2] == "swapped":
            continue
        assert row[2] == 0 and row[3] < 1e-5, report


@pytest.mark.parametrize("N,K", [(64, 256), (256, 128)])
def test_umma_tma_staged_operand(gdn_lib, N, K):
    f = _fn(gdn_lib.load())
    g = torch.Generator(device="cuda").manual_seed(7 + N + K)
    A = torch.randn(128, K, device="cuda", generator=g).to(torch.bfloat16)
    B = torch.randn(N, K, device="cuda", generator=g).to(torch.bfloat16)
    ref = A.float() @ B.float().T
    rc, D = _run(f, A, B, 0, 1, _desc(0, 128, K), _desc(1, N, K), tma=1)
    assert rc == 0 and gdn_lib.device_status() == 0
    assert float((D - ref).abs().max() / ref.abs().max()) < 1e-5


@pytest.mark.parametrize("N,K", [(64, 256), (256, 64), (128, 128)])
@pytest.mark.parametrize("b_mn", [0, 1])
def test_umma_a_operand_in_tmem(gdn_lib, N, K, b_mn):
    """A operand read from tensor memory (row per lane, K pairs per column)."""
    f = _fn(gdn_lib.load())
    g = torch.Generator(device="cuda").manual_seed(3 + N + K + b_mn)
    A = torch.randn(128, K, device="cuda", generator=g).to(torch.bfloat16)
    B = torch.randn(N, K, device="cuda", generator=g).to(torch.bfloat16)
    ref = A.float() @ B.float().T
    rc, D = _run(f, A, B, 0, b_mn, _desc(0, 128, K), _desc(b_mn, N, K), tma=2)
    assert rc == 0 and gdn_lib.device_status() == 0
    assert float((D - ref).abs().max() / ref.abs().max()) < 1e-5
