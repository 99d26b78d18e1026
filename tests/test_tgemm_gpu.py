"""The backward's batched tensor-core GEMM (tcgen05 kind::tf32, through the
testing entry point gdn_testing_tgemm) against a plain fp64 matmul of the
same fp32 arrays: every transposition of A and B, N and K in {64, 256}, the
column scale, alpha, beta * Cin and both masks, over more units than one
wave of CTAs (so each CTA walks several units and alternates its stages).

Tolerance: relative Frobenius error per unit <= 2e-3 (each operand rounds to
tf32, 2^-11 relative; fp32 accumulation), and masked entries exactly zero."""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _fn(gdn_lib):
    f = gdn_lib.load().gdn_testing_tgemm
    vp, i32, i64, fl = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    f.argtypes = [vp, i64, i32, i32, vp, i64, i32, i32, vp, fl, vp, i64, i32, vp, i64, i32, i32,
                  fl, i32, i64, i32, i32, vp]
    f.restype = ctypes.c_int
    return f


def _tile(M):
    """[units][R][256] -> the tiled state layout: (r, c) at ((c / 4) R + r) 4 + c % 4."""
    u, R, W = M.shape
    return M.reshape(u, R, W // 4, 4).permute(0, 2, 1, 3).contiguous()


def _run(gdn_lib, tA, tB, N, K, batch, alpha=1.0, beta=0.0, with_cin=False, with_col=False,
         mask=0, seed=0, tiled=False, b_bf16=False):
    g = torch.Generator().manual_seed(seed)
    A = torch.randn((batch, K, 64) if tA else (batch, 64, K), generator=g)
    B = torch.randn((batch, N, K) if tB else (batch, K, N), generator=g)
    if b_bf16:   # the reference takes the bf16 values the kernel reads
        B = B.to(torch.bfloat16).float()
    Bstore = _tile(B) if tiled else B
    if b_bf16:
        Bstore = Bstore.to(torch.bfloat16)
    Cin = torch.randn((batch, 64, N), generator=g) if with_cin else None
    col = torch.rand((batch, N), generator=g) + 0.5 if with_col else None
    Ad, Bd = A.to(DEV), Bstore.to(DEV)
    Cind = Cin.to(DEV) if Cin is not None else None
    cold = col.to(DEV) if col is not None else None
    C = torch.full((batch, 64, N), float("nan"), device=DEV)
    rc = _fn(gdn_lib)(Ad.data_ptr(), A[0].numel(), A.shape[2], int(tA), Bd.data_ptr(),
                      B[0].numel(), B.shape[2], int(tB),
                      Cind.data_ptr() if Cind is not None else None, beta, C.data_ptr(),
                      64 * N, N, cold.data_ptr() if cold is not None else None, N, N, K, alpha,
                      mask, batch, B.shape[1] if tiled else 0, int(b_bf16),
                      torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rc == 0 and gdn_lib.device_status() == 0
    Ap = A.double().transpose(1, 2) if tA else A.double()
    Bp = B.double().transpose(1, 2) if tB else B.double()
    ref = alpha * torch.bmm(Ap, Bp)
    if col is not None:
        ref = ref * col.double()[:, None, :]
    if Cin is not None:
        ref = ref + beta * Cin.double()
    m = torch.arange(64)[:, None]
    n = torch.arange(N)[None, :]
    keep = torch.ones(64, N, dtype=torch.bool)
    if mask == 1:
        keep = n <= m
    elif mask == 2:
        keep = n < m
    ref = ref * keep
    got = C.cpu().double()
    assert torch.all(got[:, ~keep] == 0)
    err = (got - ref).flatten(1).norm(dim=1) / ref.flatten(1).norm(dim=1)
    return float(err.max())


@pytest.mark.parametrize("tA", [0, 1])
@pytest.mark.parametrize("tB", [0, 1])
@pytest.mark.parametrize("N,K", [(64, 64), (64, 256), (256, 64), (256, 256)])
def test_tgemm_transpositions_and_shapes(gdn_lib, tA, tB, N, K):
    assert _run(gdn_lib, tA, tB, N, K, batch=37, seed=N + K + 2 * tA + tB) <= 2e-3


@pytest.mark.parametrize("tB", [0, 1])
def test_tgemm_tiled_state_operand(gdn_lib, tB):
    """B in the backward's tiled state layout (the chunk states and dS' at
    dv = 256): B' = the 256 x 256 matrix (dO S, -dU S, U dS') or its transpose
    (U~ - W S^T, with alpha = -1 and Cin)."""
    if tB:
        err = _run(gdn_lib, 0, 1, 256, 256, batch=333, alpha=-1.0, beta=1.0, with_cin=True,
                   seed=21, tiled=True)
    else:
        err = _run(gdn_lib, 0, 0, 256, 256, batch=333, seed=22, tiled=True)
    assert err <= 2e-3


@pytest.mark.parametrize("tB", [0, 1])
def test_tgemm_tiled_bf16_state_operand(gdn_lib, tB):
    """B in the tiled layout with bf16 elements (the backward's chunk-start
    states at bf16 I/O), widened exactly while staging: the same shapes as
    the fp32 tiled case, against the product of the bf16 values."""
    if tB:
        err = _run(gdn_lib, 0, 1, 256, 256, batch=333, alpha=-1.0, beta=1.0, with_cin=True,
                   seed=23, tiled=True, b_bf16=True)
    else:
        err = _run(gdn_lib, 0, 0, 256, 256, batch=333, seed=24, tiled=True, b_bf16=True)
    assert err <= 2e-3


def test_tgemm_many_units_epilogue_terms(gdn_lib):
    """700 units over at most 2 CTAs a SM: alpha, the column scale and
    beta * Cin (C = Cin in place is how the backward accumulates)."""
    assert _run(gdn_lib, 0, 0, 256, 256, batch=700, alpha=-1.0, beta=1.0, with_cin=True,
                with_col=True, seed=5) <= 2e-3


@pytest.mark.parametrize("mask", [1, 2])
def test_tgemm_masks(gdn_lib, mask):
    assert _run(gdn_lib, 0, 1, 64, 256, batch=50, alpha=0.5, mask=mask, seed=6 + mask) <= 2e-3


def test_tgemm_in_place_accumulate(gdn_lib):
    """C = 1 * (A B) + 1 * C with Cin and C the same array (every element is
    read by the thread that writes it, once)."""
    g = torch.Generator().manual_seed(9)
    batch, N, K = 333, 64, 256
    A = torch.randn((batch, 64, K), generator=g)
    B = torch.randn((batch, N, K), generator=g)
    C0 = torch.randn((batch, 64, N), generator=g)
    Ad, Bd, Cd = A.to(DEV), B.to(DEV), C0.to(DEV)
    rc = _fn(gdn_lib)(Ad.data_ptr(), 64 * K, K, 0, Bd.data_ptr(), N * K, K, 1, Cd.data_ptr(), 1.0,
                      Cd.data_ptr(), 64 * N, N, None, 0, N, K, 1.0, 0, batch, 0, 0,
                      torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rc == 0 and gdn_lib.device_status() == 0
    ref = torch.bmm(A.double(), B.double().transpose(1, 2)) + C0.double()
    err = float(((Cd.cpu().double() - ref).norm() / ref.norm()))
    assert err <= 2e-3


def test_tgemm_rejects_unsupported_shapes(gdn_lib):
    f = _fn(gdn_lib)
    buf = torch.zeros(64 * 256, device=DEV)
    p = buf.data_ptr()
    s = torch.cuda.current_stream().cuda_stream
    assert f(p, 0, 256, 0, p, 0, 128, 0, None, 0.0, p, 0, 128, None, 0, 128, 256, 1.0, 0, 1, 0, 0, s) != 0
    assert f(p, 0, 130, 0, p, 0, 256, 0, None, 0.0, p, 0, 256, None, 0, 256, 128, 1.0, 0, 1, 0, 0, s) != 0
    assert f(p, 0, 256, 0, p, 0, 256, 0, None, 0.0, p, 0, 256, None, 0, 256, 256, 1.0, 3, 1, 0, 0, s) != 0
    # a tiled B must be 256 columns wide with R = K (or N when transposed)
    assert f(p, 0, 64, 0, p, 0, 64, 0, None, 0.0, p, 0, 64, None, 0, 64, 64, 1.0, 0, 1, 64, 0, s) != 0
    # bf16 elements only for a tiled B
    assert f(p, 0, 256, 0, p, 0, 256, 0, None, 0.0, p, 0, 256, None, 0, 256, 256, 1.0, 0, 1, 0, 1, s) != 0
    # the transposed A and a row-major B stored [K][N] are read 32 bytes a
    # lane: lda / ldb multiples of 8 floats, addresses and unit strides 32-byte
    # aligned (all rejected before any launch)
    GDN_ERR_ALIGNMENT = 3
    assert f(p, 0, 68, 1, p, 0, 64, 1, None, 0.0, p, 0, 64, None, 0, 64, 64, 1.0, 0, 1, 0, 0, s) != 0
    assert f(p, 0, 64, 0, p, 0, 68, 0, None, 0.0, p, 0, 64, None, 0, 64, 64, 1.0, 0, 1, 0, 0, s) != 0
    q = p + 16   # 16-byte but not 32-byte aligned
    assert f(q, 0, 64, 1, p, 0, 64, 1, None, 0.0, p, 0, 64, None, 0, 64, 64, 1.0, 0, 1, 0, 0,
             s) == GDN_ERR_ALIGNMENT
    assert f(p, 0, 64, 0, q, 0, 64, 0, None, 0.0, p, 0, 64, None, 0, 64, 64, 1.0, 0, 1, 0, 0,
             s) == GDN_ERR_ALIGNMENT
    assert f(p, 4, 64, 1, p, 0, 64, 1, None, 0.0, p, 0, 64, None, 0, 64, 64, 1.0, 0, 2, 0, 0,
             s) == GDN_ERR_ALIGNMENT
