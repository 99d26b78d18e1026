"""The tensor-core prefill's per-chunk kernel, checked on its own: decode the
128-byte-swizzled operand images it leaves behind (W, Q^, P^, U~^T and the
decay factors) and
compare them with the fp64 chunk algebra computed from the same bf16 inputs.
A layout or descriptor mistake shows up here as a wrong matrix, before the
state pass mixes everything together."""
import ctypes

import numpy as np
import pytest
import torch

import gdn_inputs
from gdn_inputs import PrefillCase

pytestmark = pytest.mark.gpu
C = 64


def _hook(lib):
    f = lib.gdn_testing_prefill_prep
    vp = ctypes.c_void_p
    f.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32, vp,
                  ctypes.c_size_t, vp]
    f.restype = ctypes.c_int
    lib.gdn_testing_prefill_image_stride.restype = ctypes.c_size_t
    return f, int(lib.gdn_testing_prefill_image_stride())


def _rows(buf, nrows):
    """[nrows*128] bytes of swizzled rows -> [nrows, 64] float64 values."""
    u16 = buf[: nrows * 128].view(np.uint16).reshape(nrows, 8, 8)
    perm = np.arange(8)[None, :] ^ (np.arange(nrows) % 8)[:, None]
    logical = np.take_along_axis(u16, perm[:, :, None].repeat(8, axis=2), axis=1)
    return (logical.reshape(nrows, 64).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _blocks(img, off):
    return np.concatenate([_rows(img[off + b * 8192:off + (b + 1) * 8192], 64)
                           for b in range(4)], axis=1)    # [64][256]


def _wq(img, off):
    """W (off 0) or Q^ (off 8192) from the interleaved [W_0 Q^_0 W_1 Q^_1 ...]
    blocks of 64 rows c each -> [256 c][64 r]."""
    return np.concatenate([_rows(img[b * 16384 + off:b * 16384 + off + 8192], 64)
                           for b in range(4)])


def _decode(img):
    W = _wq(img, 0).T                                     # [64 r][256 c]
    Q = _wq(img, 8192).T                                  # [64 r][256 c]
    P = _rows(img[65536:65536 + 8192], 64)                # [64][64]
    half = 16896                                          # U~^T rows of one half + decay block
    Ut = np.concatenate([_rows(img[73728 + h * half:73728 + h * half + 16384], 128)
                         for h in range(2)]).T            # [64 r][256 i]
    blocks = [img[73728 + h * half + 16384:73728 + (h + 1) * half].view(np.float32) for h in range(2)]
    assert np.array_equal(blocks[0], blocks[1])
    d, G = blocks[0][:64].astype(np.float64), blocks[0][64:].astype(np.float64)
    return W, Q, P, Ut, G, d


def _model_chunk(q, k, v, a, b):
    L = q.shape[0]
    G = np.cumsum(np.log(a))
    g = np.exp(G)
    Gam = np.exp(np.minimum(G[:, None] - G[None, :], 0.0))
    A = np.tril(b[:, None] * Gam * (k @ k.T), -1)
    T = np.linalg.inv(np.eye(L) + A)
    W = T @ ((b * g)[:, None] * k)
    Ut = T @ (b[:, None] * v)
    P = np.tril(Gam * (q @ k.T)) / 16.0
    Qh = g[:, None] * q / 16.0
    return W, Qh, P, Ut, G


def rel(x, y):
    return float(np.linalg.norm(x - y) / max(np.linalg.norm(y), 1e-30))


@pytest.mark.parametrize("lens,varlen", [([150], False), ([64, 3, 130], True)])
def test_prep_images_match_chunk_algebra(gdn_lib, lens, varlen):
    f, stride = _hook(gdn_lib.load())
    H = 2
    case = PrefillCase("prep", lens, H=H, seed=11, varlen=varlen)
    x = gdn_inputs.make_prefill(case, device="cpu")
    dev = {k_: (v_.cuda() if isinstance(v_, torch.Tensor) else v_) for k_, v_ in x.items()}
    T_tot = sum(lens)
    if varlen:
        N, seqlen, max_chunks = len(lens), T_tot, (T_tot + 63 * len(lens)) // 64
    else:
        N, seqlen, max_chunks = 1, lens[0], (lens[0] + 63) // 64
    buf = torch.zeros(max_chunks * H * stride, dtype=torch.uint8, device="cuda")
    rc = f(dev["q"].data_ptr(), dev["k"].data_ptr(), dev["v"].data_ptr(), dev["alpha"].data_ptr(),
           dev["beta"].data_ptr(), dev["cu_seqlens"].data_ptr() if varlen else None, N, seqlen, H,
           buf.data_ptr(), buf.numel(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0 and gdn_lib.device_status() == 0
    img_all = buf.cpu().numpy()
    f64 = lambda t: t.float().double().numpy().reshape(-1, H, t.shape[-1])
    q, k, v = f64(x["q"]), f64(x["k"]), f64(x["v"])
    al = x["alpha"].double().numpy().reshape(-1, H)
    be = x["beta"].double().numpy().reshape(-1, H)
    ci = 0
    worst = {}
    starts = np.concatenate([[0], np.cumsum(lens)])
    for n, Ln in enumerate(lens):
        for c0 in range(0, Ln, C):
            t0 = starts[n] + c0
            L = min(C, Ln - c0)
            for h in range(H):
                img = img_all[(ci * H + h) * stride:(ci * H + h + 1) * stride]
                W, Q, P, Ut, G, d = _decode(img)
                sl = slice(t0, t0 + L)
                Wm, Qm, Pm, Um, Gm = _model_chunk(q[sl, h], k[sl, h], v[sl, h], al[sl, h],
                                                  be[sl, h])
                dm = np.exp(Gm[-1] - Gm)
                errs = dict(W=rel(W[:L], Wm), Q=rel(Q[:L], Qm), P=rel(P[:L, :L], Pm),
                            U=rel(Ut[:L], Um), G=float(np.abs(G[:L] - Gm).max()),
                            d=float(np.abs(d[:L] - dm).max()))
                assert np.all(d[L:] == 0)
                for key, val in errs.items():
                    worst[key] = max(worst.get(key, 0.0), val)
                # rows past the chunk's end must not write anything
                assert np.all(W[L:] == 0) and np.all(Ut[L:] == 0) and np.all(Q[L:] == 0)
                assert np.all(P[L:] == 0)
            ci += 1
    print("worst relative errors:", worst)
    assert worst["W"] < 2e-2 and worst["U"] < 2e-2 and worst["P"] < 2e-2
    assert worst["Q"] < 1e-2
    assert worst["G"] < 1e-4 and worst["d"] < 1e-4
