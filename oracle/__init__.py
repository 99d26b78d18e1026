"""fp64 CPU oracle for the gated delta rule -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The GPU
library never imports, links or calls it, and it shares no code with the GPU
library.

The arithmetic lives in ``gdn_oracle.c`` (plain C, fp64, one token at a time,
following "Long-Context Aware Upcycling: A New Frontier for Hybrid LLM
Scaling", Appendix A.3, Eq. 16-19).  This module only compiles it with gcc and
marshals arrays through ctypes.

Inputs are taken exactly as the GPU path receives them (fp32 or raw bfloat16
for q, k, v; fp32 alpha, beta; fp32/fp64 states) and widened to fp64 exactly.
Layouts follow the library boundary:
  q, k [T_total, H, dk];  v [T_total, H, dv];  alpha, beta [T_total, H];
  S0, S_final [N, H, dv, dk];  cu_seqlens [N+1].
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_LIB_PATH = os.path.join(_HERE, f"liboracle_{platform.machine()}.so")
_lib = None

F32, BF16 = 0, 1


def build(force: bool = False) -> str:
    """Compile the oracle into a shared library beside this file (gcc, -O2,
    OpenMP when available).  Returns the library path."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", _SRC, "-o", _LIB_PATH + ".tmp", "-lm"]
    try:
        subprocess.run(base[:3] + ["-fopenmp"] + base[3:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        vp, i32, i64p = ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(ctypes.c_int64)
        lib.oracle_gdn_prefill.argtypes = [vp, vp, vp, i32, vp, vp, vp, i64p, i32, i32, i32, i32,
                                           vp, vp, i32]
        lib.oracle_gdn_prefill.restype = i32
        lib.oracle_gdn_decode_step.argtypes = [vp, vp, vp, i32, vp, vp, vp, i32, i32, i32, i32,
                                               vp, i32]
        lib.oracle_gdn_decode_step.restype = i32
        lib.oracle_max_threads.restype = i32
        _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def _as_io(x):
    """torch tensor or numpy array -> (contiguous numpy array, dtype code)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.bfloat16:
                return x.view(torch.int16).numpy().view(np.uint16), BF16
            if x.dtype == torch.float32:
                return x.numpy(), F32
            raise TypeError(f"unsupported io dtype {x.dtype}")
    except ImportError:  # pragma: no cover
        pass
    x = np.ascontiguousarray(x)
    if x.dtype == np.float32:
        return x, F32
    if x.dtype == np.uint16:
        return x, BF16
    raise TypeError(f"unsupported io dtype {x.dtype}")


def _as(x, dtype):
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(x, dtype=dtype)


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def prefill(q, k, v, alpha, beta, S0=None, cu_seqlens=None, nthreads: int = 0):
    """Run the token recurrence over every (sequence, head).

    q, k: [B, T, H, dk] or [T_total, H, dk]; v likewise with dv.
    alpha, beta: [B, T, H] or [T_total, H] fp32.  S0: [N, H, dv, dk] or None.
    cu_seqlens: None (dense [B, T]) or N+1 offsets.
    Returns (out fp64 shaped like v, S_final fp64 [N, H, dv, dk], threads used).
    """
    qa, dt = _as_io(q)
    ka, dt_k = _as_io(k)
    va, dt_v = _as_io(v)
    assert dt == dt_k == dt_v, "q, k, v must share one dtype"
    out_shape = va.shape
    H, dk = qa.shape[-2], qa.shape[-1]
    dv = va.shape[-1]
    if cu_seqlens is None:
        B, T = (qa.shape[0], qa.shape[1]) if qa.ndim == 4 else (1, qa.shape[0])
        cu = np.arange(B + 1, dtype=np.int64) * T
    else:
        cu = _as(cu_seqlens, np.int64)
    N = len(cu) - 1
    a = _as(alpha, np.float32)
    b = _as(beta, np.float32)
    s0 = _as(S0, np.float64) if S0 is not None else None
    if s0 is not None:
        assert s0.shape == (N, H, dv, dk)
    out = np.zeros(out_shape, dtype=np.float64)
    sf = np.zeros((N, H, dv, dk), dtype=np.float64)
    used = _load().oracle_gdn_prefill(
        _ptr(qa), _ptr(ka), _ptr(va), dt, _ptr(a), _ptr(b), _ptr(s0),
        cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), N, H, dk, dv, _ptr(out), _ptr(sf),
        int(nthreads))
    if used < 0:
        raise MemoryError("oracle allocation failed")
    return out, sf, used


def decode_step(q, k, v, alpha, beta, S, nthreads: int = 0):
    """One token per sequence against the cached fp64 state S [N, H, dv, dk],
    which is updated in place.  q, k: [N, H, dk]; v: [N, H, dv];
    alpha, beta: [N, H].  Returns out fp64 [N, H, dv]."""
    qa, dt = _as_io(q)
    ka, _ = _as_io(k)
    va, _ = _as_io(v)
    N, H, dk = qa.shape
    dv = va.shape[-1]
    assert isinstance(S, np.ndarray) and S.dtype == np.float64 and S.flags.c_contiguous
    assert S.shape == (N, H, dv, dk)
    a = _as(alpha, np.float32)
    b = _as(beta, np.float32)
    out = np.zeros((N, H, dv), dtype=np.float64)
    used = _load().oracle_gdn_decode_step(_ptr(qa), _ptr(ka), _ptr(va), dt, _ptr(a), _ptr(b),
                                          _ptr(S), N, H, dk, dv, _ptr(out), int(nthreads))
    if used < 0:
        raise MemoryError("oracle allocation failed")
    return out
