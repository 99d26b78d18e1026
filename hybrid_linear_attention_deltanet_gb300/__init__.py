"""GB300-native Gated DeltaNet (gated delta rule) sequence mixer.

Thin ctypes binding over the C ABI in ``include/gdn.h``: it checks tensor
shapes, dtypes and devices, reads sizes off the tensors, and passes raw device
pointers and the current CUDA stream.  Every step of the computation runs in
the library's CUDA kernels; there is no CPU or PyTorch fallback, and calls
raise when the compiled library is missing.

    out, S_final = prefill(q, k, v, alpha, beta, S0=None, cu_seqlens=None)
    out, S_final = prefill(..., workspace=ws)  # caller-owned scratch, nothing allocated
    out = decode_step(q, k, v, alpha, beta, S)          # S updated in place
    grads = prefill_backward(q, k, v, alpha, beta, dout, S0, dS_final)   # training
    x = prepare(qkv, conv_w, a_raw, b_raw, A_log, dt_bias, heads)   # -> q, k, v, alpha, beta
    y = output_norm_gate(out, g, w)                     # Eq. 20 read-out
    y = decode_layer_step(qkv, conv_w, a_raw, b_raw, A_log, dt_bias, conv_state, S, g, w)

Recurrence (Appendix A.3, Eq. 16-19 of "Long-Context Aware Upcycling"):
S_t = alpha_t S_{t-1}(I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
o_t = S_t q_t / sqrt(dk), with the state stored as [dv, dk].
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_NAME = "libgdn_gb300.so"
_lib = None

GDN_F32, GDN_BF16 = 0, 1
_STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "alignment",
           4: "CUDA error", 5: "device timeout", 6: "malformed cu_seqlens"}


class GDNError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__(f"{fn} failed with status {code} ({_STATUS.get(code, 'unknown')})")
        self.code = code


def lib_path() -> str:
    return os.path.join(_HERE, LIB_NAME)


def load():
    """Load the compiled library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = lib_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{LIB_NAME} is not built; run __graft_entry__.build() "
                           f"(or python -m hybrid_linear_attention_deltanet_gb300._build)")
    lib = ctypes.CDLL(path)
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    lib.gdn_prefill.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i64, i32, i32, i32, i32,
                                vp]
    lib.gdn_prefill.restype = ctypes.c_int
    lib.gdn_decode_step.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp]
    lib.gdn_decode_step.restype = ctypes.c_int
    lib.gdn_get_device_status.argtypes = [vp]
    lib.gdn_get_device_status.restype = ctypes.c_int
    lib.gdn_version.restype = ctypes.c_char_p
    lib.gdn_status_string.argtypes = [ctypes.c_int]
    lib.gdn_status_string.restype = ctypes.c_char_p
    lib.gdn_kernel_launches.restype = ctypes.c_uint64
    lib.gdn_prefill_path.argtypes = [ctypes.c_int32]
    lib.gdn_prefill_path.restype = ctypes.c_char_p
    lib.gdn_prefill_scan.argtypes = [vp] * 9 + [i32, i64, i32, i32, i32, i32, i32, vp]
    lib.gdn_prefill_scan.restype = ctypes.c_int
    lib.gdn_prefill_backward.argtypes = [vp] * 15 + [i32, i64, i32, i32, i32, i32, vp]
    lib.gdn_prefill_backward.restype = ctypes.c_int
    lib.gdn_prepare.argtypes = [vp] * 14 + [i32, i64, i32, i32, i32, i32, vp]
    lib.gdn_prepare.restype = ctypes.c_int
    lib.gdn_prepare_decode_step.argtypes = [vp] * 12 + [i32, i32, i32, i32, i32, vp]
    lib.gdn_prepare_decode_step.restype = ctypes.c_int
    lib.gdn_output_norm_gate.argtypes = [vp, vp, vp, ctypes.c_float, i32, vp, i64, i32, i32, i32,
                                         vp]
    lib.gdn_decode_layer_step.argtypes = [vp] * 10 + [ctypes.c_float, i32, vp, i32, i32, i32,
                                                      i32, i32, vp]
    lib.gdn_decode_layer_step.restype = ctypes.c_int
    lib.gdn_output_norm_gate.restype = ctypes.c_int
    sz = ctypes.c_size_t
    lib.gdn_prefill_workspace_size.argtypes = [i32, i64, i32, i32, i32, i32, i32]
    lib.gdn_prefill_workspace_size.restype = sz
    lib.gdn_prefill_ws.argtypes = [vp] * 9 + [i32, i64, i32, i32, i32, i32, vp, sz, vp]
    lib.gdn_prefill_ws.restype = ctypes.c_int
    lib.gdn_prefill_scan_workspace_size.argtypes = [i32, i64, i32, i32, i32, i32, i32, i32]
    lib.gdn_prefill_scan_workspace_size.restype = sz
    lib.gdn_prefill_scan_ws.argtypes = [vp] * 9 + [i32, i64, i32, i32, i32, i32, i32, vp, sz,
                                                    vp]
    lib.gdn_prefill_scan_ws.restype = ctypes.c_int
    lib.gdn_prefill_backward_workspace_size.argtypes = [i32, i64, i32, i32, i32, i32, i32]
    lib.gdn_prefill_backward_workspace_size.restype = sz
    lib.gdn_prefill_backward_ws.argtypes = [vp] * 15 + [i32, i64, i32, i32, i32, i32, vp, sz, vp]
    lib.gdn_prefill_backward_ws.restype = ctypes.c_int
    lib.gdn_prefill_layer.argtypes = [vp] * 12 + [ctypes.c_float, i32, vp, vp, i32, i64, i32,
                                                  i32, i32, i32, vp]
    lib.gdn_prefill_layer.restype = ctypes.c_int
    lib.gdn_release_scratch.restype = ctypes.c_int
    lib.gdn_testing_scratch_reserved.argtypes = [vp]
    lib.gdn_testing_scratch_reserved.restype = ctypes.c_int
    _lib = lib
    return lib


def _ws_args(workspace):
    """(pointer, bytes) of a caller workspace: a uint8 CUDA tensor."""
    if not isinstance(workspace, torch.Tensor) or workspace.dtype != torch.uint8 \
            or not workspace.is_contiguous():
        raise TypeError("workspace must be a contiguous torch.uint8 tensor")
    return ctypes.c_void_p(workspace.data_ptr()), workspace.numel()


def prefill_workspace_size(batch, seqlen, heads, dk=256, dv=256, io_dtype=torch.bfloat16,
                           varlen=False) -> int:
    """Bytes of device workspace ``prefill(..., workspace=...)`` needs
    (``gdn_prefill_workspace_size``)."""
    n = load().gdn_prefill_workspace_size(batch, seqlen, heads, dk, dv, _io_code(io_dtype),
                                          int(bool(varlen)))
    if n == ctypes.c_size_t(-1).value:
        raise ValueError("unsupported prefill arguments")
    return int(n)


def prefill_scan_workspace_size(batch, seqlen, heads, dk=256, dv=256, io_dtype=torch.bfloat16,
                                varlen=False, segments=8) -> int:
    n = load().gdn_prefill_scan_workspace_size(batch, seqlen, heads, dk, dv, _io_code(io_dtype),
                                               int(bool(varlen)), int(segments))
    if n == ctypes.c_size_t(-1).value:
        raise ValueError("unsupported prefill_scan arguments")
    return int(n)


def prefill_backward_workspace_size(batch, seqlen, heads, dk=256, dv=256,
                                    io_dtype=torch.bfloat16, varlen=False) -> int:
    n = load().gdn_prefill_backward_workspace_size(batch, seqlen, heads, dk, dv,
                                                   _io_code(io_dtype), int(bool(varlen)))
    if n == ctypes.c_size_t(-1).value:
        raise ValueError("unsupported prefill_backward arguments")
    return int(n)


def release_scratch() -> None:
    """Hand the library's scratch pool on the current device back to the system
    (``gdn_release_scratch``; synchronises the device)."""
    rc = load().gdn_release_scratch()
    if rc != 0:
        raise GDNError("gdn_release_scratch", rc)


def scratch_reserved() -> int:
    """Bytes the library's scratch pool holds mapped on the current device."""
    v = ctypes.c_uint64(0)
    rc = load().gdn_testing_scratch_reserved(ctypes.byref(v))
    if rc != 0:
        raise GDNError("gdn_testing_scratch_reserved", rc)
    return int(v.value)


def version() -> str:
    return load().gdn_version().decode()


def kernel_launches() -> int:
    """Cumulative count of the library's kernel launches in this process."""
    return int(load().gdn_kernel_launches())


def prefill_path(io_dtype=torch.bfloat16) -> str:
    """Kernel path gdn_prefill takes for this I/O dtype."""
    return load().gdn_prefill_path(_io_code(io_dtype)).decode()


def _stream_handle(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _io_code(dtype):
    if dtype == torch.bfloat16:
        return GDN_BF16
    if dtype == torch.float32:
        return GDN_F32
    raise TypeError(f"q/k/v must be bfloat16 or float32, got {dtype}")


def _check(t, name, dtype, device):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def prefill(q, k, v, alpha, beta, S0=None, cu_seqlens=None, out=None, S_final=None,
            return_final: bool = True, stream=None, workspace=None):
    """Chunkwise prefill (``gdn_prefill``).

    Dense: q, k [B, T, H, dk]; v [B, T, H, dv]; alpha, beta [B, T, H] fp32.
    Varlen: the same with B = 1 (or no batch axis) and ``cu_seqlens`` int32
    [N + 1] on the device.  S0 / S_final: [N, H, dv, dk] fp32.
    ``workspace``: a uint8 CUDA tensor of at least
    :func:`prefill_workspace_size` bytes (``gdn_prefill_ws``: the call then
    allocates nothing); None takes scratch from the library's pool.
    Returns (out, S_final); S_final is None when ``return_final`` is False.
    """
    return _prefill_call(q, k, v, alpha, beta, S0, cu_seqlens, out, S_final, return_final,
                         stream, workspace, None)


def prefill_scan(q, k, v, alpha, beta, S0=None, cu_seqlens=None, segments=8, out=None,
                 S_final=None, return_final: bool = True, stream=None, workspace=None):
    """``gdn_prefill_scan``: :func:`prefill` with every sequence cut into
    ``segments`` pieces of whole chunks, run as a scan over the segments
    (dense or packed, bf16 or fp32).  Returns (out, S_final)."""
    if int(segments) < 1:
        raise ValueError("segments must be >= 1")
    return _prefill_call(q, k, v, alpha, beta, S0, cu_seqlens, out, S_final, return_final,
                         stream, workspace, int(segments))


def _prefill_call(q, k, v, alpha, beta, S0, cu_seqlens, out, S_final, return_final, stream,
                  workspace, segments):
    lib = load()
    dev = q.device
    io = q.dtype
    _io_code(io)
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check(t, name, io, dev)
    _check(alpha, "alpha", torch.float32, dev)
    _check(beta, "beta", torch.float32, dev)
    if q.dim() not in (3, 4) or k.shape != q.shape:
        raise ValueError("q and k must be [B, T, H, dk] (or [T, H, dk]) and equal in shape")
    H, dk, dv = q.shape[-2], q.shape[-1], v.shape[-1]
    if v.shape[:-1] != q.shape[:-1] or alpha.shape != q.shape[:-1] or beta.shape != q.shape[:-1]:
        raise ValueError("v, alpha, beta must match q's leading [.., T, H] axes")
    if cu_seqlens is None:
        B, T = (q.shape[0], q.shape[1]) if q.dim() == 4 else (1, q.shape[0])
        N, seqlen = B, T
    else:
        _check(cu_seqlens, "cu_seqlens", torch.int32, dev)
        if q.dim() == 4 and q.shape[0] != 1:
            raise ValueError("varlen input must have batch axis 1")
        N = cu_seqlens.numel() - 1
        seqlen = q.shape[-3]
    if S0 is not None:
        _check(S0, "S0", torch.float32, dev)
        if tuple(S0.shape) != (N, H, dv, dk):
            raise ValueError(f"S0 must be [{N}, {H}, {dv}, {dk}]")
    if out is None:
        out = torch.empty_like(v)
    else:
        _check(out, "out", io, dev)
    if S_final is None and return_final:
        S_final = torch.empty((N, H, dv, dk), dtype=torch.float32, device=dev)
    elif S_final is not None:
        _check(S_final, "S_final", torch.float32, dev)
    with torch.cuda.device(dev):
        args = (_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(S0), _ptr(cu_seqlens),
                _ptr(out), _ptr(S_final), N, seqlen, H, dk, dv, _io_code(io))
        if segments is not None:
            args = args + (segments,)
        name = "gdn_prefill" if segments is None else "gdn_prefill_scan"
        if workspace is None:
            rc = getattr(lib, name)(*args, _stream_handle(stream))
        else:
            name += "_ws"
            rc = getattr(lib, name)(*args, *_ws_args(workspace), _stream_handle(stream))
    if rc != 0:
        raise GDNError(name, rc)
    return out, S_final


def prefill_backward(q, k, v, alpha, beta, dout, S0=None, dS_final=None, cu_seqlens=None,
                     want_dS0: bool = True, stream=None, workspace=None):
    """Gradients of the prefill (``gdn_prefill_backward``) for
    L = <dout, out> + <dS_final, S_final>: returns dict dq, dk, dv (dtype of
    q), dalpha, dbeta (fp32) and dS0 ([N, H, dv, dk] fp32, or None when
    ``want_dS0`` is False).  Arguments as in :func:`prefill`; dout like out."""
    lib = load()
    dev, io = q.device, q.dtype
    _io_code(io)
    for name, t in (("q", q), ("k", k), ("v", v), ("dout", dout)):
        _check(t, name, io, dev)
    _check(alpha, "alpha", torch.float32, dev)
    _check(beta, "beta", torch.float32, dev)
    if q.dim() not in (3, 4) or k.shape != q.shape or dout.shape != v.shape:
        raise ValueError("q, k must be [B, T, H, dk] (or [T, H, dk]); dout shaped like v")
    H, dk, dv = q.shape[-2], q.shape[-1], v.shape[-1]
    if v.shape[:-1] != q.shape[:-1] or alpha.shape != q.shape[:-1] or beta.shape != q.shape[:-1]:
        raise ValueError("v, alpha, beta must match q's leading [.., T, H] axes")
    if cu_seqlens is None:
        B, T = (q.shape[0], q.shape[1]) if q.dim() == 4 else (1, q.shape[0])
        N, seqlen = B, T
    else:
        _check(cu_seqlens, "cu_seqlens", torch.int32, dev)
        if q.dim() == 4 and q.shape[0] != 1:
            raise ValueError("varlen input must have batch axis 1")
        N, seqlen = cu_seqlens.numel() - 1, q.shape[-3]
    for name, t in (("S0", S0), ("dS_final", dS_final)):
        if t is not None:
            _check(t, name, torch.float32, dev)
            if tuple(t.shape) != (N, H, dv, dk):
                raise ValueError(f"{name} must be [{N}, {H}, {dv}, {dk}]")
    g = dict(dq=torch.empty_like(q), dk=torch.empty_like(k), dv=torch.empty_like(v),
             dalpha=torch.empty_like(alpha), dbeta=torch.empty_like(beta),
             dS0=torch.empty((N, H, dv, dk), dtype=torch.float32, device=dev) if want_dS0 else None)
    with torch.cuda.device(dev):
        args = (_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(S0), _ptr(cu_seqlens),
                _ptr(dout), _ptr(dS_final), _ptr(g["dq"]), _ptr(g["dk"]), _ptr(g["dv"]),
                _ptr(g["dalpha"]), _ptr(g["dbeta"]), _ptr(g["dS0"]), N, seqlen, H, dk, dv,
                _io_code(io))
        if workspace is None:
            rc = lib.gdn_prefill_backward(*args, _stream_handle(stream))
        else:
            rc = lib.gdn_prefill_backward_ws(*args, *_ws_args(workspace), _stream_handle(stream))
    if rc != 0:
        raise GDNError("gdn_prefill_backward", rc)
    return g


def decode_step(q, k, v, alpha, beta, S, out=None, stream=None):
    """One token per sequence (``gdn_decode_step``): q, k [N, H, dk];
    v [N, H, dv]; alpha, beta [N, H]; S [N, H, dv, dk] fp32 updated in place.
    Returns out [N, H, dv] in the dtype of v."""
    lib = load()
    dev = q.device
    io = q.dtype
    _io_code(io)
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check(t, name, io, dev)
    _check(alpha, "alpha", torch.float32, dev)
    _check(beta, "beta", torch.float32, dev)
    _check(S, "S", torch.float32, dev)
    N, H, dk = q.shape
    dv = v.shape[-1]
    if tuple(S.shape) != (N, H, dv, dk) or alpha.shape != (N, H) or beta.shape != (N, H):
        raise ValueError("shape mismatch in decode_step arguments")
    if out is None:
        out = torch.empty_like(v)
    else:
        _check(out, "out", io, dev)
    with torch.cuda.device(dev):
        rc = lib.gdn_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(S),
                                 _ptr(out), N, H, dk, dv, _io_code(io), _stream_handle(stream))
    if rc != 0:
        raise GDNError("gdn_decode_step", rc)
    return out


GATE_ACT = {"silu": 0, "sigmoid": 1}


def prepare(qkv, conv_w, a_raw, b_raw, A_log, dt_bias, heads, dk=256, dv=256, cu_seqlens=None,
            conv_state_in=None, conv_state_out=None, stream=None):
    """Pre-recurrence steps (``gdn_prepare``): short conv + SiLU on the packed
    q|k|v projection, q/k L2 normalisation, decay and write strength.

    qkv [B, T, C] or [T, C] (C = H*(2*dk + dv)); conv_w [C, 4] fp32;
    a_raw, b_raw [B, T, H] / [T, H] fp32; A_log, dt_bias [H] fp32;
    conv_state_in / conv_state_out [N, 3, C] in qkv's dtype (or None).
    Returns dict q, k [.., H, dk], v [.., H, dv], alpha, beta [.., H] ready
    for :func:`prefill`.
    """
    lib = load()
    dev, io = qkv.device, qkv.dtype
    _io_code(io)
    H = heads
    C = H * (2 * dk + dv)
    _check(qkv, "qkv", io, dev)
    if qkv.shape[-1] != C or qkv.dim() not in (2, 3):
        raise ValueError(f"qkv must be [B, T, {C}] or [T, {C}]")
    lead = tuple(qkv.shape[:-1])
    for name, t in (("a_raw", a_raw), ("b_raw", b_raw)):
        _check(t, name, torch.float32, dev)
        if tuple(t.shape) != lead + (H,):
            raise ValueError(f"{name} must be {list(lead + (H,))}")
    _check(conv_w, "conv_w", torch.float32, dev)
    if tuple(conv_w.shape) != (C, 4):
        raise ValueError(f"conv_w must be [{C}, 4]")
    for name, t in (("A_log", A_log), ("dt_bias", dt_bias)):
        _check(t, name, torch.float32, dev)
        if tuple(t.shape) != (H,):
            raise ValueError(f"{name} must be [{H}]")
    if cu_seqlens is None:
        B, T = (qkv.shape[0], qkv.shape[1]) if qkv.dim() == 3 else (1, qkv.shape[0])
        N, seqlen = B, T
    else:
        _check(cu_seqlens, "cu_seqlens", torch.int32, dev)
        if qkv.dim() == 3 and qkv.shape[0] != 1:
            raise ValueError("varlen input must have batch axis 1")
        N, seqlen = cu_seqlens.numel() - 1, qkv.shape[-2]
    for name, t in (("conv_state_in", conv_state_in), ("conv_state_out", conv_state_out)):
        if t is not None:
            _check(t, name, io, dev)
            if tuple(t.shape) != (N, 3, C):
                raise ValueError(f"{name} must be [{N}, 3, {C}]")
    out = dict(q=torch.empty(lead + (H, dk), dtype=io, device=dev),
               k=torch.empty(lead + (H, dk), dtype=io, device=dev),
               v=torch.empty(lead + (H, dv), dtype=io, device=dev),
               alpha=torch.empty(lead + (H,), dtype=torch.float32, device=dev),
               beta=torch.empty(lead + (H,), dtype=torch.float32, device=dev))
    with torch.cuda.device(dev):
        rc = lib.gdn_prepare(_ptr(qkv), _ptr(conv_w), _ptr(a_raw), _ptr(b_raw), _ptr(A_log),
                             _ptr(dt_bias), _ptr(cu_seqlens), _ptr(conv_state_in),
                             _ptr(conv_state_out), _ptr(out["q"]), _ptr(out["k"]),
                             _ptr(out["v"]), _ptr(out["alpha"]), _ptr(out["beta"]), N, seqlen,
                             H, dk, dv, _io_code(io), _stream_handle(stream))
    if rc != 0:
        raise GDNError("gdn_prepare", rc)
    return out


def prepare_decode_step(qkv, conv_w, a_raw, b_raw, A_log, dt_bias, conv_state, heads, dk=256,
                        dv=256, out=None, stream=None):
    """``gdn_prepare_decode_step``: one token per sequence, qkv [N, C],
    a_raw / b_raw [N, H], conv_state [N, 3, C] updated in place.  Returns
    dict q, k [N, H, dk], v [N, H, dv], alpha, beta [N, H] (or fills ``out``)."""
    lib = load()
    dev, io = qkv.device, qkv.dtype
    _io_code(io)
    H = heads
    C = H * (2 * dk + dv)
    _check(qkv, "qkv", io, dev)
    if qkv.dim() != 2 or qkv.shape[1] != C:
        raise ValueError(f"qkv must be [N, {C}]")
    N = qkv.shape[0]
    _check(conv_state, "conv_state", io, dev)
    _check(conv_w, "conv_w", torch.float32, dev)
    for name, t in (("a_raw", a_raw), ("b_raw", b_raw)):
        _check(t, name, torch.float32, dev)
    if (tuple(conv_state.shape) != (N, 3, C) or tuple(conv_w.shape) != (C, 4)
            or tuple(a_raw.shape) != (N, H) or tuple(b_raw.shape) != (N, H)):
        raise ValueError("shape mismatch in prepare_decode_step arguments")
    if out is None:
        out = dict(q=torch.empty((N, H, dk), dtype=io, device=dev),
                   k=torch.empty((N, H, dk), dtype=io, device=dev),
                   v=torch.empty((N, H, dv), dtype=io, device=dev),
                   alpha=torch.empty((N, H), dtype=torch.float32, device=dev),
                   beta=torch.empty((N, H), dtype=torch.float32, device=dev))
    with torch.cuda.device(dev):
        rc = lib.gdn_prepare_decode_step(
            _ptr(qkv), _ptr(conv_w), _ptr(a_raw), _ptr(b_raw), _ptr(A_log), _ptr(dt_bias),
            _ptr(conv_state), _ptr(out["q"]), _ptr(out["k"]), _ptr(out["v"]), _ptr(out["alpha"]),
            _ptr(out["beta"]), N, H, dk, dv, _io_code(io), _stream_handle(stream))
    if rc != 0:
        raise GDNError("gdn_prepare_decode_step", rc)
    return out


def output_norm_gate(o, g, w, eps=1e-5, act="silu", y=None, stream=None):
    """Eq. 20 read-out (``gdn_output_norm_gate``): o / rms(o) * w * act(g)
    per (token, head) over dv.  o, g [.., H, dv] (same dtype); w [dv] fp32.
    ``y`` defaults to a new tensor; pass ``y=o`` to normalise in place."""
    lib = load()
    dev, io = o.device, o.dtype
    _io_code(io)
    _check(o, "o", io, dev)
    _check(g, "g", io, dev)
    _check(w, "w", torch.float32, dev)
    if g.shape != o.shape or o.dim() < 2 or tuple(w.shape) != (o.shape[-1],):
        raise ValueError("o and g must share [.., H, dv]; w must be [dv]")
    H, dv = o.shape[-2], o.shape[-1]
    tokens = o.numel() // (H * dv)
    if y is None:
        y = torch.empty_like(o)
    else:
        _check(y, "y", io, dev)
    with torch.cuda.device(dev):
        rc = lib.gdn_output_norm_gate(_ptr(o), _ptr(g), _ptr(w), float(eps), GATE_ACT[act], _ptr(y),
                                      tokens, H, dv, _io_code(io), _stream_handle(stream))
    if rc != 0:
        raise GDNError("gdn_output_norm_gate", rc)
    return y


def decode_layer_step(qkv, conv_w, a_raw, b_raw, A_log, dt_bias, conv_state, S, gate, norm_w,
                      eps=1e-5, act="silu", y=None, stream=None):
    """One fused decode step of the mixer core (``gdn_decode_layer_step``):
    conv + SiLU + L2 norm + gates, the state update, and Eq. 20's gated
    RMSNorm.  qkv [N, C]; conv_state [N, 3, C] and S [N, H, dv, dk] updated in
    place; gate [N, H, dv]; norm_w [dv].  Returns y [N, H, dv]."""
    lib = load()
    dev, io = qkv.device, qkv.dtype
    _io_code(io)
    N, H, dv, dk = S.shape
    C = H * (2 * dk + dv)
    _check(qkv, "qkv", io, dev)
    _check(conv_state, "conv_state", io, dev)
    _check(gate, "gate", io, dev)
    _check(S, "S", torch.float32, dev)
    for name, t in (("conv_w", conv_w), ("a_raw", a_raw), ("b_raw", b_raw), ("A_log", A_log),
                    ("dt_bias", dt_bias), ("norm_w", norm_w)):
        _check(t, name, torch.float32, dev)
    if (tuple(qkv.shape) != (N, C) or tuple(conv_state.shape) != (N, 3, C)
            or tuple(conv_w.shape) != (C, 4) or tuple(a_raw.shape) != (N, H)
            or tuple(b_raw.shape) != (N, H) or tuple(gate.shape) != (N, H, dv)
            or tuple(norm_w.shape) != (dv,)):
        raise ValueError("shape mismatch in decode_layer_step arguments")
    if y is None:
        y = torch.empty_like(gate)
    else:
        _check(y, "y", io, dev)
    with torch.cuda.device(dev):
        rc = lib.gdn_decode_layer_step(
            _ptr(qkv), _ptr(conv_w), _ptr(a_raw), _ptr(b_raw), _ptr(A_log), _ptr(dt_bias),
            _ptr(conv_state), _ptr(S), _ptr(gate), _ptr(norm_w), float(eps), GATE_ACT[act],
            _ptr(y), N, H, dk, dv, _io_code(io), _stream_handle(stream))
    if rc != 0:
        raise GDNError("gdn_decode_layer_step", rc)
    return y


def prefill_layer(qkv, conv_w, a_raw, b_raw, A_log, dt_bias, gate, norm_w, heads, S0=None,
                  cu_seqlens=None, conv_state_in=None, conv_state_out=None, eps=1e-5, act="silu",
                  y=None, S_final=None, return_final=True, stream=None):
    """The mixer core over whole sequences in one call (``gdn_prefill_layer``):
    what :func:`prepare`, :func:`prefill` and :func:`output_norm_gate` compute,
    as the pre-recurrence pass and then the tensor-core prefill with the gated
    RMSNorm applied inside it (for sequences in the segmented form, the
    pre-recurrence steps inside the prefill's tile loads too); bf16, dk = dv =
    256.  qkv [B, T, C] or [T, C]
    (packed with ``cu_seqlens``); a_raw, b_raw [.., H]; gate [.., H, dv];
    S0 / S_final [N, H, dv, dk]; conv states [N, 3, C].  Returns (y, S_final)."""
    lib = load()
    dev, io = qkv.device, qkv.dtype
    if io != torch.bfloat16:
        raise TypeError("prefill_layer takes bf16 projections")
    H, dk, dv = heads, 256, 256
    C = H * (2 * dk + dv)
    _check(qkv, "qkv", io, dev)
    if qkv.shape[-1] != C or qkv.dim() not in (2, 3):
        raise ValueError(f"qkv must be [B, T, {C}] or [T, {C}]")
    lead = tuple(qkv.shape[:-1])
    for name, t in (("a_raw", a_raw), ("b_raw", b_raw)):
        _check(t, name, torch.float32, dev)
        if tuple(t.shape) != lead + (H,):
            raise ValueError(f"{name} must be {list(lead + (H,))}")
    for name, t, shape in (("conv_w", conv_w, (C, 4)), ("A_log", A_log, (H,)),
                           ("dt_bias", dt_bias, (H,)), ("norm_w", norm_w, (dv,))):
        _check(t, name, torch.float32, dev)
        if tuple(t.shape) != shape:
            raise ValueError(f"{name} must be {list(shape)}")
    _check(gate, "gate", io, dev)
    if tuple(gate.shape) != lead + (H, dv):
        raise ValueError(f"gate must be {list(lead + (H, dv))}")
    if cu_seqlens is None:
        B, T = (qkv.shape[0], qkv.shape[1]) if qkv.dim() == 3 else (1, qkv.shape[0])
        N, seqlen = B, T
    else:
        _check(cu_seqlens, "cu_seqlens", torch.int32, dev)
        if qkv.dim() == 3 and qkv.shape[0] != 1:
            raise ValueError("varlen input must have batch axis 1")
        N, seqlen = cu_seqlens.numel() - 1, qkv.shape[-2]
    for name, t in (("conv_state_in", conv_state_in), ("conv_state_out", conv_state_out)):
        if t is not None:
            _check(t, name, io, dev)
            if tuple(t.shape) != (N, 3, C):
                raise ValueError(f"{name} must be [{N}, 3, {C}]")
    if S0 is not None:
        _check(S0, "S0", torch.float32, dev)
        if tuple(S0.shape) != (N, H, dv, dk):
            raise ValueError(f"S0 must be [{N}, {H}, {dv}, {dk}]")
    if y is None:
        y = torch.empty_like(gate)
    else:
        _check(y, "y", io, dev)
    if S_final is None and return_final:
        S_final = torch.empty((N, H, dv, dk), dtype=torch.float32, device=dev)
    elif S_final is not None:
        _check(S_final, "S_final", torch.float32, dev)
    with torch.cuda.device(dev):
        rc = lib.gdn_prefill_layer(
            _ptr(qkv), _ptr(conv_w), _ptr(a_raw), _ptr(b_raw), _ptr(A_log), _ptr(dt_bias),
            _ptr(conv_state_in), _ptr(conv_state_out), _ptr(S0), _ptr(cu_seqlens), _ptr(gate),
            _ptr(norm_w), float(eps), GATE_ACT[act], _ptr(y), _ptr(S_final), N, seqlen, H, dk,
            dv, GDN_BF16, _stream_handle(stream))
    if rc != 0:
        raise GDNError("gdn_prefill_layer", rc)
    return y, S_final


def device_status(stream=None) -> int:
    """Synchronise the stream; return and clear the device status word."""
    return int(load().gdn_get_device_status(_stream_handle(stream)))
