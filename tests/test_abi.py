"""The C-ABI library loads, exports every entry point include/gdn.h declares,
and rejects malformed host arguments before touching the GPU.  CPU only: no
call here reaches a CUDA runtime function.

The pointers below are fake addresses.  Every call therefore asserts an exact
host-check code (1-3): a call that got past all host checks would go on to the
device (code 4 on a machine without one, a launch on fake addresses on a
machine with one).  The launch-counter fixture fails any test that launches,
and the tests that pass fake addresses do not run at all where a CUDA device
is visible, so that a missed host check can never reach a GPU."""
import ctypes
import glob
import os
import re

import pytest

import hybrid_linear_attention_deltanet_gb300 as gdn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdn.h")
HEADERS = sorted(glob.glob(os.path.join(ROOT, "include", "*.h")))


def declared_functions(headers=(HEADER,)):
    names = set()
    for h in headers:
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names.update(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(gdn_\w+)\s*\(", text,
                                flags=re.M))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(gdn.lib_path()):
        from hybrid_linear_attention_deltanet_gb300 import _build
        _build.build()
    return gdn.load()


def _device_visible() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


# tests that hand the library fake device addresses
fake_addresses = pytest.mark.skipif(_device_visible(),
                                    reason="fake device addresses are only passed where no GPU "
                                           "is visible")


@pytest.fixture(autouse=True)
def no_launch(request):
    if "lib" not in request.fixturenames:
        yield
        return
    lib = request.getfixturevalue("lib")
    before = lib.gdn_kernel_launches()
    yield
    assert lib.gdn_kernel_launches() == before, "a host-argument test launched a kernel"


def test_header_declares_the_boundary():
    names = declared_functions()
    for fn in ("gdn_prefill", "gdn_decode_step", "gdn_get_device_status", "gdn_version",
               "gdn_status_string"):
        assert fn in names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions(HEADERS)
    assert len(HEADERS) >= 2 and "gdn_testing_bounded_wait" in names and "gdn_prepare" in names
    for fn in names:
        assert hasattr(lib, fn), fn


def test_version_and_status_strings(lib):
    assert b"sm_103a" in lib.gdn_version()
    assert lib.gdn_status_string(0) == b"ok"
    assert lib.gdn_status_string(3).startswith(b"pointer")


P = ctypes.c_void_p
A16 = P(0x10000)          # aligned fake device addresses: validation fails before any use
A16b = P(0x20000)
MIS = P(0x10004)


def _prefill(lib, q=A16, k=A16, v=A16, alpha=A16, beta=A16, S0=None, cu=None, out=A16b,
             S_final=None, batch=1, T=64, H=6, dk=256, dv=256, io=1):
    return lib.gdn_prefill(q, k, v, alpha, beta, S0, cu, out, S_final, batch, T, H, dk, dv, io,
                           None)


@fake_addresses
def test_prefill_rejects_bad_host_arguments(lib):
    assert _prefill(lib, q=None) == 1
    assert _prefill(lib, out=None) == 1
    assert _prefill(lib, batch=0) == 1
    assert _prefill(lib, H=0) == 1
    assert _prefill(lib, T=-1) == 1
    assert _prefill(lib, dk=128) == 2
    assert _prefill(lib, dv=384) == 2
    assert _prefill(lib, dv=128) == 2
    assert _prefill(lib, io=7) == 2
    assert _prefill(lib, q=MIS) == 3
    assert _prefill(lib, S_final=MIS) == 3
    assert _prefill(lib, cu=P(0x30002)) == 3
    assert _prefill(lib, alpha=P(0x40001)) == 3
    # 4-byte alignment is enough for alpha / beta: the call gets past the
    # alignment check and stops at the later overlap check (out over q), so it
    # never launches, with or without a GPU
    assert _prefill(lib, alpha=P(0x40004), beta=P(0x50004), out=A16) == 1
    # out overlapping an input range
    assert _prefill(lib, q=P(0x100000), k=P(0x200000), v=P(0x300000), alpha=P(0x400000),
                    beta=P(0x500000), out=P(0x100000 + 4096)) == 1


@fake_addresses
def test_decode_rejects_bad_host_arguments(lib):
    f = lambda **kw: lib.gdn_decode_step(kw.get("q", A16), A16, A16, A16, A16,
                                         kw.get("S", P(0x800000)), kw.get("out", P(0x900000)),
                                         kw.get("N", 4), 6, kw.get("dk", 256), 256, 1, None)
    assert f(S=None) == 1
    assert f(N=0) == 1
    assert f(dk=64) == 2
    assert lib.gdn_decode_step(A16, A16, A16, A16, A16, P(0x800000), P(0x900000), 4, 6, 256, 384,
                               1, None) == 2
    assert f(q=MIS) == 3
    assert f(out=P(0x800000 + 1024)) == 1      # out inside the state


def _prepare(lib, qkv=A16, conv_w=A16, a_raw=A16, b_raw=A16, cu=None, sin=None, sout=None,
             q=P(0x100000), k=P(0x200000), v=P(0x300000), alpha=P(0x400000), beta=P(0x500000),
             batch=1, T=64, H=6, dk=256, dv=256, io=1):
    return lib.gdn_prepare(qkv, conv_w, a_raw, b_raw, A16, A16, cu, sin, sout, q, k, v, alpha, beta,
                           batch, T, H, dk, dv, io, None)


@fake_addresses
def test_prepare_rejects_bad_host_arguments(lib):
    assert _prepare(lib, batch=0) == 1
    assert _prepare(lib, T=-1) == 1
    assert _prepare(lib, conv_w=None) == 1
    assert _prepare(lib, q=None) == 1
    assert _prepare(lib, dk=128) == 2
    assert _prepare(lib, dv=384) == 2
    assert _prepare(lib, io=7) == 2
    assert _prepare(lib, qkv=MIS) == 3
    assert _prepare(lib, sout=P(0x600008)) == 3
    assert _prepare(lib, a_raw=P(0x40001)) == 3
    assert _prepare(lib, q=P(0x10000 + 4096)) == 1                  # q inside qkv
    assert _prepare(lib, sin=P(0x700000), sout=P(0x700000)) == 1    # state in place: not here
    assert _prepare(lib, k=P(0x100000 + 1024)) == 1                 # two outputs overlap


@fake_addresses
def test_prepare_decode_rejects_bad_host_arguments(lib):
    f = lambda st=P(0x700000), q=P(0x100000), H=6, dv=256, io=1: lib.gdn_prepare_decode_step(
        A16, A16, A16, A16, A16, A16, st, q, P(0x200000), P(0x300000), P(0x400000), P(0x500000),
        4, H, 256, dv, io, None)
    assert f(st=None) == 1
    assert f(H=0) == 1
    assert f(dv=128) == 2
    assert f(st=P(0x700004)) == 3
    assert f(q=P(0x700000 + 2048)) == 1                                # q inside the state


@fake_addresses
def test_output_norm_gate_rejects_bad_host_arguments(lib):
    f = lambda o=A16, g=P(0x200000), w=P(0x300000), eps=1e-5, act=0, y=P(0x400000), dv=256, io=1: \
        lib.gdn_output_norm_gate(o, g, w, ctypes.c_float(eps), act, y, 64, 6, dv, io, None)
    assert f(act=5) == 2
    assert f(dv=128) == 2
    assert f(io=3) == 2
    assert f(eps=-1.0) == 1
    assert f(g=None) == 1
    assert f(y=MIS) == 3
    assert f(y=P(0x200000)) == 1                                      # y over g
    assert f(y=P(0x10000 + 1024)) == 1                                # y partly over o


@fake_addresses
def test_prefill_backward_rejects_bad_host_arguments(lib):
    f = lambda q=A16, dout=P(0x600000), dq=P(0x100000), dS0=None, dv=256, io=1, batch=1, T=64: \
        lib.gdn_prefill_backward(q, A16b, A16b, A16b, A16b, None, None, dout, None, dq,
                                 P(0x200000), P(0x300000), P(0x400000), P(0x500000), dS0, batch,
                                 T, 6, 256, dv, io, None)
    assert f(batch=0) == 1
    assert f(dout=None) == 1
    assert f(dv=384) == 2
    assert f(io=5) == 2
    assert f(q=MIS) == 3
    assert f(dS0=P(0x700008)) == 3
    assert f(dq=P(0x600000 + 1024)) == 1                              # dq over dout
    assert f(dq=P(0x200000 + 1024)) == 1                              # dq over dk


def test_fault_hook_rejects_bad_arguments(lib):
    f = lib.gdn_testing_bounded_wait
    f.argtypes = [ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p]
    assert f(2, 1000, None) == 1
    assert f(0, -1, None) == 1
    assert f(1, 3_000_000_000, None) == 1


@fake_addresses
def test_prefill_scan_rejects_bad_host_arguments(lib):
    f = lambda q=A16, out=A16b, batch=1, T=4096, dv=256, io=1, seg=4: lib.gdn_prefill_scan(
        q, A16, A16, A16, A16, None, None, out, None, batch, T, 6, 256, dv, io, seg, None)
    assert f(seg=0) == 1
    assert f(seg=-3) == 1
    assert f(batch=0) == 1
    assert f(dv=384) == 2
    assert f(io=7) == 2
    assert f(q=MIS) == 3
    assert f(out=A16) == 1                                              # out over q


@fake_addresses
def test_prefill_layer_rejects_bad_host_arguments(lib):
    def f(qkv=A16, y=A16b, io=1, dv=256, act=0, eps=1e-5, batch=1, T=128, S0=None):
        return lib.gdn_prefill_layer(qkv, P(0x30000), P(0x40000), P(0x50000), P(0x60000),
                                     P(0x60100), None, None, S0, None, P(0x70000), P(0x80000),
                                     eps, act, y, None, batch, T, 2, 256, dv, io, None)
    assert f(io=0) == 2                      # fp32: the fused layer is bf16 only
    assert f(dv=512) == 2
    assert f(act=2) == 1
    assert f(eps=-1.0) == 1
    assert f(batch=0) == 1
    assert f(qkv=MIS) == 3
    assert f(S0=MIS) == 3
    assert f(y=P(0x10000 + 4096)) == 1       # y over qkv


SIZE_MAX = ctypes.c_size_t(-1).value


def _ws_size_fns(lib):
    sz, i32, i64 = ctypes.c_size_t, ctypes.c_int32, ctypes.c_int64
    lib.gdn_prefill_workspace_size.argtypes = [i32, i64, i32, i32, i32, i32, i32]
    lib.gdn_prefill_workspace_size.restype = sz
    lib.gdn_prefill_scan_workspace_size.argtypes = [i32, i64, i32, i32, i32, i32, i32, i32]
    lib.gdn_prefill_scan_workspace_size.restype = sz
    lib.gdn_prefill_backward_workspace_size.argtypes = [i32, i64, i32, i32, i32, i32, i32]
    lib.gdn_prefill_backward_workspace_size.restype = sz
    return (lib.gdn_prefill_workspace_size, lib.gdn_prefill_scan_workspace_size,
            lib.gdn_prefill_backward_workspace_size)


def _up(x, a):
    return (x + a - 1) // a * a


def _plain_bf16_bytes(B, T, H, dv, varlen):
    """gdn.h's layout of the plain bf16 prefill scratch, restated: chunk offsets
    of a packed batch (4 (N + 1) bytes rounded to 256), then one operand image
    per (chunk, head) of 107520 bytes at dv = 256 (141312 at dv = 512) over the
    chunk bound, then a 4-byte flag per (chunk, head) rounded to 256."""
    items = _chunks(B, T, varlen) * H
    img = 107520 if dv == 256 else 141312
    return items * img + _up(items * 4, 256) + (_up(4 * (B + 1), 256) if varlen else 0)


def _chunks(B, T, varlen):
    return B * -(-T // 64) if not varlen else (T + 63 * B) // 64


def _segmented_bytes(B, T, H, dv, varlen, work, slots):
    """gdn.h's layout of the segmented form: chunk offsets, token starts and
    sequences of the slots, the sequences' first slots, a role byte per slot,
    the launch order (12 bytes per slot), the per-chunk scratch, three fp32
    states per (slot, head)."""
    ints = _up(4 * (slots + 1), 256)
    state = _up(slots * H * dv * 256 * 4, 256)
    return (3 * ints + _up(4 * (B + 1), 256) + _up(slots, 256) + _up(12 * slots, 256) +
            _up(work, 256) + 3 * state)


def test_workspace_size_follows_the_documented_layout(lib):
    ws, ws_scan, _ = _ws_size_fns(lib)
    for (B, T, H, dv, varlen) in [(4, 8192, 6, 256, 0), (3, 1000, 6, 256, 1), (1, 100, 2, 512, 0),
                                  (2, 0, 6, 256, 1), (1, 65472, 6, 256, 0), (2, 65472, 6, 256, 1)]:
        assert ws(B, T, H, 256, dv, 1, varlen) == _plain_bf16_bytes(B, T, H, dv, varlen), \
            (B, T, H, dv, varlen)
    # from 1024 chunks on (65,473 tokens: T of a dense batch, T_total of a
    # packed one) the call takes the segmented form
    for (B, T, H, dv, varlen) in [(1, 65473, 6, 256, 0), (1, 65536, 6, 256, 0),
                                  (16, 388611, 6, 256, 1), (2, 100000, 3, 512, 1)]:
        mc = _chunks(B, T, varlen)
        work = _plain_bf16_bytes(mc, 64, H, dv, 0)       # the images over the same chunks
        want = _segmented_bytes(B, T, H, dv, varlen, work, B + mc // 160 + 1)
        assert ws(B, T, H, 256, dv, 1, varlen) == want, (B, T, H, dv, varlen)
        # fp32: the CUDA-core path's arrays take the images' place
        work32 = ws(mc, 64, H, 256, dv, 0, 0)
        assert ws(B, T, H, 256, dv, 0, varlen) == \
            _segmented_bytes(B, T, H, dv, varlen, work32, B + mc // 160 + 1)
    # gdn_prefill_scan: the segmented layout with min(B * segments, B + chunks) slots
    for (B, T, H, dv, io, varlen, seg) in [(1, 64, 6, 256, 1, 0, 8), (2, 1000, 2, 256, 1, 0, 3),
                                           (3, 5000, 2, 512, 0, 1, 4), (1, 65536, 6, 256, 1, 0, 1)]:
        mc = _chunks(B, T, varlen)
        work = ws(mc, 64, H, 256, dv, io, 0)
        assert ws_scan(B, T, H, 256, dv, io, varlen, seg) == \
            _segmented_bytes(B, T, H, dv, varlen, work, min(B * seg, B + mc)), (B, T, seg)


def test_workspace_size_queries_reject_bad_arguments(lib):
    ws, ws_scan, ws_bwd = _ws_size_fns(lib)
    for f in (ws, ws_bwd):
        assert f(0, 64, 6, 256, 256, 1, 0) == SIZE_MAX
        assert f(1, 64, 6, 128, 256, 1, 0) == SIZE_MAX
        assert f(1, 64, 6, 256, 384, 1, 0) == SIZE_MAX
        assert f(1, 64, 6, 256, 256, 7, 0) == SIZE_MAX
        assert f(1, -1, 6, 256, 256, 1, 0) == SIZE_MAX
    assert ws_scan(1, 4096, 6, 256, 256, 1, 0, 0) == SIZE_MAX
    assert ws_scan(1, 4096, 0, 256, 256, 1, 0, 4) == SIZE_MAX
    assert ws_scan(1, 4096, 6, 256, 256, 2, 0, 4) == SIZE_MAX


def test_workspace_sizes_scale_with_the_problem(lib):
    ws, ws_scan, ws_bwd = _ws_size_fns(lib)
    # fp32 I/O (CUDA-core path): linear in the number of (chunk, head) units
    a, b = ws(1, 64 * 8, 6, 256, 256, 0, 0), ws(1, 64 * 16, 6, 256, 256, 0, 0)
    assert 0 < a < b and b - a == a - ws(1, 0, 6, 256, 256, 0, 0)
    # the segmented form holds the plain images plus the per-segment states
    assert ws_scan(1, 8192, 6, 256, 256, 1, 0, 8) > ws(1, 8192, 6, 256, 256, 1, 0)
    assert ws(1, 65536, 6, 256, 256, 1, 0) > ws(1, 65472, 6, 256, 256, 1, 0) + 3 * 6 * 2**18 * 4
    # the backward holds at least the forward's images (bf16) and grows with T
    assert ws_bwd(4, 8192, 6, 256, 256, 1, 0) > ws(4, 8192, 6, 256, 256, 1, 0)
    assert ws_bwd(1, 1024, 6, 256, 256, 0, 0) < ws_bwd(1, 2048, 6, 256, 256, 0, 0)


@fake_addresses
def test_workspace_entry_points_reject_bad_workspaces(lib):
    sz, i32, i64 = ctypes.c_size_t, ctypes.c_int32, ctypes.c_int64
    f = lib.gdn_prefill_ws
    f.argtypes = [P] * 9 + [i32, i64, i32, i32, i32, i32, P, sz, P]
    need = _ws_size_fns(lib)[0](1, 64, 6, 256, 256, 1, 0)
    ins = dict(q=P(0x100000), k=P(0x200000), v=P(0x300000), alpha=P(0x400000),
               beta=P(0x500000), out=P(0x600000))
    call = lambda ws, n: f(ins["q"], ins["k"], ins["v"], ins["alpha"], ins["beta"], None, None,
                           ins["out"], None, 1, 64, 6, 256, 256, 1, ws, n, None)
    assert call(None, need) == 1                      # the problem needs scratch
    assert call(P(0x10000000), need - 1) == 1          # too small
    assert call(P(0x10000010), need) == 3             # not 256-byte aligned
    assert call(P(0x100000), need) == 1                # over q
    g = lib.gdn_prefill_backward_ws
    g.argtypes = [P] * 15 + [i32, i64, i32, i32, i32, i32, P, sz, P]
    needb = _ws_size_fns(lib)[2](1, 64, 6, 256, 256, 1, 0)
    callb = lambda ws, n: g(P(0x100000), P(0x200000), P(0x300000), P(0x400000), P(0x500000),
                            None, None, P(0x600000), None, P(0x700000), P(0x800000),
                            P(0x900000), P(0xa00000), P(0xb00000), None, 1, 64, 6, 256, 256, 1,
                            ws, n, None)
    assert callb(None, needb) == 1
    assert callb(P(0x10000200), needb) == 3           # not 1024-byte aligned
    assert callb(P(0x10000000), needb - 1) == 1
