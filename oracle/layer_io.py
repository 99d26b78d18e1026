"""fp64 oracle for the steps of a Gated DeltaNet layer that surround the
recurrence -- TEST INFRASTRUCTURE ONLY (same rules as the rest of ``oracle``:
only ``tests/``, the smoke check and the benchmark's CPU legs may use it).

Source: "Long-Context Aware Upcycling: A New Frontier for Hybrid LLM Scaling",
Appendix A.3 "GDN Layer Architecture":

* Before the recurrence (the paragraph after Table 8, and the text under
  Eq. 16-21): q, k and v each pass through a short causal 1-D convolution of
  kernel size 4 followed by SiLU; the forget gate is
  g_t = -exp(A_log) * softplus(W_alpha x_t + Delta_bias), so the decay the
  recurrence uses is alpha_t = e^{g_t}; the write strength is
  beta_t = sigmoid(W_beta x_t).
* After the recurrence (Eq. 20): the read-out o_t is RMS-normalised and
  multiplied by a gate computed from W_G x_t, before W_O (Eq. 21).

Readings where the pages are silent or garbled (each one is a choice, stated
once here and relied on by the tests):

* The convolution is depthwise and causal with no bias: output channel c at
  token t is sum_j w[c, j] * x[t - 3 + j, c], j = 0..3, so tap 3 multiplies
  the current token.  Before a sequence's first token the input is the
  carried convolution state (the three previous inputs, oldest first), or
  zero when no state is given.  Each sequence of a packed batch starts over.
* q and k are L2-normalised per head after the SiLU: x / sqrt(sum x^2 + eps),
  eps = 1e-6 (the normalisation the workloads of the recurrence assume).
* Eq. 20's gate is garbled.  The reading here is the usual gated RMSNorm of
  the cited GDN module: y = o / sqrt(mean(o^2) + eps) * w * act(W_G x), the
  mean taken over the dv values of one head, w a learned [dv] weight shared
  by the heads, act = SiLU (sigmoid also offered).
* softplus(x) = log(1 + e^x), computed here as logaddexp(0, x).

Layouts (the library's): a packed projection ``qkv`` [T, C] with
C = H*(2*dk + dv) channels ordered q | k | v, each block head-major; conv
weights [C, 4]; conv state [N, 3, C]; a_raw, b_raw (the W_alpha x and
W_beta x projections) [T, H]; A_log, dt_bias [H]; o and the gate input g
[T, H, dv].
"""
from __future__ import annotations

import numpy as np

KERNEL = 4            # short convolution width (Table 8's paragraph)
L2_EPS = 1e-6


def widen(x) -> np.ndarray:
    """fp32 or raw-bfloat16 (uint16) input -> exact fp64 copy."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.bfloat16:
                x = x.view(torch.int16).numpy().view(np.uint16)
            else:
                x = x.numpy()
    except ImportError:  # pragma: no cover
        pass
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return x.astype(np.float64)


def silu(x):
    """x * sigmoid(x)."""
    return x / (1.0 + np.exp(-x))


def sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def softplus(x):
    return np.logaddexp(0.0, x)


def _seq_bounds(T, cu_seqlens):
    if cu_seqlens is None:
        return [(0, T)]
    cu = [int(c) for c in widen(cu_seqlens).astype(np.int64)]
    return list(zip(cu[:-1], cu[1:]))


def short_conv_silu(x, w, cu_seqlens=None, conv_state=None):
    """Causal depthwise convolution of width 4, then SiLU, per sequence
    (Appendix A.3, the paragraph after Table 8: short convolution, kernel
    size 4, with SiLU, on q, k and v).

    x [T, C]; w [C, 4]; conv_state [N, 3, C] or None (zero history).
    Returns (y [T, C] fp64, final_state [N, 3, C] fp64): the final state is
    the last three inputs of (history, sequence), oldest first.
    """
    x = widen(x)
    w = widen(w)
    T, C = x.shape
    bounds = _seq_bounds(T, cu_seqlens)
    hist = (np.zeros((len(bounds), KERNEL - 1, C)) if conv_state is None
            else widen(conv_state).reshape(len(bounds), KERNEL - 1, C))
    y = np.zeros((T, C))
    final = np.zeros((len(bounds), KERNEL - 1, C))
    for n, (a, b) in enumerate(bounds):
        ext = np.concatenate([hist[n], x[a:b]], axis=0)      # [3 + L, C]
        L = b - a
        acc = np.zeros((L, C))
        for j in range(KERNEL):
            acc += w[:, j] * ext[j:j + L]
        y[a:b] = silu(acc)
        final[n] = ext[L:L + KERNEL - 1]
    return y, final


def l2_normalize(x, eps=L2_EPS):
    """x / sqrt(sum(x^2) + eps) over the last axis: the per-head q / k
    normalisation the recurrence's inputs assume (a reading: the pages do not
    state it for GDN)."""
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


def gates(a_raw, b_raw, A_log, dt_bias):
    """alpha = exp(-exp(A_log) * softplus(a_raw + dt_bias)), beta = sigmoid(b_raw):
    the forget gate g_t of Eq. 16 (alpha = e^{g_t}) and the write strength of
    Eq. 18, as the text under Eq. 16-21 defines them.
    a_raw, b_raw [..., H]; A_log, dt_bias [H]."""
    g = -np.exp(widen(A_log)) * softplus(widen(a_raw) + widen(dt_bias))
    return np.exp(g), sigmoid(widen(b_raw))


def prepare(qkv, conv_w, a_raw, b_raw, A_log, dt_bias, H, dk, dv, cu_seqlens=None,
            conv_state=None):
    """The layer's pre-recurrence steps for a packed batch (Appendix A.3:
    Table 8's paragraph and the text under Eq. 16-21), in order: convolution
    + SiLU of the packed q|k|v projection, q / k normalisation, gates.

    Returns dict of fp64 arrays: q, k [T, H, dk]; v [T, H, dv]; alpha, beta
    [T, H]; conv_state [N, 3, C] (the state after the last token).
    """
    y, final = short_conv_silu(qkv, conv_w, cu_seqlens, conv_state)
    T = y.shape[0]
    q = y[:, :H * dk].reshape(T, H, dk)
    k = y[:, H * dk:2 * H * dk].reshape(T, H, dk)
    v = y[:, 2 * H * dk:].reshape(T, H, dv)
    alpha, beta = gates(a_raw, b_raw, A_log, dt_bias)
    return dict(q=l2_normalize(q), k=l2_normalize(k), v=v, alpha=alpha, beta=beta,
                conv_state=final)


def prepare_decode_step(qkv, conv_w, a_raw, b_raw, A_log, dt_bias, conv_state, H, dk, dv):
    """One token per sequence, the decode form of `prepare` (the same
    passages): qkv [N, C], conv_state [N, 3, C] (fp64, updated in place).
    Returns q, k [N, H, dk]; v [N, H, dv]; alpha, beta [N, H]."""
    assert isinstance(conv_state, np.ndarray) and conv_state.dtype == np.float64
    N = conv_state.shape[0]
    cu = np.arange(N + 1)
    r = prepare(qkv, conv_w, a_raw, b_raw, A_log, dt_bias, H, dk, dv, cu, conv_state)
    conv_state[...] = r.pop("conv_state")
    return r


def output_norm_gate(o, g, w, eps, act="silu"):
    """Eq. 20 read-out (Appendix A.3), in this module's reading of the garbled
    equation: o / sqrt(mean(o^2) + eps) * w * act(g) per head.
    o, g [..., dv]; w [dv]."""
    o = widen(o)
    gv = widen(g)
    gate = silu(gv) if act == "silu" else sigmoid(gv)
    r = o / np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + float(eps))
    return r * widen(w) * gate
