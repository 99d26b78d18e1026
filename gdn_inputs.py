"""Seeded synthetic inputs for the gated delta rule -- shared by the tests, the
benchmark and the smoke check.

This module holds none of the recurrence's arithmetic.  It only draws random
tensors, in a fixed order, shaped like the workloads of "Long-Context Aware
Upcycling: A New Frontier for Hybrid LLM Scaling" (6 GDN heads of head
dimension 256, Table 8 and the HyLo model card; 8K and 64K training lengths,
Section 4; long-context decode, Section 4.4).

Recipe (all draws fp32 standard normal from one ``torch.Generator`` seeded
with ``seed``, in this order):
  lengths (varlen only: integers uniform in [lo, hi] inclusive),
  q, k, v, alpha_raw, beta_raw, S0.
Then alpha = exp(-softplus(alpha_raw)) in (0, 1), beta = sigmoid(beta_raw) in
(0, 1), q and k are L2-normalised per (token, head) over the key dimension in
fp32, S0 = s0_std * N(0, 1) (or omitted), and q, k, v are cast to the I/O
dtype last.  alpha, beta and S0 stay fp32.

A generator on a CUDA device draws a different (but equally seeded) stream
than one on the CPU; either way both the GPU path and the oracle consume the
very same tensors, so parity never depends on the device the draws ran on.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch
import torch.nn.functional as F

H_PAGES = 6        # GDN heads per layer (HyLo model card: gdn_num_heads)
D_PAGES = 256      # GDN head dimension (Table 8: d_h = 256)


@dataclass
class PrefillCase:
    name: str
    lengths: list          # per-sequence token counts
    H: int = H_PAGES
    dk: int = D_PAGES
    dv: int = D_PAGES
    io_dtype: torch.dtype = torch.bfloat16
    s0_std: float | None = 0.02   # None: zero initial state (S0 pointer NULL)
    seed: int = 0
    varlen: bool = False          # pack through cu_seqlens

    @property
    def total_tokens(self) -> int:
        return int(sum(self.lengths))


@dataclass
class DecodeCase:
    name: str
    N: int
    steps: int
    H: int = H_PAGES
    dk: int = D_PAGES
    dv: int = D_PAGES
    io_dtype: torch.dtype = torch.bfloat16
    s0_std: float = 0.02
    seed: int = 2


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn(shape, g, device):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32)


def varlen_lengths(n_seq: int, lo: int, hi: int, seed: int) -> list:
    """Sequence lengths uniform on [lo, hi] inclusive, first draw of ``seed``
    on the CPU generator (so every device packs the same lengths)."""
    g = _gen("cpu", seed)
    return [int(x) for x in torch.randint(lo, hi + 1, (n_seq,), generator=g)]


def make_prefill(case: PrefillCase, device="cpu") -> dict:
    """Inputs in the library's boundary layouts.

    dense : q, k [B, T, H, dk]; v [B, T, H, dv]; alpha, beta [B, T, H]
    varlen: q, k [1, T_total, H, dk] ...; cu_seqlens int32 [N + 1]
    S0 [N, H, dv, dk] fp32 or None.
    """
    g = _gen(device, case.seed)
    if case.varlen:
        # the lengths were drawn first by the caller with the same seed; burn
        # one draw here so that the remaining stream order matches the recipe
        _ = torch.randint(0, 2, (len(case.lengths),), generator=g, device=device)
        B, T = 1, case.total_tokens
    else:
        assert len(set(case.lengths)) == 1, "dense batches share one length"
        B, T = len(case.lengths), case.lengths[0]
    N, H, dk, dv = len(case.lengths), case.H, case.dk, case.dv
    q = _randn((B, T, H, dk), g, device)
    k = _randn((B, T, H, dk), g, device)
    v = _randn((B, T, H, dv), g, device)
    a_raw = _randn((B, T, H), g, device)
    b_raw = _randn((B, T, H), g, device)
    S0 = None
    if case.s0_std is not None:
        S0 = _randn((N, H, dv, dk), g, device) * case.s0_std
    q = F.normalize(q, dim=-1)
    k = F.normalize(k, dim=-1)
    alpha = torch.exp(-F.softplus(a_raw))
    beta = torch.sigmoid(b_raw)
    out = dict(q=q.to(case.io_dtype).contiguous(), k=k.to(case.io_dtype).contiguous(),
               v=v.to(case.io_dtype).contiguous(), alpha=alpha.contiguous(),
               beta=beta.contiguous(), S0=S0, cu_seqlens=None)
    if case.varlen:
        cu = [0]
        for L in case.lengths:
            cu.append(cu[-1] + L)
        out["cu_seqlens"] = torch.tensor(cu, dtype=torch.int32, device=device)
    return out


def make_decode(case: DecodeCase, device="cpu", steps: int | None = None) -> dict:
    """Per-step inputs for ``steps`` consecutive decode steps, drawn up front:
    q, k [steps, N, H, dk]; v [steps, N, H, dv]; alpha, beta [steps, N, H];
    S [N, H, dv, dk] fp32 (the state the first step starts from)."""
    steps = case.steps if steps is None else steps
    g = _gen(device, case.seed)
    N, H, dk, dv = case.N, case.H, case.dk, case.dv
    q = _randn((steps, N, H, dk), g, device)
    k = _randn((steps, N, H, dk), g, device)
    v = _randn((steps, N, H, dv), g, device)
    a_raw = _randn((steps, N, H), g, device)
    b_raw = _randn((steps, N, H), g, device)
    S = _randn((N, H, dv, dk), g, device) * case.s0_std
    q = F.normalize(q, dim=-1)
    k = F.normalize(k, dim=-1)
    return dict(q=q.to(case.io_dtype).contiguous(), k=k.to(case.io_dtype).contiguous(),
                v=v.to(case.io_dtype).contiguous(),
                alpha=torch.exp(-F.softplus(a_raw)).contiguous(),
                beta=torch.sigmoid(b_raw).contiguous(), S=S.contiguous())


# The five workloads: shapes, dtypes and seeds of the 8K / 64K training
# lengths and of long-context decode, plus the small fp32 case.
def prefill_small_fp32() -> PrefillCase:
    return PrefillCase("prefill B=1 T=512 H=6 d=256 fp32 S0=0", [512],
                       io_dtype=torch.float32, s0_std=None, seed=0)


def prefill_8k() -> PrefillCase:
    return PrefillCase("prefill B=4 T=8192 H=6 d=256 bf16", [8192] * 4, seed=1)


def decode_256x1000() -> DecodeCase:
    return DecodeCase("decode N=256 H=6 d=256 bf16 x1000 steps", N=256, steps=1000, seed=2)


def prefill_8k_dv512() -> PrefillCase:
    return PrefillCase("prefill B=4 T=8192 H=6 dk=256 dv=512 bf16", [8192] * 4, dv=512, seed=5)


def decode_256_dv512() -> DecodeCase:
    return DecodeCase("decode N=256 H=6 dk=256 dv=512 bf16 x200 steps", N=256, steps=200, dv=512,
                      seed=6)


def prefill_64k() -> PrefillCase:
    return PrefillCase("prefill B=1 T=65536 H=6 d=256 bf16 S0=0", [65536], s0_std=None, seed=3)


def prefill_varlen16() -> PrefillCase:
    lengths = varlen_lengths(16, 1024, 65536, seed=4)
    return PrefillCase("varlen prefill N=16 len~U[1024,65536] H=6 d=256 bf16", lengths,
                       seed=4, varlen=True)


# ---------------------------------------------------------------------------
# Inputs of the layer steps around the recurrence (Appendix A.3: short
# convolution + SiLU, gates, Eq. 20's gated read-out).  Parameters are drawn
# like a fresh initialisation of the layer (no trained weights exist here):
#   qkv (the packed q|k|v projection) ~ N(0, 1)       [.., C], C = H (2 dk + dv)
#   conv_w ~ U(-0.5, 0.5) (1/sqrt(fan-in 4))          [C, 4]
#   a_raw, b_raw ~ N(0, 1)                            [.., H]
#   A_log = log U(1, 16)                              [H]
#   dt_bias ~ U(-5, -2)                               [H]
#   conv_state_in ~ N(0, 1) or omitted                [N, 3, C]
#   g (the W_G projection) ~ N(0, 1)                  [.., H, dv]
#   norm_w = 1 + 0.1 N(0, 1)                          [dv]
# drawn in that order from one CPU generator seeded with ``seed``, then qkv,
# the states and g are cast to the I/O dtype.  Varlen lengths are the
# caller's.


@dataclass
class LayerCase:
    name: str
    lengths: list
    H: int = H_PAGES
    dk: int = D_PAGES
    dv: int = D_PAGES
    io_dtype: torch.dtype = torch.bfloat16
    seed: int = 0
    varlen: bool = False
    carry_state: bool = True      # conv_state_in given (else zero history)

    @property
    def total_tokens(self) -> int:
        return int(sum(self.lengths))

    @property
    def channels(self) -> int:
        return self.H * (2 * self.dk + self.dv)


def make_layer(case: LayerCase, device="cpu") -> dict:
    g = _gen("cpu", case.seed)
    N, H, dv, C = len(case.lengths), case.H, case.dv, case.channels
    if case.varlen:
        lead = (case.total_tokens,)
    else:
        assert len(set(case.lengths)) == 1, "dense batches share one length"
        lead = (N, case.lengths[0])
    qkv = _randn(lead + (C,), g, "cpu")
    conv_w = torch.rand((C, 4), generator=g) - 0.5
    a_raw = _randn(lead + (H,), g, "cpu")
    b_raw = _randn(lead + (H,), g, "cpu")
    A_log = torch.log(1.0 + 15.0 * torch.rand((H,), generator=g))
    dt_bias = -5.0 + 3.0 * torch.rand((H,), generator=g)
    state = _randn((N, 3, C), g, "cpu") if case.carry_state else None
    gate = _randn(lead + (H, dv), g, "cpu")
    norm_w = 1.0 + 0.1 * _randn((dv,), g, "cpu")
    io = case.io_dtype
    out = dict(qkv=qkv.to(io), conv_w=conv_w, a_raw=a_raw, b_raw=b_raw, A_log=A_log,
               dt_bias=dt_bias, conv_state=None if state is None else state.to(io),
               g=gate.to(io), norm_w=norm_w, cu_seqlens=None)
    if case.varlen:
        cu = [0]
        for L in case.lengths:
            cu.append(cu[-1] + L)
        out["cu_seqlens"] = torch.tensor(cu, dtype=torch.int32)
    return {k: (v.to(device).contiguous() if isinstance(v, torch.Tensor) else v)
            for k, v in out.items()}


def layer_8k() -> LayerCase:
    return LayerCase("layer steps B=4 T=8192 H=6 d=256 bf16", [8192] * 4, seed=7)


def layer_decode_256() -> LayerCase:
    """One decode step's layer inputs for 256 sequences (as 256 one-token sequences)."""
    return LayerCase("layer steps decode N=256 H=6 d=256 bf16", [1] * 256, seed=8, varlen=True)
