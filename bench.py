"""Benchmark of the Gated DeltaNet hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Workload of the headline line: chunkwise prefill of 4 sequences x 8192
tokens, 6 heads of dimension 256, bf16 q/k/v/out, fp32 alpha/beta/state,
S0 ~ N(0, 0.02^2) (the 8K training length).  One step = one gdn_prefill call
over that batch, inputs resident in HBM.  `value` is prefill throughput in
Mtok/s per layer (a token = all 6 heads of one layer) over all ranks.
The metric also names decode state GB/s: the same line carries, under
"decode", 1000 consecutive gdn_decode_step calls over 256 sequences (fp32
256x256 states per head updated in place) with their own roofline.

Multi-GPU: replicas only (the path has no exchange step); each rank runs the
same workload on its own GPU, timed between barriers, max time over ranks.

--impl reference times the fp64 CPU oracle (the parity reference) on a
bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GDN prefill Mtok/s/layer and decode state GB/s; % of GB300 roofline"
C = 64
DK = DV = 256
H = 6


def prefill_flops(lengths, H=H, dk=DK, dv=DV):
    """Counted chunked-form FLOPs at C = 64: per (chunk, head)
    C^2 (6 dk + 4 dv) + 6 C dk dv + C^3 / 3 (full C x C products; elementwise
    work not counted).  Partial chunks are counted as full chunks."""
    f_chunk = C * C * (6 * dk + 4 * dv) + 6 * C * dk * dv + C ** 3 / 3
    chunks = sum((L + C - 1) // C for L in lengths)
    return f_chunk * chunks * H


def prefill_bytes(lengths, io_bytes=2, H=H, s0=True, s_final=True, dv=DV):
    """Algorithmic bytes: q, k, v in, out written (io dtype), alpha and beta
    (fp32) per token-head, plus S0 read and S_final written per sequence."""
    tok = sum(lengths)
    per_tok = H * ((2 * DK + 2 * dv) * io_bytes + 8)
    state = len(lengths) * H * dv * DK * 4
    return tok * per_tok + state * (int(s0) + int(s_final))


def decode_bytes(N, io_bytes=2, dv=DV):
    """Per step: the fp32 state read and written once, q, k, v, out and
    alpha, beta once."""
    return N * H * (2 * dv * DK * 4 + (2 * DK + 2 * dv) * io_bytes + 8)


def prepare_bytes(T_total, N, H=H, dk=DK, dv=DV, io_bytes=2, state=True):
    """gdn_prepare: read the packed q|k|v projection and the two gate inputs,
    write q, k, v, alpha, beta; carried convolution state in and out; conv
    weights and per-head parameters once."""
    C = H * (2 * dk + dv)
    per_tok = 2 * C * io_bytes + 4 * H * 4
    return T_total * per_tok + (2 * N * 3 * C * io_bytes if state else 0) + C * 16 + 2 * H * 4


def backward_flops(lengths, H=H, dk=DK, dv=DV):
    """FLOPs the chunked backward executes per call (C = 64 rows a chunk,
    padded chunks counted whole): the forward re-run for the chunk-start
    states (KK^T, QK^T, W, U~, U and S' per chunk; with bf16 I/O the U and S'
    products run inside the tensor-core forward prefill) plus the reverse
    state pass
    (K dS'^T, Ph^T dO, dO^T Qh, dU^T W) and the per-chunk gradient products
    (U, dO S, dU S, U dS', K dS'^T at C x d x d; dPh, dT, T^T dW, T^T dU, T^T dT,
    dA, (M + M^T) K, FG^T Q, FG K at C x C x d)."""
    chunks = sum((L + C - 1) // C for L in lengths) * H
    big = 2 * C * dk * dv                      # one C x d x d product
    small_k, small_v = 2 * C * C * dk, 2 * C * C * dv
    fwd = 2 * small_k + small_k + small_v + 2 * big
    rev = big + small_v + 2 * big
    local = 5 * big + small_v + small_k + small_v + small_k + small_v + 4 * C * C * C \
        + 3 * small_k
    return chunks * (fwd + rev + local)


def norm_gate_bytes(rows, dv=DV, io_bytes=2):
    """gdn_output_norm_gate: read o and g, write y, per (token, head) row."""
    return rows * dv * io_bytes * 3 + dv * 4


# fp32 FMA peak of the CUDA cores, from the unit counts and the maximum SM
# clock (152 SMs x 128 FP32 lanes x 2 FLOP x 2.07 GHz)
FP32_FMA_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12


def TF32_TFLOPS(peaks):
    """Dense tf32 tensor peak: the bf16 figure scaled by the nominal ratio
    (1.1 PFLOP/s tf32 against 2.25 bf16)."""
    return peaks["bf16"] * 1.1 / 2.25


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm_gbs=d["hbm_gbs"], bf16=d["bf16_tflops"],
                    bf16_sus=d.get("bf16_tflops_sustained", d["bf16_tflops"]), src="measured")
    return dict(hbm_gbs=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


def source_sha(paths):
    h = hashlib.sha256()
    for p in paths:
        h.update(open(os.path.join(ROOT, p), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_key):
    """DRAM bytes per launch of a kernel from the committed ncu summary, or
    None when the kernel's sources changed since the counters were taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(kernel_key)
    if not d:
        return None
    if source_sha(d["sources"]) != d["source_sha"]:
        return None
    return d["dram_bytes_per_launch"]


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.text = self.proc.communicate(timeout=5)[0]
            except Exception:
                self.proc.kill()
                self.text = ""
        else:
            self.text = ""

    def summary(self):
        rows = [r.split(",") for r in self.text.strip().splitlines() if r.count(",") >= 8]
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
            except ValueError:
                continue
            for nm, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm),
                "window": "nvidia-smi every 100 ms from before the timed prefill steps (GPU kept "
                          "busy by untimed steps) through the e2e and decode timing"}


class Replicas:
    """Rank bookkeeping for replica runs: a barrier around timed regions, the
    max of a time over ranks, and the sum of work over ranks.  `dist` is
    torch.distributed (gloo) or None for a single process."""

    def __init__(self, dist, world):
        self.dist, self.world = dist, world

    def barrier(self):
        if self.dist is not None:
            self.dist.barrier()

    def max(self, x: float) -> float:
        return self._reduce(x, "MAX")

    def sum(self, x: float) -> float:
        return self._reduce(x, "SUM")

    def _reduce(self, x, op):
        if self.dist is None:
            return float(x)
        import torch
        t = torch.tensor([float(x)], dtype=torch.float64)
        self.dist.all_reduce(t, op=getattr(self.dist.ReduceOp, op))
        return float(t.item())


def throughput(units_all_ranks: float, ms_max: float) -> float:
    """Whole-job rate: the units every rank processed over the slowest rank's time."""
    return units_all_ranks / (ms_max * 1e-3)


# ------------------------------------------------------------------ ours
def run_ours(args, rank, world, local_rank, dist):
    import torch

    import gdn_inputs
    import hybrid_linear_attention_deltanet_gb300 as gdn

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    gdn.load()
    stream = torch.cuda.current_stream(dev)
    peaks = load_peaks()

    rep = Replicas(dist, world)
    barrier, max_over_ranks = rep.barrier, rep.max

    case = gdn_inputs.prefill_8k()
    x = gdn_inputs.make_prefill(case, device=dev)
    out = torch.empty_like(x["v"])
    S_final = torch.empty_like(x["S0"])

    def step():
        gdn.prefill(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["S0"], out=out,
                    S_final=S_final)

    for _ in range(args.warmup):
        step()
    assert gdn.device_status() == 0
    torch.cuda.synchronize(dev)

    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(dev.index)
    sampler.__enter__()
    # nvidia-smi needs a moment to start sampling: keep the GPU busy with
    # untimed prefill steps meanwhile, so the sampled window holds the timed
    # steps (and the e2e and decode timing after them) under load
    t_spin = time.perf_counter() + 0.6
    while time.perf_counter() < t_spin:
        step()
        torch.cuda.synchronize(dev)
    barrier()
    torch.cuda.synchronize(dev)
    n0 = gdn.kernel_launches()
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    n1 = gdn.kernel_launches()
    barrier()
    assert gdn.device_status() == 0
    ms_local = ev0.elapsed_time(ev1) / args.steps
    ms = max_over_ranks(ms_local)
    tokens = case.total_tokens
    value = throughput(rep.sum(tokens), ms) / 1e6
    flops = prefill_flops(case.lengths)
    achieved_tf = flops / (ms_local * 1e-3) / 1e12
    path = gdn.prefill_path(case.io_dtype)

    # ---- end to end, through the same public call, as a serving loop would
    # run it: pinned host buffers, two device buffer sets, and one stream each
    # for host-to-device copies, compute and device-to-host copies, so that
    # the inputs of step i+1 and the outputs of step i-1 travel while step i
    # computes.  Every step copies all its inputs in and its outputs out
    # inside the timed region (pipeline fill and drain included).
    names = ("q", "k", "v", "alpha", "beta", "S0")
    host = {n: x[n].cpu().pin_memory() for n in names}
    dset = [{n: torch.empty_like(x[n]) for n in names} for _ in range(2)]
    douts = [(torch.empty_like(out), torch.empty_like(S_final)) for _ in range(2)]
    h_out = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    h_sf = [torch.empty(S_final.shape, dtype=S_final.dtype).pin_memory() for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_cmp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    for e in ev_in + ev_cmp + ev_out:
        e.record(stream)

    def e2e_step(i):
        b = i & 1
        s_in.wait_event(ev_cmp[b])            # step i-2 has finished reading set b
        with torch.cuda.stream(s_in):
            for n in names:
                dset[b][n].copy_(host[n], non_blocking=True)
        ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        stream.wait_event(ev_out[b])          # step i-2's outputs have left set b
        xb = dset[b]
        gdn.prefill(xb["q"], xb["k"], xb["v"], xb["alpha"], xb["beta"], xb["S0"],
                    out=douts[b][0], S_final=douts[b][1])
        ev_cmp[b].record(stream)
        s_out.wait_event(ev_cmp[b])
        with torch.cuda.stream(s_out):
            h_out[b].copy_(douts[b][0], non_blocking=True)
            h_sf[b].copy_(douts[b][1], non_blocking=True)
        ev_out[b].record(s_out)

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    e2e_steps = max(3, min(args.steps, 10))
    barrier()
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_start.record(s_in)
    for i in range(e2e_steps):
        e2e_step(i)
    e_end.record(s_out)
    torch.cuda.synchronize(dev)
    barrier()
    assert gdn.device_status() == 0
    e2e_ms = max_over_ranks(e_start.elapsed_time(e_end) / e2e_steps)
    h2d = sum(host[n].numel() * host[n].element_size() for n in names)
    d2h = h_out[0].numel() * h_out[0].element_size() + h_sf[0].numel() * h_sf[0].element_size()

    # ---- decode: 1000 consecutive steps over 256 sequences
    dcase = gdn_inputs.decode_256x1000()
    dsteps = dcase.steps
    d = gdn_inputs.make_decode(dcase, device=dev)
    S = d["S"].clone()
    dout = torch.empty(d["v"].shape[1:], dtype=d["v"].dtype, device=dev)
    for t in range(3):
        gdn.decode_step(d["q"][t], d["k"][t], d["v"][t], d["alpha"][t], d["beta"][t], S, out=dout)
    S.copy_(d["S"])
    torch.cuda.synchronize(dev)
    barrier()
    dn0 = gdn.kernel_launches()
    ev0.record(stream)
    for t in range(dsteps):
        gdn.decode_step(d["q"][t], d["k"][t], d["v"][t], d["alpha"][t], d["beta"][t], S, out=dout)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    dn1 = gdn.kernel_launches()
    barrier()
    assert gdn.device_status() == 0
    sampler.__exit__(None, None, None)
    d_ms_local = ev0.elapsed_time(ev1) / dsteps
    d_ms = max_over_ranks(d_ms_local)
    dbytes = decode_bytes(dcase.N)
    d_gbs_local = dbytes / (d_ms_local * 1e-3) / 1e9

    # ---- dv = 512 (the value expansion dv = 2 dk of Table 8): decode over the
    # same 256 sequences and the 8K prefill, each timed on its own
    dcase5 = gdn_inputs.decode_256_dv512()
    d5 = gdn_inputs.make_decode(dcase5, device=dev)
    S5 = d5["S"]
    dout5 = torch.empty(d5["v"].shape[1:], dtype=d5["v"].dtype, device=dev)
    for t in range(3):
        gdn.decode_step(d5["q"][t], d5["k"][t], d5["v"][t], d5["alpha"][t], d5["beta"][t], S5,
                        out=dout5)
    torch.cuda.synchronize(dev)
    ev0.record(stream)
    for t in range(dcase5.steps):
        gdn.decode_step(d5["q"][t], d5["k"][t], d5["v"][t], d5["alpha"][t], d5["beta"][t], S5,
                        out=dout5)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    d5_ms = max_over_ranks(ev0.elapsed_time(ev1) / dcase5.steps)
    del d5, S5, dout5
    pcase5 = gdn_inputs.prefill_8k_dv512()
    x5 = gdn_inputs.make_prefill(pcase5, device=dev)
    out5, sf5 = torch.empty_like(x5["v"]), torch.empty_like(x5["S0"])
    step5 = lambda: gdn.prefill(x5["q"], x5["k"], x5["v"], x5["alpha"], x5["beta"], x5["S0"],
                                out=out5, S_final=sf5)
    for _ in range(2):
        step5()
    torch.cuda.synchronize(dev)
    p5_steps = 5
    ev0.record(stream)
    for _ in range(p5_steps):
        step5()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    assert gdn.device_status() == 0
    p5_ms = max_over_ranks(ev0.elapsed_time(ev1) / p5_steps)
    del x5, out5, sf5

    # ---- the 64K single-sequence prefill: gdn_prefill (which cuts a sequence
    # of 1024 chunks into 7 segments) and the uncut chain (gdn_prefill_scan
    # with one segment per sequence) beside it
    c64 = gdn_inputs.prefill_64k()
    x64 = gdn_inputs.make_prefill(c64, device=dev)
    o64 = torch.empty_like(x64["v"])
    s64 = torch.empty((1, H, DV, DK), dtype=torch.float32, device=dev)
    p64_plain = lambda: gdn.prefill(x64["q"], x64["k"], x64["v"], x64["alpha"], x64["beta"], None,
                                    out=o64, S_final=s64)
    p64_scan = lambda: gdn.prefill_scan(x64["q"], x64["k"], x64["v"], x64["alpha"], x64["beta"],
                                        None, segments=1, out=o64, S_final=s64)

    def time_calls(fn, n=5):
        for _ in range(2):
            fn()
        torch.cuda.synchronize(dev)
        ev0.record(stream)
        for _ in range(n):
            fn()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        return ev0.elapsed_time(ev1) / n

    p64_ms = time_calls(p64_plain)
    p64s_ms = time_calls(p64_scan)
    assert gdn.device_status() == 0
    f64 = prefill_flops(c64.lengths)
    del x64, o64, s64

    # ---- the small fp32 prefill (the 1e-4 parity workload, CUDA-core path)
    # and the packed varlen prefill of 16 sequences of U[1024, 65536] tokens
    c0 = gdn_inputs.prefill_small_fp32()
    x0 = gdn_inputs.make_prefill(c0, device=dev)
    p0 = lambda: gdn.prefill(x0["q"], x0["k"], x0["v"], x0["alpha"], x0["beta"], x0["S0"])
    p0_ms = time_calls(p0, n=20)
    f0 = prefill_flops(c0.lengths)
    del x0
    cv = gdn_inputs.prefill_varlen16()
    xv = gdn_inputs.make_prefill(cv, device=dev)
    ov = torch.empty_like(xv["v"])
    sv = torch.empty_like(xv["S0"])
    pv = lambda: gdn.prefill(xv["q"], xv["k"], xv["v"], xv["alpha"], xv["beta"], xv["S0"],
                             xv["cu_seqlens"], out=ov, S_final=sv)
    pv_ms = time_calls(pv, n=5)
    assert gdn.device_status() == 0
    fv = prefill_flops(cv.lengths)
    del xv, ov, sv

    # ---- backward of the 8K prefill (gdn_prefill_backward), dout and dS_final
    # drawn once; each call recomputes the forward internally
    bx = x
    gen_b = torch.Generator(device=dev)
    gen_b.manual_seed(11)
    b_dout = torch.randn(bx["v"].shape, generator=gen_b, device=dev).to(bx["v"].dtype)
    b_dsf = torch.randn(bx["S0"].shape, generator=gen_b, device=dev) * 0.1
    bstep = lambda: gdn.prefill_backward(bx["q"], bx["k"], bx["v"], bx["alpha"], bx["beta"],
                                         b_dout, bx["S0"], b_dsf)
    for _ in range(2):
        bstep()
    torch.cuda.synchronize(dev)
    bn0 = gdn.kernel_launches()
    ev0.record(stream)
    b_steps = 3
    for _ in range(b_steps):
        bstep()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    assert gdn.device_status() == 0
    bw_ms = max_over_ranks(ev0.elapsed_time(ev1) / b_steps)
    bw_launches = int(gdn.kernel_launches() - bn0) // b_steps
    bw_flops = backward_flops(case.lengths)
    del b_dout, b_dsf

    # ---- the layer steps around the recurrence on the 8K workload
    # (gdn_prepare: conv + SiLU, q/k L2 norm, gates; gdn_output_norm_gate:
    # Eq. 20's gated RMSNorm) and one decode step's gdn_prepare_decode_step
    lcase = gdn_inputs.layer_8k()
    lx = gdn_inputs.make_layer(lcase, device=dev)
    lstate = torch.empty_like(lx["conv_state"])
    lstep = lambda: gdn.prepare(lx["qkv"], lx["conv_w"], lx["a_raw"], lx["b_raw"], lx["A_log"],
                                lx["dt_bias"], lcase.H, conv_state_in=lx["conv_state"],
                                conv_state_out=lstate)
    lo = torch.randn(lx["g"].shape, device=dev).to(lx["g"].dtype)
    ly = torch.empty_like(lo)
    gstep = lambda: gdn.output_norm_gate(lo, lx["g"], lx["norm_w"], 1e-5, "silu", y=ly)

    def time_it(fn, n):
        for _ in range(3):
            fn()
        torch.cuda.synchronize(dev)
        c0 = gdn.kernel_launches()
        ev0.record(stream)
        for _ in range(n):
            fn()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        return ev0.elapsed_time(ev1) / n, int(gdn.kernel_launches() - c0) // n

    prep_ms, prep_launch = time_it(lstep, 10)
    ng_ms, ng_launch = time_it(gstep, 10)
    assert gdn.device_status() == 0
    prep_b = prepare_bytes(lcase.total_tokens, len(lcase.lengths))
    ng_b = norm_gate_bytes(lcase.total_tokens * lcase.H)
    # the whole mixer core over the same inputs: gdn_prefill_layer (the
    # pre-recurrence steps inside the prefill's prep, the gated RMSNorm inside
    # its state pass) against the three separate calls
    lS0 = torch.randn((len(lcase.lengths), lcase.H, lcase.dv, lcase.dk), device=dev) * 0.02
    lsf = torch.empty_like(lS0)
    lyf = torch.empty_like(lx["g"])
    fstep = lambda: gdn.prefill_layer(lx["qkv"], lx["conv_w"], lx["a_raw"], lx["b_raw"],
                                      lx["A_log"], lx["dt_bias"], lx["g"], lx["norm_w"], lcase.H,
                                      S0=lS0, conv_state_in=lx["conv_state"],
                                      conv_state_out=lstate, y=lyf, S_final=lsf)

    def three_step():
        p = gdn.prepare(lx["qkv"], lx["conv_w"], lx["a_raw"], lx["b_raw"], lx["A_log"],
                        lx["dt_bias"], lcase.H, conv_state_in=lx["conv_state"],
                        conv_state_out=lstate)
        o, _ = gdn.prefill(p["q"], p["k"], p["v"], p["alpha"], p["beta"], lS0, S_final=lsf)
        gdn.output_norm_gate(o, lx["g"], lx["norm_w"], 1e-5, "silu", y=lyf)

    lf_ms, lf_launch = time_it(fstep, 10)
    l3_ms, l3_launch = time_it(three_step, 10)
    assert gdn.device_status() == 0
    del lx, lstate, lo, ly, lS0, lsf, lyf
    dl = gdn_inputs.layer_decode_256()
    dl_steps = 200
    gen = torch.Generator(device=dev)
    gen.manual_seed(dl.seed)
    dqkv = torch.randn((dl_steps, len(dl.lengths), dl.channels), generator=gen,
                       device=dev).to(dl.io_dtype)
    dlx = gdn_inputs.make_layer(dl, device=dev)
    dl_out = gdn.prepare_decode_step(dlx["qkv"], dlx["conv_w"], dlx["a_raw"], dlx["b_raw"],
                                     dlx["A_log"], dlx["dt_bias"], dlx["conv_state"], dl.H)
    dl_i = [0]

    def dstep():
        gdn.prepare_decode_step(dqkv[dl_i[0] % dl_steps], dlx["conv_w"], dlx["a_raw"],
                                dlx["b_raw"], dlx["A_log"], dlx["dt_bias"], dlx["conv_state"],
                                dl.H, out=dl_out)
        dl_i[0] += 1

    # a step this small is bound by the host's call rate, so the 200 steps are
    # replayed from a CUDA graph, as a serving loop would run them
    for _ in range(3):
        dstep()
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            for _ in range(dl_steps):
                dstep()
    stream.wait_stream(cap)
    graph.replay()
    torch.cuda.synchronize(dev)
    ev0.record(stream)
    graph.replay()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    pd_ms = ev0.elapsed_time(ev1) / dl_steps
    assert gdn.device_status() == 0
    del graph
    pd_b = prepare_bytes(len(dl.lengths), len(dl.lengths))
    # the whole mixer core of a decode step: fused (one cluster launch) and as
    # three calls (prepare, recurrence, gated RMSNorm), 200 consecutive steps
    # over 256 sequences with fresh projections each step
    S_l = torch.randn((len(dl.lengths), dl.H, dl.dv, dl.dk), generator=gen, device=dev) * 0.02
    dgate = torch.randn((dl_steps, len(dl.lengths), dl.H, dl.dv), generator=gen,
                        device=dev).to(dl.io_dtype)
    y_l = torch.empty_like(dgate[0])
    o_l = torch.empty_like(dgate[0])
    fl_i = [0]

    def fused_step():
        i = fl_i[0] % dl_steps
        gdn.decode_layer_step(dqkv[i], dlx["conv_w"], dlx["a_raw"], dlx["b_raw"], dlx["A_log"],
                              dlx["dt_bias"], dlx["conv_state"], S_l, dgate[i], dlx["norm_w"],
                              1e-5, "silu", y=y_l)
        fl_i[0] += 1

    def three_calls():
        i = fl_i[0] % dl_steps
        p = gdn.prepare_decode_step(dqkv[i], dlx["conv_w"], dlx["a_raw"], dlx["b_raw"],
                                    dlx["A_log"], dlx["dt_bias"], dlx["conv_state"], dl.H,
                                    out=dl_out)
        gdn.decode_step(p["q"], p["k"], p["v"], p["alpha"], p["beta"], S_l, out=o_l)
        gdn.output_norm_gate(o_l, dgate[i], dlx["norm_w"], 1e-5, "silu", y=y_l)
        fl_i[0] += 1

    fused_ms, fused_launch = time_it(fused_step, dl_steps)
    three_ms, three_launch = time_it(three_calls, dl_steps)
    assert gdn.device_status() == 0
    C_l = dl.channels
    nl = len(dl.lengths)
    fused_b = (decode_bytes(nl) - nl * dl.H * (3 * 512 + 8)      # state, out -> y, gates
               + nl * (C_l * 2 + 2 * 3 * C_l * 2 + dl.H * 8) + nl * dl.H * dl.dv * 2
               + C_l * 16 + dl.dv * 4)
    del dqkv, dlx, dl_out, S_l, dgate, y_l, o_l

    res = None
    if rank == 0:
        clocks = sampler.summary()
        cpu = cpu_baseline(args)
        res = {
            "metric": METRIC,
            "value": round(value, 4),
            "unit": "Mtok/s/layer",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(ms, 4),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16" if path.startswith("tcgen05") else "f32",
            "data": "synthetic",
            "config": {
                "workload": case.name,
                "global_batch": 4 * world, "seq_len": 8192, "heads": H, "head_dim": DK,
                "chunk": C, "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                "prefill_path": path,
                "l2": "inputs larger than L2 (q, k, v = 302 MB per step)",
            },
            "roofline": {
                "bound": "tensor",
                "achieved": round(achieved_tf, 3),
                "peak": peaks["bf16"],
                "unit": "TFLOP/s",
                "frac": round(achieved_tf / peaks["bf16"], 5),
                "traffic": ncu_traffic("prefill"),
                "kernel": "whole gdn_prefill call (chunk prep + state pass)",
                "counted_flops_per_launch": flops,
                "peak_source": f"{peaks['src']} bf16 dense (burst)",
                "hbm_gbs_achieved": round(prefill_bytes(case.lengths) / (ms_local * 1e-3) / 1e9, 2),
            },
            "cpu_baseline": cpu,
            "e2e": {"value": round(throughput(tokens * world, e2e_ms) / 1e6, 4),
                    "unit": "Mtok/s/layer", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": round(e2e_ms, 4),
                    "pipeline": "two buffer sets; H2D of step i+1 and D2H of step i-1 "
                                "overlap step i on separate streams"},
            "gpu_launches": int(n1 - n0),
            "dv512": {
                "decode": {"workload": dcase5.name,
                           "value": round(throughput(decode_bytes(dcase5.N, dv=512) * world,
                                                     d5_ms) / 1e9, 2),
                           "unit": "GB/s", "ms_per_step": round(d5_ms, 4),
                           "frac_of_hbm": round(decode_bytes(dcase5.N, dv=512) / (d5_ms * 1e-3)
                                                / 1e9 / peaks["hbm_gbs"], 4)},
                "prefill": {"workload": pcase5.name,
                            "value": round(throughput(pcase5.total_tokens * world, p5_ms) / 1e6, 4),
                            "unit": "Mtok/s/layer", "ms_per_step": round(p5_ms, 4),
                            "path": gdn.prefill_path(pcase5.io_dtype),
                            "counted_tflops": round(prefill_flops(pcase5.lengths, dv=512)
                                                    / (p5_ms * 1e-3) / 1e12, 3)},
            },
            "prefill_small_fp32": {
                "workload": c0.name,
                "value": round(throughput(c0.total_tokens * world, p0_ms) / 1e6, 4),
                "unit": "Mtok/s/layer", "ms_per_step": round(p0_ms, 4),
                "path": gdn.prefill_path(c0.io_dtype),
                "roofline": {"bound": "alu", "unit": "TFLOP/s",
                             "achieved": round(f0 / (p0_ms * 1e-3) / 1e12, 3),
                             "peak": round(FP32_FMA_TFLOPS, 1),
                             "frac": round(f0 / (p0_ms * 1e-3) / 1e12 / FP32_FMA_TFLOPS, 4),
                             "traffic": ncu_traffic("prefill_fp32"),
                             "counted_flops_per_launch": f0,
                             "peak_source": "fp32 FMA of the CUDA cores: 152 SMs x 128 lanes "
                                            "x 2 FLOP x 2.07 GHz",
                             "l2": "inputs (9.4 MB) fit in L2: traffic is near compulsory"},
            },
            "prefill_varlen16": {
                "workload": cv.name,
                "value": round(throughput(cv.total_tokens * world, pv_ms) / 1e6, 4),
                "unit": "Mtok/s/layer", "ms_per_step": round(pv_ms, 4),
                "tokens": cv.total_tokens,
                "roofline": {"bound": "tensor", "unit": "TFLOP/s",
                             "achieved": round(fv / (pv_ms * 1e-3) / 1e12, 3),
                             "peak": peaks["bf16"],
                             "frac": round(fv / (pv_ms * 1e-3) / 1e12 / peaks["bf16"], 5),
                             "traffic": ncu_traffic("prefill_varlen16"),
                             "counted_flops_per_launch": fv,
                             "kernel": "whole gdn_prefill call (segment plan, chunk prep, "
                                       "state passes, scan)",
                             "peak_source": f"{peaks['src']} bf16 dense (burst)"},
            },
            "prefill_64k": {
                "workload": c64.name,
                "gdn_prefill": {"ms_per_step": round(p64_ms, 4),
                                "value": round(c64.total_tokens / (p64_ms * 1e-3) / 1e6, 3),
                                "unit": "Mtok/s/layer",
                                "counted_tflops": round(f64 / (p64_ms * 1e-3) / 1e12, 2),
                                "roofline": {
                                    "bound": "tensor", "unit": "TFLOP/s",
                                    "achieved": round(f64 / (p64_ms * 1e-3) / 1e12, 3),
                                    "peak": peaks["bf16"],
                                    "frac": round(f64 / (p64_ms * 1e-3) / 1e12 / peaks["bf16"], 5),
                                    "traffic": ncu_traffic("prefill_64k"),
                                    "counted_flops_per_launch": f64,
                                    "kernel": "whole gdn_prefill call (7 segments: chunk prep, "
                                              "two state passes, scan)",
                                    "peak_source": f"{peaks['src']} bf16 dense (burst)"}},
                "uncut_chain": {
                    "ms_per_step": round(p64s_ms, 4),
                    "value": round(c64.total_tokens / (p64s_ms * 1e-3) / 1e6, 3),
                    "unit": "Mtok/s/layer",
                    "counted_tflops": round(f64 / (p64s_ms * 1e-3) / 1e12, 2)},
            },
            "backward": {
                "workload": case.name + " (gdn_prefill_backward, dout and dS_final given)",
                "ms_per_step": round(bw_ms, 3),
                "value": round(throughput(tokens * world, bw_ms) / 1e6, 3),
                "unit": "Mtok/s/layer",
                "launches_per_step": bw_launches,
                "roofline": {"bound": "tensor", "unit": "TFLOP/s",
                             "achieved": round(bw_flops / (bw_ms * 1e-3) / 1e12, 3),
                             "peak": round(TF32_TFLOPS(peaks), 1),
                             "frac": round(bw_flops / (bw_ms * 1e-3) / 1e12 / TF32_TFLOPS(peaks), 4),
                             "executed_flops_per_call": bw_flops,
                             "peak_source": f"tf32 dense = {peaks['src']} bf16 burst x 1.1 / 2.25 "
                                            "(nominal tf32 : bf16)"},
                "path": "chunked form: forward re-run (bf16 tensor cores) storing the "
                        "chunk-start states, reverse state pass on the bf16 tensor cores, "
                        "chunk-gradient GEMMs on the tf32 tensor cores, T and the C x C terms "
                        "on the CUDA cores",
            },
            "layer_prefill": {
                "workload": lcase.name + " (gdn_prefill_layer: projections in, y out)",
                "ms_per_step": round(lf_ms, 4),
                "value": round(throughput(lcase.total_tokens * world, lf_ms) / 1e6, 4),
                "unit": "Mtok/s/layer", "launches_per_step": lf_launch,
                "three_calls_ms_per_step": round(l3_ms, 4),
                "three_calls_launches_per_step": l3_launch,
                "path": "pre-recurrence steps as their own pass, then the fused prefill "
                        "whose per-chunk workers apply the gated RMSNorm behind the chains"},
            "layer_steps": {
                "prepare": {"workload": lcase.name + " (gdn_prepare)",
                            "ms_per_step": round(prep_ms, 4),
                            "value": round(prep_b / (prep_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                            "algorithmic_bytes_per_launch": prep_b,
                            "frac_of_hbm": round(prep_b / (prep_ms * 1e-3) / 1e9
                                                 / peaks["hbm_gbs"], 4),
                            "mtok_per_s": round(lcase.total_tokens / (prep_ms * 1e-3) / 1e6, 2),
                            "launches_per_step": prep_launch},
                "output_norm_gate": {"workload": lcase.name + " (gdn_output_norm_gate)",
                                     "ms_per_step": round(ng_ms, 4),
                                     "value": round(ng_b / (ng_ms * 1e-3) / 1e9, 2),
                                     "unit": "GB/s", "algorithmic_bytes_per_launch": ng_b,
                                     "frac_of_hbm": round(ng_b / (ng_ms * 1e-3) / 1e9
                                                          / peaks["hbm_gbs"], 4),
                                     "launches_per_step": ng_launch},
                "prepare_decode_step": {"workload": dl.name + f" x{dl_steps} steps (CUDA graph)",
                                        "ms_per_step": round(pd_ms, 5),
                                        "value": round(pd_b / (pd_ms * 1e-3) / 1e9, 2),
                                        "unit": "GB/s", "algorithmic_bytes_per_launch": pd_b},
                "decode_layer_step": {
                    "workload": "fused decode step of the mixer core, 256 sequences x 6 heads, "
                                f"bf16, x{dl_steps} steps (gdn_decode_layer_step)",
                    "ms_per_step": round(fused_ms, 5),
                    "value": round(fused_b / (fused_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                    "frac_of_hbm": round(fused_b / (fused_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                    "algorithmic_bytes_per_launch": fused_b,
                    "launches_per_step": fused_launch,
                    "three_calls_ms_per_step": round(three_ms, 5),
                    "three_calls_launches_per_step": three_launch},
            },
            "clocks": clocks,
            "decode": {
                "workload": dcase.name,
                "value": round(throughput(dbytes * world, d_ms) / 1e9, 2), "unit": "GB/s",
                "tokens_per_s": round(throughput(dcase.N * world, d_ms), 1),
                "ms_per_step": round(d_ms, 5), "steps": dsteps,
                "gpu_launches": int(dn1 - dn0),
                "roofline": {"bound": "hbm", "achieved": round(d_gbs_local, 2),
                             "peak": peaks["hbm_gbs"], "unit": "GB/s",
                             "frac": round(d_gbs_local / peaks["hbm_gbs"], 4),
                             "traffic": ncu_traffic("decode"),
                             "algorithmic_bytes_per_launch": dbytes,
                             "peak_source": f"{peaks['src']} HBM copy"},
            },
        }
    return res


def cpu_baseline(args, min_seconds=10.0):
    """The oracle, as it stands, on the prefill workload itself: whole passes
    over all 4 x 8192 tokens of all 4 x 6 (sequence, head) units, repeated
    until at least `min_seconds` of host time have passed (about 10 s of CPU
    work: one pass takes about 2 s on 16 host threads)."""
    import gdn_inputs
    import oracle
    case = gdn_inputs.prefill_8k()
    x = gdn_inputs.make_prefill(case, device="cpu")
    passes, used = 0, 1
    t = time.perf_counter()
    while True:
        _, _, used = oracle.prefill(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["S0"])
        passes += 1
        if time.perf_counter() - t >= min_seconds:
            break
    dt = time.perf_counter() - t
    tok = passes * case.total_tokens
    return {"value": round(tok / dt / 1e6, 8), "unit": "Mtok/s/layer", "cores": int(used),
            "kind": "oracle", "seconds": round(dt, 3),
            "sample": f"{passes} full pass(es) of the prefill workload (4 sequences x 8192 "
                      f"tokens x 6 heads, {tok} token-layers), fp64 token recurrence",
            "nproc": os.cpu_count(), "cpu_model": cpu_model(),
            "single_core": single_core_oracle()}


def cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


def single_core_oracle():
    """The oracle on one host thread over the whole small fp32 workload (512
    tokens x 6 heads), and that per-token-head rate carried over to the other
    prefill workloads (the recurrence costs the same per token and head at
    dk = dv = 256)."""
    import gdn_inputs
    import oracle
    c0 = gdn_inputs.prefill_small_fp32()
    x = gdn_inputs.make_prefill(c0, device="cpu")
    t = time.perf_counter()
    oracle.prefill(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["S0"], nthreads=1)
    dt = time.perf_counter() - t
    rate = c0.total_tokens / dt                      # tokens (x 6 heads) per second
    ext = {c.name: round(c.total_tokens / rate, 1)
           for c in (gdn_inputs.prefill_8k(), gdn_inputs.prefill_64k(),
                     gdn_inputs.prefill_varlen16())}
    return {"value": round(rate / 1e6, 8), "unit": "Mtok/s/layer", "cores": 1,
            "seconds": round(dt, 3), "sample": "the small fp32 workload in full "
                                               f"({c0.total_tokens} tokens x 6 heads)",
            "extrapolated_seconds": ext}


def run_profile(args):
    """Only the library's kernels of one family, for a profiler: W warm-up
    then K steps of the 8K prefill workload, of the 256-sequence decode, of
    the 8K layer steps around the recurrence, or of the 8K backward."""
    import torch

    import gdn_inputs
    import hybrid_linear_attention_deltanet_gb300 as gdn
    dev = torch.device("cuda", 0)
    gdn.load()
    if args.profile == "prefill":
        x = gdn_inputs.make_prefill(gdn_inputs.prefill_8k(), device=dev)
        out, sf = torch.empty_like(x["v"]), torch.empty_like(x["S0"])
        for _ in range(args.warmup + args.steps):
            gdn.prefill(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["S0"], out=out,
                        S_final=sf)
    elif args.profile == "layer_fused":
        # gdn_prefill_layer on the 8K layer inputs, per step
        lc = gdn_inputs.layer_8k()
        lx = gdn_inputs.make_layer(lc, device=dev)
        S0 = torch.randn((len(lc.lengths), lc.H, lc.dv, lc.dk), device=dev) * 0.02
        st = torch.empty_like(lx["conv_state"])
        for _ in range(args.warmup + args.steps):
            gdn.prefill_layer(lx["qkv"], lx["conv_w"], lx["a_raw"], lx["b_raw"], lx["A_log"],
                              lx["dt_bias"], lx["g"], lx["norm_w"], lc.H, S0=S0,
                              conv_state_in=lx["conv_state"], conv_state_out=st)
    elif args.profile in ("prefill_64k", "prefill_fp32", "prefill_varlen8"):
        if args.profile == "prefill_64k":
            c = gdn_inputs.prefill_64k()
        elif args.profile == "prefill_fp32":
            c = gdn_inputs.prefill_small_fp32()
        else:   # the first 8 of the varlen workload's 16 sequences (149K tokens)
            c = gdn_inputs.PrefillCase("varlen prefill N=8 (the first 8 of the N=16 draw) bf16",
                                       gdn_inputs.prefill_varlen16().lengths[:8], seed=4,
                                       varlen=True)
        x = gdn_inputs.make_prefill(c, device=dev)
        for _ in range(args.warmup + args.steps):
            gdn.prefill(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["S0"], x["cu_seqlens"])
    elif args.profile == "backward":
        x = gdn_inputs.make_prefill(gdn_inputs.prefill_8k(), device=dev)
        dout = torch.randn(x["v"].shape, device=dev).to(x["v"].dtype)
        dsf = torch.randn(x["S0"].shape, device=dev) * 0.1
        for _ in range(args.warmup + args.steps):
            gdn.prefill_backward(x["q"], x["k"], x["v"], x["alpha"], x["beta"], dout, x["S0"],
                                 dsf)
    elif args.profile == "tgemm":
        # the backward's tensor-core GEMM in its dO S shape (B' = S in the
        # tiled state layout, bf16 as the forward re-run stores it; K = dv =
        # 256, N = dk = 256) on 1500 units: 197 MB of S, 98 MB each of dO and C
        import ctypes
        f = gdn.load().gdn_testing_tgemm
        vp, i32, i64, fl = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
        f.argtypes = [vp, i64, i32, i32, vp, i64, i32, i32, vp, fl, vp, i64, i32, vp, i64, i32,
                      i32, fl, i32, i64, i32, i32, vp]
        units = 1500
        A = torch.randn(units, 64, 256, device=dev)
        B = torch.randn(units, 256, 256, device=dev).to(torch.bfloat16)
        C = torch.empty(units, 64, 256, device=dev)
        st = torch.cuda.current_stream().cuda_stream
        for _ in range(args.warmup + args.steps):
            assert f(A.data_ptr(), 64 * 256, 256, 0, B.data_ptr(), 256 * 256, 256, 0, None, 0.0,
                     C.data_ptr(), 64 * 256, 256, None, 0, 256, 256, 1.0, 0, units, 256, 1,
                     st) == 0
    elif args.profile == "decode_layer":
        lc = gdn_inputs.layer_decode_256()
        lx = gdn_inputs.make_layer(lc, device=dev)
        S = torch.randn((len(lc.lengths), lc.H, lc.dv, lc.dk), device=dev) * 0.02
        for _ in range(args.warmup + args.steps):
            gdn.decode_layer_step(lx["qkv"], lx["conv_w"], lx["a_raw"], lx["b_raw"], lx["A_log"],
                                  lx["dt_bias"], lx["conv_state"], S,
                                  lx["g"].reshape(len(lc.lengths), lc.H, lc.dv), lx["norm_w"])
    elif args.profile == "layer":
        # gdn_prepare then gdn_output_norm_gate on the 8K layer inputs, per step
        lc = gdn_inputs.layer_8k()
        lx = gdn_inputs.make_layer(lc, device=dev)
        st = torch.empty_like(lx["conv_state"])
        o = torch.randn(lx["g"].shape, device=dev).to(lx["g"].dtype)
        for _ in range(args.warmup + args.steps):
            gdn.prepare(lx["qkv"], lx["conv_w"], lx["a_raw"], lx["b_raw"], lx["A_log"],
                        lx["dt_bias"], lc.H, conv_state_in=lx["conv_state"], conv_state_out=st)
            gdn.output_norm_gate(o, lx["g"], lx["norm_w"], 1e-5, "silu")
    else:
        case = gdn_inputs.decode_256x1000()
        d = gdn_inputs.make_decode(case, device=dev, steps=args.warmup + args.steps)
        S = d["S"]
        for t in range(args.warmup + args.steps):
            gdn.decode_step(d["q"][t], d["k"][t], d["v"][t], d["alpha"][t], d["beta"][t], S)
    torch.cuda.synchronize(dev)
    assert gdn.device_status() == 0


# ------------------------------------------------------------- reference
def run_reference(args, rank):
    if rank != 0:
        return None
    import gdn_inputs
    import oracle
    case = gdn_inputs.prefill_8k()
    x = gdn_inputs.make_prefill(case, device="cpu")
    sample_tokens = 512    # per (sequence, head) unit per step: a bounded sample
    for w in range(args.warmup):
        sl = {n: x[n][:, :64].contiguous() for n in ("q", "k", "v", "alpha", "beta")}
        oracle.prefill(sl["q"], sl["k"], sl["v"], sl["alpha"], sl["beta"], x["S0"])
    times, used = [], 1
    for s in range(args.steps):
        a = (s * sample_tokens) % 8192
        sl = {n: x[n][:, a:a + sample_tokens].contiguous() for n in ("q", "k", "v", "alpha", "beta")}
        t = time.perf_counter()
        _, _, used = oracle.prefill(sl["q"], sl["k"], sl["v"], sl["alpha"], sl["beta"], x["S0"])
        times.append(time.perf_counter() - t)
    ms = 1e3 * sum(times) / len(times)
    tok = 4 * sample_tokens
    value = tok / (ms * 1e-3) / 1e6
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 8), "unit": "Mtok/s/layer",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": case.name, "global_batch": 4, "seq_len": 8192, "heads": H,
                   "head_dim": DK, "parallelism": "host cores (OpenMP over sequence x head)"},
        "cpu_baseline": {"value": round(value, 8), "unit": "Mtok/s/layer", "cores": int(used),
                         "kind": "oracle",
                         "sample": f"each step: {sample_tokens} consecutive tokens of all 4 x 6 "
                                   f"(sequence, head) units of the prefill workload"},
        "e2e": {"value": round(value, 8), "unit": "Mtok/s/layer", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--profile", choices=["prefill", "decode", "layer", "backward", "tgemm",
                                          "decode_layer",
                                          "prefill_64k", "prefill_fp32", "prefill_varlen8",
                                          "layer_fused"],
                    default=None,
                    help="run only W + K steps of one kernel family (for ncu captures); "
                         "prints no benchmark line")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if args.profile:
        run_profile(args)
        return
    if args.impl == "reference":
        res = run_reference(args, rank)
    else:
        if world > 1:
            import torch.distributed as dist_mod
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            dist_mod.init_process_group("gloo", rank=rank, world_size=world)
            dist = dist_mod
        res = run_ours(args, rank, world, local_rank, dist)
        if dist is not None:
            dist.barrier()
            dist.destroy_process_group()
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
