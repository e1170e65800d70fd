#!/usr/bin/env python
"""Benchmark of the HYPIC linear-layer state path on one GB300 (or N replicas).

One step = the whole hot path on the GDN workload: one hybrid linear layer with 32 value /
16 key heads, d_k = d_v = 128, one 32768-token cold prompt split into 16 segments of 2048
tokens (bf16 k L2-normalised, bf16 v, fp32 gates and beta), built into all 512
(S(C|0), T_C) pairs in one launch, then prefix-scan composed across the 16 segments in a
second launch. `value` is build+compose tokens/s of that step with the inputs resident in
device memory; `e2e` is the same metric through the public API with the inputs copied in
from pinned host memory and every output copied back, inside the timed region (the segments
in eight groups, so that each group's copies overlap the previous group's build and compose).

The other workloads (RetNet scalar build + compose, GLA diagonal build + compose, the same
GDN prompt cached as one 32768-token segment, the RetNet prompt as one 16384-token segment,
the channel-gated delta rule (KDA) at the GDN shape, the GDN build that also returns the
segment outputs O(C|0), the 48-layer x 64-segment GDN compose with and without the composed
entry) are measured after the main timed region and reported under "sections", each with the
oracle timed on the host cores beside it and the parity of its outputs against that oracle. `--impl reference` times the fp64 CPU oracle instead (a bounded sample
of the same workload per step, on the host cores).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl hypic|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GDN (S,T_C) build tokens/s + compose/scan GB/s, % of GB300 roofline"
# sources whose code the recorded build traffic belongs to (the launches and how the call
# splits and merges segments)
TRAFFIC_SOURCES = ["build_gdn_prep.cu", "build_gdn_tc.cu", "compose_tc.cu", "api.cu"]
UNIT = "tokens/s"
CHUNK = 64
L2_FLUSH_BYTES = 256 << 20

# algorithmic work per token per value head of the chunked (C = 64) WY/UT GDN build:
# gram 2Cd + W 2Cd + U 2Cd + X = W[S|P] 2d(2d) + state update 2d(2d); the channel-gated (KDA)
# chunked build has the same products (its gram, of the gated keys, per value head)
GDN_FLOP_PER_TOKEN_HEAD = 6 * CHUNK * 128 + 8 * 128 * 128   # 180,224
# the exact sequential form (one thread per state column), per token per value head, d = 128:
# the gate d^2 (a product per state element; KDA also on P), k^T z 2d^2 and the rank-1
# update 2d^2 on each of the S and P halves, and o = S^T q 2d^2 when the outputs are read
SEQ_D = 128
SEQ_FLOP_PER_TOKEN_HEAD = {"kda": 2 * 5 * SEQ_D * SEQ_D, "gdn": (5 + 4) * SEQ_D * SEQ_D}
SEQ_OUT_FLOP = 2 * SEQ_D * SEQ_D
# the segment outputs on the chunked form, per token per value head: Q S 2d^2, the chunk's
# Q K^T 2Cd and its masked product with the delta values 2Cd
GDN_OUT_FLOP_PER_TOKEN_HEAD = 2 * 128 * 128 + 4 * CHUNK * 128   # 65,536


# ----------------------------------------------------------------------------- helpers

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return dict(hbm_gbs=d["hbm_gbs"], bf16_tflops=d["bf16_tflops"],
                    bf16_tflops_sustained=d.get("bf16_tflops_sustained"),
                    sm_max_mhz=d.get("sm_max_mhz", 2070.0), source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0,
                sm_max_mhz=2070.0, source="fallback")


def fp32_alu_peak_tflops(sm_mhz):
    """FFMA peak: 152 SMs x 128 fp32 lanes x 2 flop x clock."""
    return 152 * 128 * 2 * sm_mhz * 1e6 / 1e12


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    if world > 1 and not torch.distributed.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, world: int, device="cpu") -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(units_per_rank: float, max_seconds: float, world: int) -> float:
    """Whole-job throughput: units processed by all ranks / the slowest rank's time."""
    return units_per_rank * world / max_seconds


def src_hash(*names):
    """Hash of the code of the named kernel sources: comments and blank lines do not count,
    so that a recorded measurement stays valid across comment-only edits."""
    import re
    h = hashlib.sha1()
    for n in names:
        with open(os.path.join(ROOT, "linear_attention_state_gdn_gb300", "csrc", n)) as f:
            text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
        for line in text.splitlines():
            code = line.split("//", 1)[0].rstrip()
            if code:
                h.update(code.encode() + b"\n")
    return h.hexdigest()[:12]


def recorded_traffic(kernel: str, source_files):
    """DRAM bytes per launch recorded from an ncu capture of this exact kernel source
    (profiles/traffic.json); None when absent or when the source changed since."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(kernel)
    if not rec or rec.get("src") != src_hash(*source_files):
        return None
    return rec.get("bytes_per_launch")


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index=0):
        self.proc = None
        self.dev = device_index

    def start(self):
        try:
            ident = str(self.dev)
            try:
                u = torch.cuda.get_device_properties(self.dev).uuid
                ident = "GPU-" + str(u)
            except Exception:
                pass
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", ident, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.15)

    def stop(self):
        if self.proc is None:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=["nvidia-smi unavailable"],
                        samples=0)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, p in zip(names, parts[4:8]):
                if p.lower().startswith("active"):
                    reasons.add(n)
        return dict(sm_mhz=statistics.median(sm) if sm else None,
                    sm_max_mhz=max(smax) if smax else None, reasons=sorted(reasons),
                    samples=len(sm))


# ----------------------------------------------------------------------------- workloads

def gdn_algorithmic_bytes(n_tok, H_k, H_v, d, n_seg):
    """Bytes the GDN build must move: k, v (bf16), log a and beta (fp32) in; S and P
    (fp32) and lam out."""
    inputs = n_tok * (H_k * d * 2 + H_v * d * 2 + H_v * 8)
    outputs = n_seg * H_v * (2 * d * d * 4 + 4)
    return inputs + outputs


def compose_algorithmic_bytes(n_seg, units, d, dense, diag=False, s0=False):
    """Compose scan bytes: read S_j and lam_j (and P_j for j >= 1 when dense), write
    prefix_j."""
    st = d * d * 4
    per_unit = n_seg * (2 * st + (d * 4 if diag else 4))
    if dense:
        per_unit += (n_seg - 1 + (1 if s0 else 0)) * st
    if s0:
        per_unit += st
    return per_unit * units


def make_workspace(hy, inp, dev, device):
    """The build's device scratch (allocated once, outside every timed region), or None."""
    need = hy.hypic_build_workspace_bytes(inp.family, dev["k"], dev["v"], inp.seg_offsets,
                                          log_gate=dev.get("log_gate"),
                                          log_gamma=dev.get("log_gamma"), beta=dev.get("beta"))
    return torch.empty(need, dtype=torch.uint8, device=device) if need else None


class Step:
    """Device buffers and the two launches of one step of a workload."""

    def __init__(self, inp, device):
        import linear_attention_state_gdn_gb300 as hy
        self.hy = hy
        self.inp = inp
        self.dev = {n: t.to(device) for n, t in inp.tensors().items()}
        self.S, self.lam, self.P = hy.build_outputs(inp.family, inp.n_seg, inp.H_v, inp.d_v,
                                                    device)
        self.prefix = torch.empty_like(self.S)
        self.workspace = make_workspace(hy, inp, self.dev, device)

    def build(self):
        d = self.dev
        self.hy.hypic_build_segments(self.inp.family, d["k"], d["v"], self.inp.seg_offsets,
                                     log_gate=d.get("log_gate"), log_gamma=d.get("log_gamma"),
                                     beta=d.get("beta"), S=self.S, lam=self.lam, P=self.P,
                                     workspace=self.workspace)

    def compose(self):
        self.hy.hypic_compose_scan(self.inp.family, self.S, self.lam, self.P,
                                   prefix=self.prefix)

    def kernel_names(self):
        d = self.dev
        b = self.hy.hypic_build_kernel_name(self.inp.family, d["k"], d["v"], self.inp.seg_offsets,
                                            log_gate=d.get("log_gate"),
                                            log_gamma=d.get("log_gamma"), beta=d.get("beta"),
                                            S=self.S, lam=self.lam, P=self.P)
        c = self.hy.hypic_compose_kernel_name(self.inp.family, self.S, self.lam, self.P)
        return b, c


def time_loop(fns, steps, warmup, flush):
    """Run `steps` iterations of the launches in `fns` after `warmup` untimed ones, with an
    L2 flush between iterations (outside the events). Returns per-function lists of
    milliseconds and the per-iteration totals."""
    for _ in range(warmup):
        for f in fns:
            f()
    torch.cuda.synchronize()
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in fns] for _ in range(steps)]
    for it in range(steps):
        flush.zero_()
        for (a, b), f in zip(ev[it], fns):
            a.record()
            f()
            b.record()
    torch.cuda.synchronize()
    per_fn = [[ev[it][i][0].elapsed_time(ev[it][i][1]) for it in range(steps)]
              for i in range(len(fns))]
    totals = [sum(per_fn[i][it] for i in range(len(fns))) for it in range(steps)]
    return per_fn, totals


def build_gdn_compose_cache(layers=48, device="cuda"):
    """The 48-layer x 32-head x 64-segment GDN cache: every layer drawn on the device and
    built into unit slice [layer*32, layer*32+32) of one [64, 1536, 128, 128] cache."""
    import ctypes
    import linear_attention_state_gdn_gb300 as hy
    from linear_attention_state_gdn_gb300 import synth
    info = synth.workload_info("gdn_compose")
    H, d, n_seg = info["H_v"], info["d"], len(info["seg_lens"])
    units = layers * H
    S, lam, P = hy.build_outputs("gdn", n_seg, units, d, device)
    lib = hy.load_library()
    stream = torch.cuda.current_stream().cuda_stream
    ws = None
    for layer in range(layers):
        inp = synth.make_workload_device("gdn_compose", layer, device)
        a = hy.make_build_args("gdn", inp.k, inp.v, inp.seg_offsets, inp.log_gate, None,
                               inp.beta, None, None, None, out_seg_stride=units)
        a.S = S.data_ptr() + layer * H * d * d * 4
        a.lam = lam.data_ptr() + layer * H * 4
        a.P = P.data_ptr() + layer * H * d * d * 4
        need = int(lib.hypic_build_workspace_bytes(ctypes.byref(a)))
        if need and (ws is None or ws.numel() < need):
            torch.cuda.synchronize()   # the previous layer's build may still read the old one
            ws = torch.empty(need, dtype=torch.uint8, device=device)
        if need:
            a.workspace, a.workspace_bytes = ws.data_ptr(), ws.numel()
        st = lib.hypic_build_segments(ctypes.byref(a), stream)
        if st != 0:
            raise hy.HypicError(st, "hypic_build_segments (gdn_compose cache)")
        del inp
    torch.cuda.synchronize()
    return S, lam, P, dict(info, units=units)


# ----------------------------------------------------------------------------- sections

def section_family(name, flush, peak, steps=20, warmup=3, oracle_budget_s=0.0):
    from linear_attention_state_gdn_gb300 import synth
    inp = synth.make_workload(name)
    st = Step(inp, "cuda")
    (tb, tc), _ = time_loop([st.build, st.compose], steps, warmup, flush)
    b_ms, c_ms = statistics.mean(tb), statistics.mean(tc)
    n_tok, d = inp.n_tok, inp.d_k
    dense = inp.family in ("gdn", "delta", "kda")
    gate_bytes = n_tok * inp.H_v * (d if inp.family in ("diag", "kda") else 1) * 4 \
        if inp.log_gate is not None else 0
    beta_bytes = n_tok * inp.H_v * 4 if inp.beta is not None else 0
    b_bytes = n_tok * (inp.H_k + inp.H_v) * d * 2 + gate_bytes + beta_bytes + \
        inp.n_seg * inp.H_v * (d * d * 4 * (2 if dense else 1) + (d * 4 if inp.family == "diag" else 4))
    c_bytes = compose_algorithmic_bytes(inp.n_seg, inp.H_v, d, dense, inp.family == "diag")
    bk, ck = st.kernel_names()
    b_gbs, c_gbs = b_bytes / b_ms / 1e6, c_bytes / c_ms / 1e6
    extra = {}
    if bk in ("build_gdn_tc", "build_kda_tc"):   # tensor-bound: the chunked-form flops against the bf16 peak
        tf = GDN_FLOP_PER_TOKEN_HEAD * n_tok * inp.H_v / (b_ms * 1e-3) / 1e12
        extra = {"build_tflops": round(tf, 1), "build_tensor_frac": round(tf / peak["bf16_tflops"], 4)}
    elif bk == "build_seq":    # fp32 CUDA-core bound: the sequential form against the FFMA peak
        tf = SEQ_FLOP_PER_TOKEN_HEAD[inp.family] * n_tok * inp.H_v / (b_ms * 1e-3) / 1e12
        alu = fp32_alu_peak_tflops(peak["sm_max_mhz"])
        extra = {"build_tflops": round(tf, 2), "build_alu_frac": round(tf / alu, 4),
                 "alu_peak_tflops": round(alu, 1)}
    out = {"build_kernel": bk, "build_ms": round(b_ms, 4), **extra,
           "build_tokens_per_s": round(n_tok / b_ms * 1e3, 1),
           "build_gbs": round(b_gbs, 1), "build_hbm_frac": round(b_gbs / peak["hbm_gbs"], 4),
           "build_bytes": b_bytes, "compose_kernel": ck, "compose_ms": round(c_ms, 4),
           "compose_gbs": round(c_gbs, 1), "compose_hbm_frac": round(c_gbs / peak["hbm_gbs"], 4),
           "compose_bytes": c_bytes}
    if oracle_budget_s:
        torch.cuda.synchronize()
        out["cpu_baseline"] = cpu_baseline(inp, gpu=(st.S, st.lam, st.P, st.prefix),
                                           budget_s=oracle_budget_s)
        out["parity"] = out["cpu_baseline"].pop("parity")
    return out


def section_outputs(name, flush, peak, steps=10, warmup=3, oracle_budget_s=0.0):
    """The build of a workload that also returns the segment outputs O(C|0) (queries drawn
    with the workload), against the roofline of the path it takes (the tensor-core GDN build:
    the bf16 peak; the exact sequential path: the fp32 FFMA peak); the oracle leg times
    oracle.outputs on a sample of heads and reports the parity of O there."""
    import linear_attention_state_gdn_gb300 as hy
    from linear_attention_state_gdn_gb300 import synth
    inp = synth.make_workload(name, with_q=True)
    dev = {n: t.cuda() for n, t in inp.tensors().items()}
    S, lam, P = hy.build_outputs(inp.family, inp.n_seg, inp.H_v, inp.d_v, "cuda")
    O = torch.empty_like(dev["v"])
    kw = dict(log_gate=dev.get("log_gate"), log_gamma=dev.get("log_gamma"), beta=dev.get("beta"))
    f = lambda: hy.hypic_build_segments(inp.family, dev["k"], dev["v"], inp.seg_offsets, S=S,
                                        lam=lam, P=P, q=dev["q"], O=O, **kw)
    (tb,), _ = time_loop([f], steps, warmup, flush)
    ms = statistics.mean(tb)
    bk = hy.hypic_build_kernel_name(inp.family, dev["k"], dev["v"], inp.seg_offsets, S=S, lam=lam,
                                    P=P, q=dev["q"], O=O, **kw)
    out = {"build_kernel": bk, "build_ms": round(ms, 4), "build_tokens_per_s": round(inp.n_tok / ms * 1e3, 1)}
    if bk == "build_gdn_tc":   # the chunked form's flops (S, T and O) against the bf16 peak
        flop = (GDN_FLOP_PER_TOKEN_HEAD + GDN_OUT_FLOP_PER_TOKEN_HEAD) * inp.n_tok * inp.H_v
        tf = flop / (ms * 1e-3) / 1e12
        out.update({"build_tflops": round(tf, 1), "build_tensor_frac": round(tf / peak["bf16_tflops"], 4)})
    else:                      # the sequential form against the FFMA peak
        flop = (SEQ_FLOP_PER_TOKEN_HEAD[inp.family] + SEQ_OUT_FLOP) * inp.n_tok * inp.H_v
        tf = flop / (ms * 1e-3) / 1e12
        alu = fp32_alu_peak_tflops(peak["sm_max_mhz"])
        out.update({"build_tflops": round(tf, 2), "build_alu_frac": round(tf / alu, 4),
                    "alu_peak_tflops": round(alu, 1)})
    if oracle_budget_s:
        torch.cuda.synchronize()
        out["cpu_baseline"] = outputs_cpu_baseline(inp, O, oracle_budget_s)
        out["parity"] = out["cpu_baseline"].pop("parity")
    return out


def section_conv_warmup(flush, peak, steps=20, warmup=3, oracle_heads=0, K=4):
    """The convolution-state warm-up on the GDN workload's prompt (16 x 2048 tokens, 32 value /
    16 key heads, d = 128) with a width-4 short convolution. Outside the timed region: each
    segment's rest (its tokens from K - 1 on) is built from the segment's own convolution
    (torch's grouped conv1d prepares the cache's inputs) with the library's build. Timed: the
    hypic_conv_warmup call, which convolves the 16 x 3 head tokens in context, builds their
    entries and composes each before its rest. Its algorithmic bytes: the rests' entries read,
    the entries in context written, the head tokens' raw k, v and the taps. The oracle leg runs
    oracle.conv_warmup on the first key head's value heads from the same rests."""
    import torch.nn.functional as F
    import linear_attention_state_gdn_gb300 as hy
    from linear_attention_state_gdn_gb300 import synth
    inp = synth.make_workload("gdn")
    dev = {n: t.cuda() for n, t in inp.tensors().items()}
    d, Hk, Hv, n_seg = inp.d_k, inp.H_k, inp.H_v, inp.n_seg
    offs = [int(x) for x in inp.seg_offsets]
    g = torch.Generator().manual_seed(2026)
    wk = (torch.randn(Hk * d, K, generator=g) * 0.5).cuda()
    wv = (torch.randn(Hv * d, K, generator=g) * 0.5).cuda()

    def local_conv(x, w, H, normalize):   # each segment convolved on its own (zeros before it)
        out = torch.empty(x.shape, dtype=torch.float32, device="cuda")
        for j in range(n_seg):
            a, b = offs[j], offs[j + 1]
            seg = x[a:b].float().reshape(b - a, H * d).t().unsqueeze(0)
            y = F.silu(F.conv1d(F.pad(seg, (K - 1, 0)), w.unsqueeze(1), groups=H * d))[0].t()
            y = y.reshape(b - a, H, d)
            if normalize:
                n = y.norm(dim=2, keepdim=True)
                y = torch.where(n > 0, y / torch.where(n > 0, n, torch.ones_like(n)), torch.zeros_like(y))
            out[a:b] = y
        return out

    kl = local_conv(dev["k"], wk, Hk, True)
    vl = local_conv(dev["v"], wv, Hv, False)
    hl = [min(K - 1, offs[j + 1] - offs[j]) for j in range(n_seg)]
    keep = torch.cat([torch.arange(offs[j] + hl[j], offs[j + 1]) for j in range(n_seg)]).cuda()
    r_offs = np.concatenate([[0], np.cumsum([offs[j + 1] - offs[j] - hl[j] for j in range(n_seg)])])
    S_r, lam_r, P_r = hy.hypic_build_segments("gdn", kl[keep].to(torch.bfloat16).contiguous(),
                                              vl[keep].to(torch.bfloat16).contiguous(), r_offs,
                                              log_gate=dev["log_gate"][keep].contiguous(),
                                              beta=dev["beta"][keep].contiguous())
    del kl, vl
    S, lam, P = torch.empty_like(S_r), torch.empty_like(lam_r), torch.empty_like(P_r)
    need = hy.hypic_warmup_workspace_bytes("gdn", offs, dev["k"], dev["v"], wk, wv, S_r, lam_r,
                                           P_rest=P_r, log_gate=dev["log_gate"], beta=dev["beta"],
                                           S=S, lam=lam, P=P)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    f = lambda: hy.hypic_conv_warmup("gdn", offs, dev["k"], dev["v"], wk, wv, S_r, lam_r, P_r,
                                     log_gate=dev["log_gate"], beta=dev["beta"], S=S, lam=lam, P=P,
                                     workspace=ws)
    (tw,), _ = time_loop([f], steps, warmup, flush)
    ms = statistics.mean(tw)
    units = n_seg * Hv
    rows = sum(hl)
    nbytes = 2 * units * (2 * d * d * 4 + 4) + rows * (Hk + Hv) * d * 2 + (Hk + Hv) * d * K * 4
    gbs = nbytes / ms / 1e6
    out = {"kernels": "conv_heads + build_seq (heads) + compose_dense_tc (head before rest)",
           "conv_k": K, "units": units, "head_tokens": rows, "warmup_ms": round(ms, 4),
           "warmup_bytes": nbytes, "warmup_gbs": round(gbs, 1),
           "warmup_hbm_frac": round(gbs / peak["hbm_gbs"], 4),
           "note": "the head entries go through the workspace (written by the head build, read "
                   "by the composition), so DRAM traffic exceeds these algorithmic bytes"}
    if oracle_heads:
        import oracle
        torch.cuda.synchronize()
        hv = sample_heads(inp, oracle_heads)
        hk = hv // (Hv // Hk)
        f64 = lambda t: t.double().cpu().numpy()
        t0 = time.perf_counter()
        S_o, T_o = oracle.conv_warmup(
            "gdn", offs, f64(inp.k[:, :hk]), f64(inp.v[:, :hv]), f64(wk[:hk * d]), f64(wv[:hv * d]), K,
            f64(S_r[:, :hv]), f64(lam_r[:, :hv]), f64(P_r[:, :hv]),
            log_gate=f64(inp.log_gate[:, :hv]), beta=f64(inp.beta[:, :hv]))
        secs = time.perf_counter() - t0
        e_S = rel_frob_max(f64(S[:, :hv]), S_o)
        e_T = rel_frob_max(oracle.materialize_T("gdn", f64(lam[:, :hv]), f64(P[:, :hv])), T_o)
        out["cpu_baseline"] = {"value": round(secs * Hv / hv * 1e3, 1), "unit": "ms per call (scaled)",
                               "cores": oracle.default_threads(), "kind": "oracle",
                               "sample": f"oracle.conv_warmup of all {n_seg} segments x {hv} of {Hv} "
                                         f"value heads from the same rests; ms scaled by {Hv}/{hv}"}
        out["parity"] = {"S": float(f"{e_S:.4g}"), "T": float(f"{e_T:.4g}"), "tol": 1e-4,
                         "ok": bool(e_S <= 1e-4 and e_T <= 1e-4),
                         "units": f"{n_seg} segments x {hv} of {Hv} value heads"}
    return out


def section_gdn_compose(flush, peak, steps=10, warmup=3, layers=48, oracle_units=0):
    import linear_attention_state_gdn_gb300 as hy
    S, lam, P, info = build_gdn_compose_cache(layers)
    prefix = torch.empty_like(S)
    f = lambda: hy.hypic_compose_scan("gdn", S, lam, P, prefix=prefix)
    (tc,), _ = time_loop([f], steps, warmup, flush)
    ms = statistics.mean(tc)
    nbytes = compose_algorithmic_bytes(S.shape[0], S.shape[1], S.shape[2], True)
    gbs = nbytes / ms / 1e6
    out = {"compose_kernel": hy.hypic_compose_kernel_name("gdn", S, lam, P),
           "units": int(S.shape[1]), "n_seg": int(S.shape[0]), "compose_ms": round(ms, 4),
           "compose_bytes": nbytes, "compose_gbs": round(gbs, 1),
           "compose_hbm_frac": round(gbs / peak["hbm_gbs"], 4)}
    # the same launch also composing the 64 entries of every unit into one: lam_total and
    # P_total = P_63 ... P_0. Algorithmic bytes add P_0 read once and the totals written;
    # the transition chain's second read of P_1 .. P_63 counts as overhead.
    U, d = S.shape[1], S.shape[2]
    lam_t = torch.empty(U, dtype=torch.float32, device=S.device)
    P_t = torch.empty((U, d, d), dtype=torch.float32, device=S.device)
    g = lambda: hy.hypic_compose_scan("gdn", S, lam, P, prefix=prefix, lam_total=lam_t, P_total=P_t)
    (tt,), _ = time_loop([g], steps, warmup, flush)
    ms_t = statistics.mean(tt)
    nbytes_t = nbytes + U * (2 * d * d * 4 + 4)
    out["with_totals"] = {"compose_ms": round(ms_t, 4), "compose_bytes": nbytes_t,
                          "compose_gbs": round(nbytes_t / ms_t / 1e6, 1),
                          "compose_hbm_frac": round(nbytes_t / ms_t / 1e6 / peak["hbm_gbs"], 4)}
    if oracle_units:
        # one unit per layer, each a different head, spread over the whole cache
        H = info["H_v"]
        units = [l * H + (7 * l) % H for l in range(S.shape[1] // H)][:oracle_units]
        torch.cuda.synchronize()
        out["cpu_baseline"] = compose_cpu_baseline(S, lam, P, prefix, units, lam_t, P_t)
        out["parity"] = out["cpu_baseline"].pop("parity")
    del S, lam, P, prefix, lam_t, P_t
    torch.cuda.empty_cache()
    return out


# ----------------------------------------------------------------------------- CPU oracle
# The cpu_baseline legs below are the only places this file executes the oracle: they time
# it on the host cores and, from the same pass, report how far the GPU results of the timed
# workload are from it (max relative Frobenius error per matrix, computed in fp64).

def rel_frob_max(got, ref):
    """Largest relative Frobenius error over the matrices (last two axes) of `got` against
    `ref`, in fp64; a matrix whose reference is exactly zero counts its absolute norm."""
    g = np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    g = g.reshape(-1, g.shape[-2] * g.shape[-1])
    r = r.reshape(-1, r.shape[-2] * r.shape[-1])
    num = np.linalg.norm(g - r, axis=1)
    den = np.linalg.norm(r, axis=1)
    e = np.where(den > 0, num / np.where(den > 0, den, 1.0), num)
    return float(e.max()) if e.size else 0.0


def sample_heads(inp, heads):
    """Value heads [0, heads) rounded down to whole key-head groups (at least one group)."""
    g = inp.H_v // inp.H_k
    return max(g, min(inp.H_v, heads) // g * g)


def oracle_step_sample(inp, heads, nthreads, want=False):
    """One oracle step on a sample: all segments of the first `heads` value heads (a whole
    number of key-head groups, with their key heads): fp64 build of (S, T) plus the fp64
    compose scan. Returns the seconds taken and, with `want`, (S, T, prefix)."""
    import oracle
    heads = sample_heads(inp, heads)
    hk = heads // (inp.H_v // inp.H_k)
    f = lambda t: None if t is None else t.double().numpy()
    k = np.ascontiguousarray(f(inp.k)[:, :hk])
    v = np.ascontiguousarray(f(inp.v)[:, :heads])
    lg = None if inp.log_gate is None else np.ascontiguousarray(f(inp.log_gate)[:, :heads])
    b = None if inp.beta is None else np.ascontiguousarray(f(inp.beta)[:, :heads])
    lgam = None if inp.log_gamma is None else np.ascontiguousarray(f(inp.log_gamma)[:heads])
    t0 = time.perf_counter()
    S, T = oracle.build_segments(inp.family, inp.seg_offsets, k, v, lg, lgam, b,
                                 nthreads=nthreads)
    pref = oracle.compose_scan(T, S, nthreads=nthreads)
    dt = time.perf_counter() - t0
    return (dt, (S, T, pref)) if want else dt


def build_parity(inp, heads, ref, gpu):
    """Errors of the GPU's S, T (= exp(lam) P materialised in fp64) and prefix states for
    value heads [0, heads) against the oracle's (S, T, prefix) of the same heads."""
    import oracle
    S_o, T_o, pref_o = ref
    S, lam, P, prefix = gpu
    d = inp.d_k
    h = slice(0, heads)
    f = lambda t: None if t is None else t[:, h].double().cpu().numpy()
    T = oracle.materialize_T(inp.family, f(lam), f(P), d_k=d)
    out = {"S": rel_frob_max(f(S), S_o), "T": rel_frob_max(T, T_o)}
    if prefix is not None:
        out["prefix"] = rel_frob_max(f(prefix), pref_o)
    tol = 1e-4 if inp.dtype == torch.float32 else 2e-2
    out = {k: float(f"{v:.3e}") for k, v in out.items()}
    out.update({"tol": tol, "ok": all(v <= tol for v in out.values()),
                "units": f"{inp.n_seg} segments x {heads} of {inp.H_v} value heads"})
    return out


def cpu_baseline(inp, gpu=None, budget_s=12.0, min_passes=1):
    """The oracle as it stands, on the host cores, on a bounded sample of the workload
    sized to roughly `budget_s` seconds; reported as tokens/s of the whole workload. With
    the GPU's outputs of the same inputs (S, lam, P, prefix), the last pass's oracle results
    also give the parity of those outputs on the sampled heads."""
    import oracle
    threads = oracle.default_threads()
    # calibration: one key-head group (n_seg units each); h heads take about h times as long
    t1 = max(oracle_step_sample(inp, 1, threads), 1e-3)
    g = inp.H_v // inp.H_k
    heads = sample_heads(inp, int(budget_s / t1 * g))
    # whole passes over the sample until the budget is used (the full workload can take
    # less than the budget on many cores)
    dt, passes, ref = 0.0, 0, None
    while passes < min_passes or dt < budget_s:
        t, ref = oracle_step_sample(inp, heads, threads, want=True)
        dt += t
        passes += 1
    tok_per_s = inp.n_tok * heads / inp.H_v * passes / dt
    out = {"value": round(tok_per_s, 2), "unit": UNIT, "cores": threads, "kind": "oracle",
           "seconds": round(dt, 2),
           "sample": f"fp64 oracle build (S, T) + compose of all {inp.n_seg} segments x "
                     f"{heads} of {inp.H_v} value heads ({inp.n_tok} tokens each), "
                     f"{passes} pass(es); tokens/s scaled by {heads}/{inp.H_v}"}
    if gpu is not None:
        out["parity"] = build_parity(inp, heads, ref, gpu)
    return out


def outputs_cpu_baseline(inp, O, budget_s):
    """oracle.outputs on the first value heads of the workload (a whole number of key-head
    groups, about budget_s seconds), timed on the host cores, and the parity of the GPU's O
    on those heads: the largest relative Frobenius error over the (segment, head) blocks."""
    import oracle
    threads = oracle.default_threads()
    g = inp.H_v // inp.H_k
    f = lambda t, hs: None if t is None else np.ascontiguousarray(t.double().numpy()[:, hs])

    def run(heads):
        hk = heads // g
        t0 = time.perf_counter()
        ref = oracle.outputs(inp.family, inp.seg_offsets, f(inp.k, slice(0, hk)), f(inp.v, slice(0, heads)),
                             f(inp.q, slice(0, hk)), f(inp.log_gate, slice(0, heads)),
                             None if inp.log_gamma is None else inp.log_gamma[:heads].double().numpy(),
                             f(inp.beta, slice(0, heads)), nthreads=threads)
        return time.perf_counter() - t0, ref
    t1, _ = run(g)
    heads = sample_heads(inp, int(budget_s / max(t1, 1e-3) * g))
    dt, ref = run(heads)
    got = O[:, :heads].double().cpu().numpy()
    worst = 0.0
    for j in range(inp.n_seg):
        a, b = int(inp.seg_offsets[j]), int(inp.seg_offsets[j + 1])
        for h in range(heads):
            r = ref[a:b, h]
            worst = max(worst, float(np.linalg.norm(got[a:b, h] - r) / max(np.linalg.norm(r), 1e-300)))
    tol = 1e-4 if inp.dtype == torch.float32 else 2e-2
    return {"value": round(inp.n_tok * heads / inp.H_v / dt, 2), "unit": UNIT, "cores": threads,
            "kind": "oracle", "seconds": round(dt, 2),
            "sample": f"fp64 oracle outputs of all {inp.n_seg} segments x {heads} of {inp.H_v} "
                      f"value heads; tokens/s scaled by {heads}/{inp.H_v}",
            "parity": {"O": float(f"{worst:.3e}"), "tol": tol, "ok": worst <= tol,
                       "units": f"{inp.n_seg} segments x {heads} of {inp.H_v} value heads"}}


def compose_cpu_baseline(S, lam, P, prefix, units, lam_t=None, P_t=None):
    """The oracle's compose scan of the GPU-built fp32 entries (lam, P, S) of the sampled
    units, consumed as data; timed on the host cores (GB/s of the algorithmic compose bytes
    of the sample) and compared with the GPU's prefix states (and composed transitions) of
    the same units."""
    import oracle
    threads = oracle.default_threads()
    f = lambda t: t[:, units].double().cpu().numpy()
    Sd, lamd, Pd = f(S), f(lam), f(P)
    t0 = time.perf_counter()
    T = oracle.materialize_T("gdn", lamd, Pd)
    pref_o = oracle.compose_scan(T, Sd, nthreads=threads)
    dt = time.perf_counter() - t0
    n_seg, U, d = Sd.shape[0], Sd.shape[1], Sd.shape[2]
    nbytes = compose_algorithmic_bytes(n_seg, U, d, True)
    par = {"prefix": float(f"{rel_frob_max(f(prefix), pref_o):.3e}")}
    if lam_t is not None:
        # the composed transition exp(lam_total) P_total, compared at its own scale: P_total
        # may carry a power of two whose exponent lam_total reports
        lt_o, Pt_o = oracle.compose_transitions("gdn", lamd, Pd)
        lt = lam_t[units].double().cpu().numpy()
        got = P_t[units].double().cpu().numpy() * np.exp(lt - lt_o)[:, None, None]
        par["T_total"] = float(f"{rel_frob_max(got[None], Pt_o[None]):.3e}")
    # The entries are the GDN build of bf16 k / v, so the bound for this workload is the bf16
    # one (2e-2). The comparison here isolates the compose's own arithmetic (the same fp32
    # entries on both sides), so the fp32 bound (1e-4) is reported beside it: the prefix states
    # meet it; the composed transition of 64 GDN transitions does not (tensor-core accumulation
    # rounds toward zero, and those roundings add up along the 63-step chain).
    errs = dict(par)
    par.update({"tol": 2e-2, "ok": all(v <= 2e-2 for v in errs.values()),
                "fp32_tol": 1e-4, "fp32_ok": {k: v <= 1e-4 for k, v in errs.items()},
                "units": f"{n_seg} segments x {U} sampled units"})
    return {"value": round(nbytes / dt / 1e9, 3), "unit": "GB/s", "cores": threads,
            "kind": "oracle", "seconds": round(dt, 2),
            "sample": f"fp64 oracle compose scan of {U} of {S.shape[1]} units x {n_seg} segments "
                      f"(the GPU-built fp32 entries as data); GB/s of the sample's algorithmic bytes",
            "parity": par}


def run_reference(args):
    """--impl reference: the fp64 oracle on the host cores, same metric and workload."""
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    from linear_attention_state_gdn_gb300 import synth
    inp = synth.make_workload("gdn")
    threads = oracle.default_threads()
    t1 = oracle_step_sample(inp, 1, threads)
    # size each step so that warmup + steps end within ~150 s
    per_step_budget = 150.0 / max(1, args.steps + args.warmup)
    g = inp.H_v // inp.H_k
    heads = sample_heads(inp, int(per_step_budget / max(t1, 1e-3) * g))
    for _ in range(args.warmup):
        oracle_step_sample(inp, heads, threads)
    times = [oracle_step_sample(inp, heads, threads) for _ in range(args.steps)]
    total = sum(times)
    tok = inp.n_tok * heads / inp.H_v
    value = tok * args.steps / total
    sample = (f"fp64 oracle build (S, T) + compose of all {inp.n_seg} segments x {heads} of "
              f"{inp.H_v} value heads per step; tokens/s scaled by {heads}/{inp.H_v}")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(total / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(),
            "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def workload_config():
    return {"workload": "gdn: one GDN linear layer, 32 value / 16 key heads, d_k=d_v=128, "
                        "one 32768-token cold prompt as 16 segments x 2048 tokens; bf16 k "
                        "(L2-normalised) and v, fp32 log-gates and beta, fp32 S and T; "
                        "build all 512 (S,T) pairs in one launch + 16-segment prefix-scan "
                        "compose",
            "tokens_per_step": 32768, "segments": 16, "heads_v": 32, "heads_k": 16, "d": 128,
            "l2": "inputs (411 MB) exceed L2; 256 MB L2 flush between timed steps",
            "parallelism": "replicas (one independent workload per GPU)"}


# ----------------------------------------------------------------------------- main arm

def e2e_measure(inp, steps=5, warmup=2, groups=8):
    """Through the public API from pinned host buffers, inside the events: H2D of k, v, log a,
    beta; build; compose; D2H of S, lam, P and the prefix states. The prompt's segments go in
    `groups` consecutive groups so that transfers overlap compute: group g's inputs copy in on
    one stream while group g - 1 builds; each group is composed as soon as it is built,
    starting from the last prefix state of the group before (the scan's own recurrence, so the
    prefix states are the ones one scan over all segments gives); and each group's S, lam, P
    and prefix states copy out on a third stream (each unit's result does not depend on the
    grouping)."""
    import linear_attention_state_gdn_gb300 as hy
    host = {n: t.pin_memory() for n, t in inp.tensors().items()}
    dev = {n: torch.empty_like(t, device="cuda") for n, t in host.items()}
    S, lam, P = hy.build_outputs(inp.family, inp.n_seg, inp.H_v, inp.d_v, "cuda")
    prefix = torch.empty_like(S)
    outs = [S, lam, P, prefix]
    host_out = [torch.empty_like(t, device="cpu").pin_memory() for t in outs]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in outs)
    offs = np.asarray(inp.seg_offsets, dtype=np.int64)
    bounds = [round(g * inp.n_seg / groups) for g in range(groups + 1)]
    grp = [(s0, s1, int(offs[s0]), int(offs[s1])) for s0, s1 in zip(bounds[:-1], bounds[1:]) if s1 > s0]
    sub = lambda d, t0, t1: {n: t[t0:t1] for n, t in d.items()}
    need = max(hy.hypic_build_workspace_bytes(inp.family, dev["k"][t0:t1], dev["v"][t0:t1],
                                              offs[s0:s1 + 1] - t0, log_gate=dev.get("log_gate"),
                                              beta=dev.get("beta")) for s0, s1, t0, t1 in grp)
    workspace = torch.empty(need, dtype=torch.uint8, device="cuda") if need else None
    comp = torch.cuda.current_stream()
    cin, cout = torch.cuda.Stream(), torch.cuda.Stream()

    def one(start_ev):
        cin.wait_event(start_ev)
        cout.wait_event(start_ev)
        loaded = []
        for s0, s1, t0, t1 in grp:            # every group's inputs, in order, on the copy-in stream
            with torch.cuda.stream(cin):
                for n in host:
                    dev[n][t0:t1].copy_(host[n][t0:t1], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(cin)
            loaded.append(ev)
        for (s0, s1, t0, t1), ev in zip(grp, loaded):
            comp.wait_event(ev)
            d = sub(dev, t0, t1)
            hy.hypic_build_segments(inp.family, d["k"], d["v"], offs[s0:s1 + 1] - t0,
                                    log_gate=d.get("log_gate"), log_gamma=dev.get("log_gamma"),
                                    beta=d.get("beta"), S=S[s0:s1], lam=lam[s0:s1], P=P[s0:s1],
                                    workspace=workspace)
            hy.hypic_compose_scan(inp.family, S[s0:s1], lam[s0:s1], None if P is None else P[s0:s1],
                                  S0=prefix[s0 - 1] if s0 > 0 else None, prefix=prefix[s0:s1])
            built = torch.cuda.Event()
            built.record(comp)
            cout.wait_event(built)
            with torch.cuda.stream(cout):
                for h, t in zip(host_out, outs):
                    if t is not None:
                        h[s0:s1].copy_(t[s0:s1], non_blocking=True)
        with torch.cuda.stream(cout):
            done = torch.cuda.Event()
            done.record(cout)
        comp.wait_event(done)

    for _ in range(warmup):
        ev = torch.cuda.Event()
        ev.record(comp)
        one(ev)
    torch.cuda.synchronize()
    ms = []
    for _ in range(steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(comp)
        one(a)
        b.record(comp)
        b.synchronize()
        ms.append(a.elapsed_time(b))
    m = statistics.mean(ms)
    # the copied-out results are the device results
    assert torch.equal(host_out[0], S.cpu()) and torch.equal(host_out[3], prefix.cpu())
    return {"value": round(inp.n_tok / m * 1e3, 1), "unit": UNIT, "ms_per_step": round(m, 4),
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "groups": len(grp)}


def build_split(hy, inp, dev):
    """True when the tensor-core GDN build of `inp` splits segments into pieces (its workspace
    then holds more than the chunk records and their 256-byte tail)."""
    need = hy.hypic_build_workspace_bytes(inp.family, dev["k"], dev["v"], inp.seg_offsets,
                                          log_gate=dev.get("log_gate"), beta=dev.get("beta"))
    records = sum((int(b - a) + CHUNK - 1) // CHUNK for a, b in
                  zip(inp.seg_offsets[:-1], inp.seg_offsets[1:])) * inp.H_v
    return need > records * CHUNK * CHUNK * 2 + 256


def build_launches(kernel_name, split=False):
    """Kernel launches of one hypic_build_segments call on the path `kernel_name`: the GDN
    tensor-core build is the chunk preparation and the chain, plus one compose launch that
    merges pieces when the call splits segments (the 16-segment workload halves its last two)."""
    if kernel_name == "build_gdn_tc":
        return 3 if split else 2
    return 1


def run_main(args):
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    init_dist(world, "nccl")
    import linear_attention_state_gdn_gb300 as hy
    from linear_attention_state_gdn_gb300 import synth
    hy.load_library()
    pk = peaks()
    inp = synth.make_workload("gdn")
    st = Step(inp, "cuda")
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    bk, ck = st.kernel_names()

    # warm-up, then exactly K timed steps bracketed by barrier + synchronize
    for _ in range(args.warmup):
        st.build()
        st.compose()
    torch.cuda.synchronize()
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(2)] for _ in range(args.steps)]
    sampler = ClockSampler(local)
    sampler.start()
    barrier(world)
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for it in range(args.steps):
        flush.zero_()
        (b0, b1), (c0, c1) = ev[it]
        b0.record()
        st.build()
        b1.record()
        c0.record()
        st.compose()
        c1.record()
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - wall0
    clocks = sampler.stop()
    assert hy.hypic_get_device_status() == 0
    build_ms = [ev[i][0][0].elapsed_time(ev[i][0][1]) for i in range(args.steps)]
    comp_ms = [ev[i][1][0].elapsed_time(ev[i][1][1]) for i in range(args.steps)]
    step_ms = [b + c for b, c in zip(build_ms, comp_ms)]
    total_s = max_over_ranks(sum(step_ms) / 1e3, world, "cuda")
    value = aggregate_throughput(inp.n_tok * args.steps, total_s, world)
    ms_per_step = total_s / args.steps * 1e3
    b_ms, c_ms = statistics.mean(build_ms), statistics.mean(comp_ms)

    # roofline of the dominant kernel (the build)
    flops = GDN_FLOP_PER_TOKEN_HEAD * inp.n_tok * inp.H_v
    nbytes = gdn_algorithmic_bytes(inp.n_tok, inp.H_k, inp.H_v, inp.d_k, inp.n_seg)
    tensor_path = bk.endswith("_tc")
    if tensor_path:
        achieved = flops / (b_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 2), "peak": pk["bf16_tflops"],
                "unit": "TFLOP/s", "peak_source": f"{pk['source']} bf16 dense (burst)"}
    else:
        achieved = flops / (b_ms * 1e-3) / 1e12
        alu = fp32_alu_peak_tflops(pk["sm_max_mhz"])
        roof = {"bound": "alu", "achieved": round(achieved, 2), "peak": round(alu, 1),
                "unit": "TFLOP/s",
                "peak_source": "derived: 152 SMs x 128 fp32 FMA lanes x 2 flop x max SM clock"}
    roof["frac"] = round(roof["achieved"] / roof["peak"], 4)
    # the tensor-core GDN build is one call of two or three launches (chunk preparation, the
    # chain, and the compose merging halved segments); the events bracket the call, so the
    # roofline covers all of them
    split = tensor_path and build_split(hy, inp, st.dev)
    roof["kernel"] = ("build_gdn_prep + build_gdn_tc" + (" + compose_dense_tc (merge)" if split else "")
                      if bk == "build_gdn_tc" else bk)
    roof["algorithmic_flop_per_launch"] = flops
    roof["algorithmic_bytes_per_launch"] = nbytes
    roof["achieved_gbs"] = round(nbytes / (b_ms * 1e-3) / 1e9, 1)
    roof["traffic"] = recorded_traffic(bk, TRAFFIC_SOURCES if tensor_path else ["build_simt.cu"])
    comp_bytes = compose_algorithmic_bytes(inp.n_seg, inp.H_v, inp.d_k, True)

    line = {"metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if tensor_path else "f32", "data": "synthetic",
            "config": workload_config(), "roofline": roof,
            "build_ms": round(b_ms, 4), "compose_ms": round(c_ms, 4),
            "compose_gbs": round(comp_bytes / (c_ms * 1e-3) / 1e9, 1),
            "compose_hbm_frac": round(comp_bytes / (c_ms * 1e-3) / 1e9 / pk["hbm_gbs"], 4),
            "kernels": {"build": bk, "compose": ck},
            "gpu_launches": (build_launches(bk, split) + 1) * args.steps,
            "clocks": {k: clocks[k] for k in ("sm_mhz", "sm_max_mhz", "reasons")},
            "clock_samples": clocks["samples"], "wall_s_timed_region": round(wall, 3),
            "peaks": pk}

    if not args.quick:
        # the last timed step's outputs, for the oracle leg's parity check
        gpu_out = tuple(None if t is None else t.cpu() for t in (st.S, st.lam, st.P, st.prefix))
        line["e2e"] = e2e_measure(inp)
        del st
        torch.cuda.empty_cache()
        oracle_leg = rank == 0 and world == 1
        sections = {}
        for name in ("retnet", "gla", "gdn_one_segment", "retnet_one_segment", "kda"):
            sections[name] = section_family(name, flush, pk, oracle_budget_s=4.0 if oracle_leg else 0.0)
        sections["gdn_outputs"] = section_outputs("gdn", flush, pk, oracle_budget_s=4.0 if oracle_leg else 0.0)
        sections["gdn_compose"] = section_gdn_compose(flush, pk, layers=args.compose_layers,
                                                      oracle_units=96 if oracle_leg else 0)
        sections["conv_warmup"] = section_conv_warmup(flush, pk, oracle_heads=2 if oracle_leg else 0)
        line["sections"] = sections
        if oracle_leg:
            line["cpu_baseline"] = cpu_baseline(inp, gpu=gpu_out)
            line["parity"] = line["cpu_baseline"].pop("parity")
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_only(args):
    """Time one workload's launches alone (for profiling runs): build + compose for the
    named workload, or the compose scan alone for gdn_compose."""
    import linear_attention_state_gdn_gb300 as hy
    from linear_attention_state_gdn_gb300 import synth
    torch.cuda.set_device(0)
    hy.load_library()
    pk = peaks()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    if args.only == "gdn_compose":
        out = section_gdn_compose(flush, pk, steps=args.steps, warmup=args.warmup,
                                  layers=args.compose_layers)
    elif args.only == "gdn_outputs":
        out = section_outputs("gdn", flush, pk, steps=args.steps, warmup=args.warmup)
    elif args.only == "conv_warmup":
        out = section_conv_warmup(flush, pk, steps=args.steps, warmup=args.warmup, oracle_heads=2)
    else:
        out = section_family(args.only, flush, pk, steps=args.steps, warmup=args.warmup)
    assert hy.hypic_get_device_status() == 0
    print(json.dumps({"only": args.only, **out}), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["hypic", "reference"], default="hypic")
    ap.add_argument("--quick", action="store_true",
                    help="main timed region only (no e2e, sections or CPU baseline)")
    ap.add_argument("--compose-layers", type=int, default=48)
    ap.add_argument("--only", choices=["gdn", "retnet", "gla", "gdn_tiny", "gdn_compose", "gdn_one_segment",
                                       "retnet_one_segment", "kda", "gdn_outputs", "conv_warmup"],
                    help="time one workload's launches alone (profiling helper; no contract line)")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)     # at least 3 untimed warm-up steps
    if args.impl == "reference":
        return run_reference(args)
    if args.only:
        return run_only(args)
    return run_main(args)


if __name__ == "__main__":
    sys.exit(main())
