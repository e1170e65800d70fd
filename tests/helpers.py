"""Shared test helpers: run the CUDA path and the fp64 oracle on the same seeded bytes and
compare them matrix by matrix with the relative Frobenius error."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from linear_attention_state_gdn_gb300 import synth

# relative Frobenius error bound per matrix, by input dtype
TOL = {torch.float32: 1e-4, torch.float64: 1e-4, torch.bfloat16: 2e-2}
COMPOSE_TOL = 1e-4   # compose inputs are fp32 tensors


def f64(t):
    return None if t is None else t.detach().double().cpu().numpy()


def to_dev(inp: synth.SegmentInputs, device="cuda"):
    return {n: t.to(device) for n, t in inp.tensors().items()}


def gpu_build(inp, device="cuda", **kw):
    import linear_attention_state_gdn_gb300 as hy
    d = to_dev(inp, device)
    S, lam, P = hy.hypic_build_segments(inp.family, d["k"], d["v"], inp.seg_offsets,
                                        log_gate=d.get("log_gate"),
                                        log_gamma=d.get("log_gamma"), beta=d.get("beta"), **kw)
    torch.cuda.synchronize()
    assert hy.hypic_get_device_status() == 0
    return S, lam, P


def oracle_build(inp, want_T=True):
    return oracle.build_segments(inp.family, inp.seg_offsets, f64(inp.k), f64(inp.v),
                                 f64(inp.log_gate), f64(inp.log_gamma), f64(inp.beta),
                                 want_T=want_T)


def oracle_seq(inp, S0=None):
    return oracle.run_sequential(inp.family, inp.seg_offsets, f64(inp.k), f64(inp.v),
                                 f64(inp.log_gate), f64(inp.log_gamma), f64(inp.beta), S0=S0)


def gpu_T(family, lam, P, d):
    """Dense fp64 T from the library's (lam, P) storage."""
    return oracle.materialize_T(family, f64(lam), f64(P), d_k=d)


def rel_errors(got, ref, lead_dims=2):
    """Relative Frobenius error of every matrix (the last two axes); matrices whose
    reference is exactly zero report the absolute norm of got instead."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    g = got.reshape(-1, got.shape[-2] * got.shape[-1])
    r = ref.reshape(-1, ref.shape[-2] * ref.shape[-1])
    num = np.linalg.norm(g - r, axis=1)
    den = np.linalg.norm(r, axis=1)
    return np.where(den > 0, num / np.where(den > 0, den, 1), num)


def assert_close(got, ref, tol, what=""):
    e = rel_errors(got, ref)
    worst = float(e.max()) if e.size else 0.0
    assert worst <= tol, f"{what}: max rel-Frobenius error {worst:.3e} > {tol:.1e}"
    return worst


def slice_heads(inp, heads):
    """The inputs of a subset of value heads, each paired with its own key head (so the
    sliced problem has H_k = H_v = len(heads) and no key sharing)."""
    g = inp.H_v // inp.H_k
    kh = [h // g for h in heads]
    out = synth.SegmentInputs(inp.family, inp.dtype, len(heads), len(heads), inp.d_k, inp.d_v,
                              inp.seg_offsets, inp.k[:, kh].contiguous(),
                              inp.v[:, heads].contiguous(), meta=dict(inp.meta))
    for n in ("log_gate", "beta"):
        t = getattr(inp, n)
        setattr(out, n, None if t is None else t[:, heads].contiguous())
    if inp.log_gamma is not None:
        out.log_gamma = inp.log_gamma[heads].contiguous()
    return out


def kernel_code_hash(name):
    """Hash of the code of a kernel source under csrc/ (comments and blank lines do not
    count). The host models of a kernel's protocol or layout record the hash of the source
    they were checked against, so that an edit to the kernel fails them until the model has
    been re-checked against the new code and the recorded hash updated."""
    import hashlib
    import os
    import re
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    path = os.path.join(root, "linear_attention_state_gdn_gb300", "csrc", name)
    with open(path) as f:
        text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
    h = hashlib.sha1()
    for line in text.splitlines():
        code = line.split("//", 1)[0].rstrip()
        if code:
            h.update(code.encode() + b"\n")
    return h.hexdigest()[:12]
