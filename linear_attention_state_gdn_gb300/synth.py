"""Seeded synthetic inputs for the segment build and the compose scan.

This module only draws random numbers and shapes them into the inputs the workloads
describe (key/value tensors, gates, segment boundaries, cached (lam, P, S) triples). It
holds none of the recurrence or composition arithmetic, so both the CUDA path and the
fp64 oracle can consume the same bytes from it.

All draws use numpy's PCG64 with a fixed draw order (k, v, gate, beta, then q when the
outputs are wanted, then lengths), are made in float32/float64 on the host and cast once
(round-to-nearest-even) to the input dtype. The oracle receives exactly the cast values,
converted to float64. q is drawn last, so the other inputs of a seed do not depend on
whether it is drawn: (S, T_C) does not read it, only the segment outputs do.

Workloads (all synthetic):

  gdn_tiny      GDN, fp32, 2 heads, d_k=d_v=32, 4 segments x 128 tokens;
                k ~ N(0,1) L2-normalised per token, v ~ N(0,1), beta = sigmoid(N(0,1)),
                log alpha = -0.1 softplus(N(0,1)).
  retnet        scalar decay, bf16, 16 heads, d=128, 8 x 2048 tokens;
                k, v ~ N(0,1)/sqrt(128); gamma_h = 1 - 2^(-5 - 3h/15).
  gla           diagonal gates, bf16, 16 heads, d=128, 16 x 2048 tokens;
                k, v ~ N(0,1)/sqrt(128); log g = logsigmoid(N(0,1))/16 per channel (fp32).
  gdn           GDN, bf16, 32 value / 16 key heads, d=128, one 32768-token prompt as
                16 x 2048; k L2-normalised; beta = sigmoid(N(0,1));
                log alpha = -0.05 softplus(N(0,1)).
  gdn_compose   48 layers x 32 heads, d=128, 64 segments with lengths uniform in
                [256, 1024]; per layer the same draw recipe as ``gdn``.
  kda           the channel-gated delta rule at the ``gdn`` shape (32 value / 16 key heads,
                d=128, 16 x 2048 tokens, bf16); the same recipe with a per-channel
                log alpha = -0.05 softplus(N(0,1)) [N, H_v, d_k].
  q (outputs)   q ~ N(0,1)/sqrt(d) per element, in the input dtype, [N, H_k, d_k].
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

FAMILY_IDS = {"linear": 0, "scalar": 1, "diag": 2, "delta": 3, "gdn": 4, "kda": 5}
DELTA_FAMILIES = ("gdn", "delta", "kda")


@dataclass
class SegmentInputs:
    """Raw inputs of one layer: tensors live on the host (CPU torch tensors)."""
    family: str
    dtype: torch.dtype
    H_k: int
    H_v: int
    d_k: int
    d_v: int
    seg_offsets: np.ndarray                 # int64 [n_seg + 1]
    k: torch.Tensor                         # [N, H_k, d_k] dtype
    v: torch.Tensor                         # [N, H_v, d_v] dtype
    log_gate: Optional[torch.Tensor] = None   # fp32: SCALAR [N,H_v] | DIAG, KDA [N,H_v,d_k] | GDN [N,H_v]
    log_gamma: Optional[torch.Tensor] = None  # fp32 [H_v] (SCALAR constant gate)
    beta: Optional[torch.Tensor] = None       # fp32 [N, H_v]
    q: Optional[torch.Tensor] = None          # [N, H_k, d_k] dtype (segment outputs only)
    meta: dict = field(default_factory=dict)

    @property
    def n_seg(self) -> int:
        return len(self.seg_offsets) - 1

    @property
    def n_tok(self) -> int:
        return int(self.seg_offsets[-1])

    def tensors(self):
        return {n: getattr(self, n) for n in ("k", "v", "log_gate", "log_gamma", "beta", "q")
                if getattr(self, n) is not None}


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def _normal(rng, shape, nthreads: int = 8) -> np.ndarray:
    """float32 N(0,1) of the given shape; large draws are split over independent
    child streams (spawned from rng) and drawn in parallel threads."""
    n = int(np.prod(shape))
    if n < (1 << 22):
        return rng.standard_normal(n, dtype=np.float32).reshape(shape)
    out = np.empty(n, dtype=np.float32)
    parts = 16
    bounds = np.linspace(0, n, parts + 1).astype(np.int64)
    children = rng.spawn(parts)

    def fill(i):
        children[i].standard_normal(out=out[bounds[i]:bounds[i + 1]], dtype=np.float32)

    with ThreadPoolExecutor(max_workers=nthreads) as ex:
        list(ex.map(fill, range(parts)))
    return out.reshape(shape)


def _to(x: np.ndarray, dtype: torch.dtype) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x)).to(dtype)


def _l2norm_rows(x: np.ndarray) -> np.ndarray:
    x64 = x.astype(np.float64)
    nrm = np.sqrt((x64 * x64).sum(axis=-1, keepdims=True))
    return x64 / np.maximum(nrm, 1e-30)


def _softplus(x):
    x = x.astype(np.float64)
    return np.where(x > 20, x, np.log1p(np.exp(np.minimum(x, 20))))


def _logsigmoid(x):
    x = x.astype(np.float64)
    return -_softplus(-x)


def _sigmoid(x):
    x = x.astype(np.float64)
    return 1.0 / (1.0 + np.exp(-x))


def offsets_from_lengths(lengths) -> np.ndarray:
    return np.concatenate([[0], np.cumsum(np.asarray(lengths, dtype=np.int64))]).astype(np.int64)


def make_inputs(family: str, H_k: int, H_v: int, d: int, seg_lens, dtype=torch.bfloat16,
                seed: int = 0, k_scale: Optional[float] = None, l2norm_k: Optional[bool] = None,
                alpha_scale: float = 0.05, beta_shift: float = 0.0, gla_div: float = 16.0,
                retnet_gammas: bool = True, per_token_scalar: bool = False,
                with_q: bool = False) -> SegmentInputs:
    """Draw one layer of inputs for any family at any size (tests use small ragged ones).

    GDN / DELTA / KDA: k L2-normalised (default), v ~ N(0,1), beta = sigmoid(N(0,1) +
                 beta_shift), GDN log alpha = -alpha_scale softplus(N(0,1)) per token, KDA
                 the same per key channel.
    SCALAR:      k, v ~ N(0,1) * k_scale (default 1/sqrt(d)); constant per-head
                 gamma_h = 1 - 2^(-5 - 3h/15) (retnet_gammas) or, with per_token_scalar,
                 a per-token log gate logsigmoid(N(0,1))/gla_div.
    DIAG:        k, v ~ N(0,1) * k_scale; log g = logsigmoid(N(0,1))/gla_div per channel.
    LINEAR:      k, v ~ N(0,1) * k_scale.
    with_q:      q ~ N(0,1) / sqrt(d), drawn after everything else.
    """
    rng = _rng(seed)
    offs = offsets_from_lengths(seg_lens)
    N = int(offs[-1])
    if l2norm_k is None:
        l2norm_k = family in DELTA_FAMILIES
    if k_scale is None:
        k_scale = 1.0 if family in DELTA_FAMILIES else 1.0 / math.sqrt(d)
    k = _normal(rng, (N, H_k, d))
    v = _normal(rng, (N, H_v, d))
    if l2norm_k:
        k = _l2norm_rows(k)
    else:
        k = k * k_scale
    if family not in DELTA_FAMILIES:
        v = v * k_scale
    inp = SegmentInputs(family, dtype, H_k, H_v, d, d, offs, _to(k, dtype), _to(v, dtype))
    if family == "gdn":
        inp.log_gate = _to(-alpha_scale * _softplus(_normal(rng, (N, H_v))), torch.float32)
    elif family == "kda":
        inp.log_gate = _to(-alpha_scale * _softplus(_normal(rng, (N, H_v, d))), torch.float32)
    elif family == "diag":
        inp.log_gate = _to(_logsigmoid(_normal(rng, (N, H_v, d))) / gla_div, torch.float32)
    elif family == "scalar":
        if per_token_scalar:
            inp.log_gate = _to(_logsigmoid(_normal(rng, (N, H_v))) / gla_div, torch.float32)
        elif retnet_gammas:
            h = np.arange(H_v, dtype=np.float64)
            inp.log_gamma = _to(np.log1p(-np.exp2(-5.0 - 3.0 * h / 15.0)), torch.float32)
        else:
            inp.log_gamma = _to(-np.abs(_normal(rng, (H_v,))) * 1e-3, torch.float32)
    if family in DELTA_FAMILIES:
        inp.beta = _to(_sigmoid(_normal(rng, (N, H_v)) + beta_shift), torch.float32)
    if with_q:
        inp.q = _to(_normal(rng, (N, H_k, d)) / math.sqrt(d), dtype)
    return inp


# --------------------------------------------------------------------------------------
# The five named workloads

WORKLOADS = ("gdn_tiny", "retnet", "gla", "gdn", "gdn_compose", "gdn_one_segment", "retnet_one_segment",
             "kda")

WORKLOAD_SEEDS = {"gdn_tiny": 1001, "retnet": 1002, "gla": 1003, "gdn": 1004, "gdn_compose": 1005,
                  "gdn_one_segment": 1006, "retnet_one_segment": 1007, "kda": 1008}


def workload_info(name: str) -> dict:
    """Sizes of a named workload, without drawing anything."""
    if name == "gdn_tiny":
        return dict(family="gdn", dtype="f32", H_k=2, H_v=2, d=32, seg_lens=[128] * 4, layers=1)
    if name == "retnet":
        return dict(family="scalar", dtype="bf16", H_k=16, H_v=16, d=128, seg_lens=[2048] * 8,
                    layers=1)
    if name == "gla":
        return dict(family="diag", dtype="bf16", H_k=16, H_v=16, d=128, seg_lens=[2048] * 16,
                    layers=1)
    if name == "gdn":
        return dict(family="gdn", dtype="bf16", H_k=16, H_v=32, d=128, seg_lens=[2048] * 16,
                    layers=1)
    if name == "retnet_one_segment":   # the RetNet prompt cached as one segment
        return dict(family="scalar", dtype="bf16", H_k=16, H_v=16, d=128, seg_lens=[16384],
                    layers=1)
    if name == "kda":   # the channel-gated delta rule at the GDN shape
        return dict(family="kda", dtype="bf16", H_k=16, H_v=32, d=128, seg_lens=[2048] * 16,
                    layers=1)
    if name == "gdn_one_segment":   # the GDN prompt cached as one segment
        return dict(family="gdn", dtype="bf16", H_k=16, H_v=32, d=128, seg_lens=[32768], layers=1)
    if name == "gdn_compose":
        lens = _rng(WORKLOAD_SEEDS[name]).integers(256, 1024, size=64, endpoint=True)
        return dict(family="gdn", dtype="bf16", H_k=16, H_v=32, d=128,
                    seg_lens=[int(x) for x in lens], layers=48)
    raise KeyError(name)


def make_workload(name: str, layer: int = 0, with_q: bool = False) -> SegmentInputs:
    """Draw the inputs of a named workload (one layer; gdn_compose takes layer in [0, 48));
    with_q also draws the queries the segment outputs read."""
    info = workload_info(name)
    seed = WORKLOAD_SEEDS[name] * 1000 + layer
    fam, d = info["family"], info["d"]
    if name == "gdn_tiny":
        inp = make_inputs("gdn", 2, 2, 32, info["seg_lens"], torch.float32, seed, alpha_scale=0.1,
                          with_q=with_q)
    elif name in ("retnet", "retnet_one_segment"):
        inp = make_inputs("scalar", 16, 16, d, info["seg_lens"], torch.bfloat16, seed, with_q=with_q)
    elif name == "gla":
        inp = make_inputs("diag", 16, 16, d, info["seg_lens"], torch.bfloat16, seed, with_q=with_q)
    else:
        inp = make_inputs(fam, info["H_k"], info["H_v"], d, info["seg_lens"], torch.bfloat16,
                          seed, alpha_scale=0.05, with_q=with_q)
    inp.meta = dict(workload=name, layer=layer, seed=seed, **info)
    return inp


# --------------------------------------------------------------------------------------
# Cached-entry triples for the compose scan

@dataclass
class ComposeInputs:
    family: str
    n_seg: int
    n_units: int
    d_k: int
    d_v: int
    lam: torch.Tensor                   # fp32 [n_seg, U] or [n_seg, U, d_k] (DIAG)
    S: torch.Tensor                     # fp32 [n_seg, U, d_k, d_v]
    P: Optional[torch.Tensor] = None    # fp32 [n_seg, U, d_k, d_k] (DELTA / GDN)
    S0: Optional[torch.Tensor] = None   # fp32 [U, d_k, d_v]


def make_compose_inputs(family: str, n_seg: int, n_units: int, d: int, seed: int = 0,
                        with_S0: bool = False, lam_scale: float = 0.5,
                        p_norm: float = 0.9) -> ComposeInputs:
    """Random cached entries with O(1) transitions, so the carried term matters.

    S ~ N(0,1); lam = -U(0, lam_scale) (a vector per row for DIAG);
    P (DELTA / GDN) = G * p_norm / (2 sqrt(d)) with G ~ N(0,1), whose spectral norm is
    close to p_norm; LINEAR has lam = 0.
    """
    rng = _rng(seed)
    S = _normal(rng, (n_seg, n_units, d, d))
    lam_shape = (n_seg, n_units, d) if family == "diag" else (n_seg, n_units)
    lam = -rng.random(lam_shape, dtype=np.float32) * lam_scale
    if family == "linear":
        lam[:] = 0
    P = None
    if family in DELTA_FAMILIES:
        P = _normal(rng, (n_seg, n_units, d, d)) * np.float32(p_norm / (2.0 * math.sqrt(d)))
    S0 = _normal(rng, (n_units, d, d)) if with_S0 else None
    t = lambda x: None if x is None else torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return ComposeInputs(family, n_seg, n_units, d, d, t(lam), t(S), t(P), t(S0))


# --------------------------------------------------------------------------------------
# Device-side draws for the 48-layer workload (host draws of ~12 G values would take
# minutes). torch's seeded generator on the target device draws the same recipe; a test
# that checks a sample on the host copies the drawn tensors back, so both sides still see
# identical bytes.

def make_inputs_device(family: str, H_k: int, H_v: int, d: int, seg_lens, dtype, seed: int,
                       device="cuda", alpha_scale: float = 0.05) -> SegmentInputs:
    """GDN / DELTA inputs drawn with torch.Generator(device) (recipe as make_inputs)."""
    assert family in ("gdn", "delta")
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    offs = offsets_from_lengths(seg_lens)
    N = int(offs[-1])
    k = torch.randn((N, H_k, d), generator=g, device=device, dtype=torch.float32)
    k = k / k.norm(dim=-1, keepdim=True).clamp_min(1e-30)
    v = torch.randn((N, H_v, d), generator=g, device=device, dtype=torch.float32)
    inp = SegmentInputs(family, dtype, H_k, H_v, d, d, offs, k.to(dtype), v.to(dtype))
    if family == "gdn":
        x = torch.randn((N, H_v), generator=g, device=device, dtype=torch.float32)
        inp.log_gate = (-alpha_scale * torch.nn.functional.softplus(x.double())).float()
    x = torch.randn((N, H_v), generator=g, device=device, dtype=torch.float32)
    inp.beta = torch.sigmoid(x.double()).float()
    return inp


def make_workload_device(name: str, layer: int = 0, device="cuda") -> SegmentInputs:
    """A named GDN workload drawn on `device` (used for the 48-layer gdn_compose cache)."""
    info = workload_info(name)
    assert info["family"] == "gdn" and info["dtype"] == "bf16"
    seed = WORKLOAD_SEEDS[name] * 1000 + layer
    inp = make_inputs_device("gdn", info["H_k"], info["H_v"], info["d"], info["seg_lens"],
                             torch.bfloat16, seed, device=device, alpha_scale=0.05)
    inp.meta = dict(workload=name, layer=layer, seed=seed, drawn_on=str(device), **info)
    return inp


def to_host(inp: SegmentInputs) -> SegmentInputs:
    """Copy of a SegmentInputs with every tensor moved to the host."""
    out = SegmentInputs(inp.family, inp.dtype, inp.H_k, inp.H_v, inp.d_k, inp.d_v,
                        inp.seg_offsets, inp.k.cpu(), inp.v.cpu(), meta=dict(inp.meta))
    for n in ("log_gate", "log_gamma", "beta"):
        t = getattr(inp, n)
        setattr(out, n, None if t is None else t.cpu())
    return out
