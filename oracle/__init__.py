"""fp64 CPU oracle for HYPIC's linear-layer state path (test infrastructure only).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
import this package. The product path (the CUDA library and its Python binding) never
does, and the two share no code: this package compiles and calls ``hypic_oracle.c``,
a token-by-token fp64 program written from the definitions on the pages (see the header
of that file for the passages it follows).

Every array goes in and out as C-contiguous float64 numpy arrays; the caller converts
bf16 / fp32 inputs to float64 exactly (every bf16 and fp32 value is a float64 value).

Parity pins: every function here is pinned in ``tests/test_oracle.py`` against closed
forms, invariants and brute force; no function is left "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hypic_oracle.c")
_LIB = os.path.join(_HERE, "libhypic_oracle.so")
_lock = threading.Lock()
_lib = None

FAMILIES = {"linear": 0, "scalar": 1, "diag": 2, "delta": 3, "gdn": 4, "kda": 5}


def build(force: bool = False) -> str:
    """Compile hypic_oracle.c into libhypic_oracle.so beside it (plain gcc, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
               "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            I = ctypes.c_int
            I64 = ctypes.c_int64
            lib.oracle_build.argtypes = [I, I, P, I, I, I, I, P, P, P, P, P, P, P, I]
            lib.oracle_run.argtypes = [I, I, P, I, I, I, I, P, P, P, P, P, P, P, I]
            lib.oracle_compose_scan.argtypes = [I, I64, I, I, P, P, P, P, I]
            lib.oracle_materialize_T.argtypes = [I, I64, I, P, P, P]
            lib.oracle_compose_transitions.argtypes = [I, I, I64, I, P, P, P, P, I]
            lib.oracle_outputs.argtypes = [I, I, P, I, I, I, I, P, P, P, P, P, P, P, P, I]
            for f in (lib.oracle_build, lib.oracle_run, lib.oracle_compose_scan,
                      lib.oracle_materialize_T, lib.oracle_compose_transitions, lib.oracle_outputs):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(a):
    if a is None:
        return None
    a = np.ascontiguousarray(a, dtype=np.float64)
    return a


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _family(family):
    return FAMILIES[family] if isinstance(family, str) else int(family)


def build_segments(family, seg_offsets, k, v, log_gate=None, log_gamma=None, beta=None,
                   H_k=None, H_v=None, want_T=True, nthreads=0):
    """(S(C|0), T_C) per segment and value head, fp64.

    k [N, H_k, d_k], v [N, H_v, d_v]; returns S [n_seg, H_v, d_k, d_v] and
    T [n_seg, H_v, d_k, d_k] (None when want_T is False).
    """
    lib = _load()
    offs = np.ascontiguousarray(seg_offsets, dtype=np.int64)
    k, v = _f64(k), _f64(v)
    log_gate, log_gamma, beta = _f64(log_gate), _f64(log_gamma), _f64(beta)
    N, Hk, dk = k.shape
    _, Hv, dv = v.shape
    n_seg = len(offs) - 1
    assert offs[0] == 0 and offs[-1] == N
    S = np.zeros((n_seg, Hv, dk, dv))
    T = np.zeros((n_seg, Hv, dk, dk)) if want_T else None
    rc = lib.oracle_build(_family(family), n_seg, _ptr(offs), Hk, Hv, dk, dv, _ptr(k), _ptr(v),
                          _ptr(log_gate), _ptr(log_gamma), _ptr(beta), _ptr(S), _ptr(T),
                          nthreads or default_threads())
    if rc != 0:
        raise RuntimeError(f"oracle_build failed ({rc})")
    return S, T


def run_sequential(family, seg_offsets, k, v, log_gate=None, log_gamma=None, beta=None,
                   S0=None, nthreads=0):
    """State after every segment of one sequential pass, fp64: [n_seg, H_v, d_k, d_v]."""
    lib = _load()
    offs = np.ascontiguousarray(seg_offsets, dtype=np.int64)
    k, v = _f64(k), _f64(v)
    log_gate, log_gamma, beta, S0 = _f64(log_gate), _f64(log_gamma), _f64(beta), _f64(S0)
    N, Hk, dk = k.shape
    _, Hv, dv = v.shape
    n_seg = len(offs) - 1
    out = np.zeros((n_seg, Hv, dk, dv))
    rc = lib.oracle_run(_family(family), n_seg, _ptr(offs), Hk, Hv, dk, dv, _ptr(k), _ptr(v),
                        _ptr(log_gate), _ptr(log_gamma), _ptr(beta), _ptr(S0), _ptr(out),
                        nthreads or default_threads())
    if rc != 0:
        raise RuntimeError(f"oracle_run failed ({rc})")
    return out


def outputs(family, seg_offsets, k, v, q, log_gate=None, log_gamma=None, beta=None, S_init=None,
            nthreads=0):
    """o_t = S_t^T q_t for every token, fp64: [N_tok, H_v, d_v]. Each segment starts from
    S_init[seg, h] ([n_seg, H_v, d_k, d_v]; None = zero state, the outputs O(C|0))."""
    lib = _load()
    offs = np.ascontiguousarray(seg_offsets, dtype=np.int64)
    k, v, q = _f64(k), _f64(v), _f64(q)
    log_gate, log_gamma, beta, S_init = _f64(log_gate), _f64(log_gamma), _f64(beta), _f64(S_init)
    N, Hk, dk = k.shape
    _, Hv, dv = v.shape
    assert q.shape == k.shape
    n_seg = len(offs) - 1
    out = np.zeros((N, Hv, dv))
    rc = lib.oracle_outputs(_family(family), n_seg, _ptr(offs), Hk, Hv, dk, dv, _ptr(k), _ptr(v),
                            _ptr(q), _ptr(log_gate), _ptr(log_gamma), _ptr(beta), _ptr(S_init),
                            _ptr(out), nthreads or default_threads())
    if rc != 0:
        raise RuntimeError(f"oracle_outputs failed ({rc})")
    return out


def compose_scan(T, S, S0=None, nthreads=0):
    """prefix_j = T_j prefix_{j-1} + S_j; T [n_seg, U, d_k, d_k], S [n_seg, U, d_k, d_v]."""
    lib = _load()
    T, S, S0 = _f64(T), _f64(S), _f64(S0)
    n_seg, U, dk, dv = S.shape
    assert T.shape == (n_seg, U, dk, dk)
    out = np.zeros_like(S)
    rc = lib.oracle_compose_scan(n_seg, U, dk, dv, _ptr(T), _ptr(S), _ptr(S0), _ptr(out),
                                 nthreads or default_threads())
    if rc != 0:
        raise RuntimeError(f"oracle_compose_scan failed ({rc})")
    return out


def compose_transitions(family, lam, P=None, d_k=None):
    """Transition of the entry composed from n_seg consecutive segments, log-scaled:
    lam_total = sum_j lam_j and (delta / gdn) P_total = P_{n-1} ... P_0, fp64.

    lam [n_seg, U] (diag [n_seg, U, d_k]; ignored for linear, pass d_k and a [n_seg, U]
    array of zeros or any values), P [n_seg, U, d_k, d_k] for delta / gdn. Returns
    (lam_total [U] or [U, d_k], P_total [U, d_k, d_k] or None).
    """
    lib = _load()
    fam = _family(family)
    lam = _f64(lam)
    dense = fam in (FAMILIES["delta"], FAMILIES["gdn"], FAMILIES["kda"])
    if fam == FAMILIES["diag"]:
        n_seg, U, d_k = lam.shape
    else:
        n_seg, U = lam.shape[:2]
    if dense:
        P = _f64(P)
        d_k = P.shape[-1]
        assert P.shape == (n_seg, U, d_k, d_k)
    assert d_k is not None
    lam_total = np.zeros((U, d_k) if fam == FAMILIES["diag"] else (U,))
    P_total = np.zeros((U, d_k, d_k)) if dense else None
    rc = lib.oracle_compose_transitions(fam, n_seg, U, d_k, _ptr(lam), _ptr(P), _ptr(lam_total),
                                        _ptr(P_total), default_threads())
    if rc != 0:
        raise RuntimeError(f"oracle_compose_transitions failed ({rc})")
    return lam_total, P_total


def materialize_T(family, lam, P=None, d_k=None):
    """Dense fp64 T from the library's log-scaled storage T = exp(lam) P.

    lam has shape [..., ] (scalar families, GDN, DeltaNet) or [..., d_k] (DIAG);
    P [..., d_k, d_k] for DELTA / GDN. Returns [..., d_k, d_k].
    """
    lib = _load()
    fam = _family(family)
    lam = _f64(lam)
    if fam == FAMILIES["diag"]:
        d_k = lam.shape[-1]
        lead = lam.shape[:-1]
    elif fam in (FAMILIES["delta"], FAMILIES["gdn"], FAMILIES["kda"]):
        P = _f64(P)
        d_k = P.shape[-1]
        lead = P.shape[:-2]
    else:
        assert d_k is not None
        lead = lam.shape
    n = int(np.prod(lead)) if len(lead) else 1
    out = np.zeros(lead + (d_k, d_k))
    rc = lib.oracle_materialize_T(fam, n, d_k, _ptr(lam), _ptr(P), _ptr(out))
    if rc != 0:
        raise RuntimeError(f"oracle_materialize_T failed ({rc})")
    return out


# ------------------------------------------------------------------ convolution-state warm-up
# "Cut First-Token Latency by 3.25x: Introducing HYPIC ..." (besthub.dev), paragraph "For linear
# layers": for convolutional variants HYPIC adds a "convolution state warm-up" patch to keep
# cached segments aligned. The pages do not define the convolution; the reading here is the
# short convolution of the Gated DeltaNet layer ("Gated Delta Networks: Improving Mamba2 with
# Delta Rule", reference 7 of the episode-companion page): a causal depthwise convolution of
# width K over the token axis, then SiLU, on k and v, with k L2-normalised per token and head
# afterwards for the delta-rule families. A segment's tokens from K-1 on have their whole
# window inside the segment, so their entry (the "rest") is position-independent and cached; the
# first K-1 tokens (the "head") see the preceding segment's last raw tokens and are rebuilt in
# context, then composed before the rest: T = T_rest T_head, S = T_rest S_head + S_rest.

DELTA_FAMILIES = ("delta", "gdn", "kda")


def silu(x):
    """x * sigmoid(x), fp64."""
    x = np.asarray(x, dtype=np.float64)
    return x / (1.0 + np.exp(-x))


def short_conv(x, w, start=0, stop=None, normalize=False):
    """The convolved (then SiLU, then optionally L2-normalised) value of tokens [start, stop) of
    a token stream x [N, H, D]: y[t, h, c] = silu(sum_{tau < K} w[h D + c, tau] x[t - K + 1 + tau,
    h, c]), with x taken as 0 before token 0. w [H D, K] fp64 (tap K-1 on the token itself).
    Returns [stop - start, H, D]. Plain loops over taps and tokens."""
    x = _f64(x)
    w = _f64(w)
    N, H, D = x.shape
    K = w.shape[1]
    stop = N if stop is None else stop
    out = np.zeros((stop - start, H, D))
    wk = w.reshape(H, D, K)
    for t in range(start, stop):
        acc = np.zeros((H, D))
        for tau in range(K):
            s = t - (K - 1) + tau
            if s >= 0:
                acc += wk[:, :, tau] * x[s]
        y = silu(acc)
        if normalize:
            n = np.sqrt((y * y).sum(axis=1, keepdims=True))
            y = np.where(n > 0, y / np.where(n > 0, n, 1.0), 0.0)
        out[t - start] = y
    return out


def head_lengths(seg_offsets, K):
    """Tokens of each segment rebuilt in context: min(K - 1, length)."""
    offs = np.asarray(seg_offsets, dtype=np.int64)
    return np.minimum(K - 1, offs[1:] - offs[:-1])


def conv_warmup(family, seg_offsets, k_raw, v_raw, wk, wv, K, S_rest, lam_rest, P_rest=None,
                log_gate=None, log_gamma=None, beta=None):
    """Entries of the prompt's segments in context, from the cached entries of their rests,
    fp64. k_raw [N, H_k, d], v_raw [N, H_v, d]: the prompt's raw (pre-convolution) inputs in
    order; wk [H_k d, K], wv [H_v d, K]; log_gate / log_gamma / beta as for build_segments, over
    the prompt's tokens; S_rest [n_seg, H_v, d, d], lam_rest, P_rest: the entries of each
    segment's tokens from its head length on. Returns (S [n_seg, H_v, d, d], T [n_seg, H_v, d, d])
    with T dense."""
    fam = family
    offs = np.asarray(seg_offsets, dtype=np.int64)
    n_seg = len(offs) - 1
    hl = head_lengths(offs, K)
    # 1. the heads' tokens, convolved over the prompt's stream (their windows reach back into
    #    the preceding segment), and their gates
    rows = [int(offs[j]) + i for j in range(n_seg) for i in range(int(hl[j]))]
    Hk, Hv, d = k_raw.shape[1], v_raw.shape[1], v_raw.shape[2]
    kh = np.zeros((len(rows), Hk, d))
    vh = np.zeros((len(rows), Hv, d))
    for r, t in enumerate(rows):
        kh[r] = short_conv(k_raw, wk, t, t + 1, normalize=fam in DELTA_FAMILIES)[0]
        vh[r] = short_conv(v_raw, wv, t, t + 1)[0]
    pick = lambda a: None if a is None else _f64(a)[rows]
    head_offs = np.concatenate([[0], np.cumsum(hl)]).astype(np.int64)
    # 2. the heads' entries (from a zero state)
    S_h, T_h = build_segments(fam, head_offs, kh, vh, pick(log_gate), log_gamma, pick(beta))
    # 3. composed before the rests
    T_r = materialize_T(fam, lam_rest, P_rest, d_k=d)
    S = np.einsum("suij,sujk->suik", T_r, S_h) + _f64(S_rest)
    T = np.einsum("suij,sujk->suik", T_r, T_h)
    return S, T
