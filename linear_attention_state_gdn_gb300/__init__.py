"""Python binding of libhypic (include/hypic.h): argument marshalling only.

Every step of the segment build and the compose scan runs in the CUDA library; this
module turns torch CUDA tensors into the C structs of the ABI, calls the entry points of
the same names, and raises on a non-OK status. There is no CPU path: if the library is
not built, or no GPU is present, the calls raise.

    S, lam, P = hypic_build_segments("gdn", k, v, seg_offsets, log_gate=log_a, beta=beta)
    prefix = hypic_compose_scan("gdn", S, lam, P)
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import numpy as np
import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
# HYPIC_LIBRARY selects another build of the library (the debug-bounds build libhypic_dbg.so)
LIB_PATH = os.environ.get("HYPIC_LIBRARY") or os.path.join(_PKG, "libhypic.so")

FAMILY = {"linear": 0, "scalar": 1, "diag": 2, "delta": 3, "gdn": 4, "kda": 5}
DENSE = ("delta", "gdn", "kda")
DTYPE = {torch.bfloat16: 0, torch.float32: 1}
STATUS = {0: "HYPIC_OK", 1: "HYPIC_ERR_INVALID_ARG", 2: "HYPIC_ERR_ALIGNMENT",
          3: "HYPIC_ERR_UNSUPPORTED", 4: "HYPIC_ERR_RANGE", 5: "HYPIC_ERR_CUDA",
          6: "HYPIC_ERR_TIMEOUT"}
MAX_SEGMENTS = 1024


class HypicError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)}")


class BuildArgs(ctypes.Structure):
    _fields_ = [("family", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("n_seg", ctypes.c_int32), ("H_k", ctypes.c_int32), ("H_v", ctypes.c_int32),
                ("d_k", ctypes.c_int32), ("d_v", ctypes.c_int32), ("reserved0", ctypes.c_int32),
                ("out_seg_stride", ctypes.c_int64), ("seg_offsets", ctypes.c_void_p),
                ("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("log_gate", ctypes.c_void_p),
                ("log_gamma", ctypes.c_void_p), ("beta", ctypes.c_void_p),
                ("S", ctypes.c_void_p), ("lam", ctypes.c_void_p), ("P", ctypes.c_void_p),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
                ("q", ctypes.c_void_p), ("O", ctypes.c_void_p), ("S_init", ctypes.c_void_p)]


class ComposeArgs(ctypes.Structure):
    _fields_ = [("family", ctypes.c_int32), ("n_seg", ctypes.c_int32),
                ("n_units", ctypes.c_int64), ("d_k", ctypes.c_int32), ("d_v", ctypes.c_int32),
                ("S", ctypes.c_void_p), ("lam", ctypes.c_void_p), ("P", ctypes.c_void_p),
                ("S0", ctypes.c_void_p), ("prefix", ctypes.c_void_p),
                ("lam_total", ctypes.c_void_p), ("P_total", ctypes.c_void_p)]


class WarmupArgs(ctypes.Structure):
    _fields_ = [("family", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("n_seg", ctypes.c_int32), ("H_k", ctypes.c_int32), ("H_v", ctypes.c_int32),
                ("d_k", ctypes.c_int32), ("d_v", ctypes.c_int32), ("conv_k", ctypes.c_int32),
                ("seg_offsets", ctypes.c_void_p), ("k_raw", ctypes.c_void_p), ("v_raw", ctypes.c_void_p),
                ("conv_wk", ctypes.c_void_p), ("conv_wv", ctypes.c_void_p), ("log_gate", ctypes.c_void_p),
                ("log_gamma", ctypes.c_void_p), ("beta", ctypes.c_void_p), ("S_rest", ctypes.c_void_p),
                ("lam_rest", ctypes.c_void_p), ("P_rest", ctypes.c_void_p), ("S", ctypes.c_void_p),
                ("lam", ctypes.c_void_p), ("P", ctypes.c_void_p), ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_size_t)]


_lib = None
_lock = threading.Lock()


def load_library(path: str = LIB_PATH):
    """Load libhypic.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(
                    f"libhypic.so not found at {path}: build it with "
                    "`python -c 'import __graft_entry__ as g; g.build()'` (needs nvcc)")
            lib = ctypes.CDLL(path)
            lib.hypic_build_segments.argtypes = [ctypes.POINTER(BuildArgs), ctypes.c_void_p]
            lib.hypic_build_segments.restype = ctypes.c_int
            lib.hypic_build_segments_static_ws.argtypes = [ctypes.POINTER(BuildArgs), ctypes.c_void_p]
            lib.hypic_build_segments_static_ws.restype = ctypes.c_int
            lib.hypic_compose_scan.argtypes = [ctypes.POINTER(ComposeArgs), ctypes.c_void_p]
            lib.hypic_compose_scan.restype = ctypes.c_int
            lib.hypic_build_workspace_bytes.argtypes = [ctypes.POINTER(BuildArgs)]
            lib.hypic_build_workspace_bytes.restype = ctypes.c_size_t
            lib.hypic_get_device_status.argtypes = [ctypes.c_void_p]
            lib.hypic_get_device_status.restype = ctypes.c_int
            lib.hypic_status_string.argtypes = [ctypes.c_int]
            lib.hypic_status_string.restype = ctypes.c_char_p
            for f, t in ((lib.hypic_build_kernel_name, BuildArgs),
                         (lib.hypic_compose_kernel_name, ComposeArgs)):
                f.argtypes = [ctypes.POINTER(t)]
                f.restype = ctypes.c_char_p
            lib.hypic_probe_wait_timeout.argtypes = [ctypes.c_uint32, ctypes.c_void_p]
            lib.hypic_probe_wait_timeout.restype = ctypes.c_int
            lib.hypic_warmup_workspace_bytes.argtypes = [ctypes.POINTER(WarmupArgs)]
            lib.hypic_warmup_workspace_bytes.restype = ctypes.c_size_t
            lib.hypic_conv_warmup.argtypes = [ctypes.POINTER(WarmupArgs), ctypes.c_void_p]
            lib.hypic_conv_warmup.restype = ctypes.c_int
            lib.hypic_abi_version.argtypes = []
            lib.hypic_abi_version.restype = ctypes.c_int32
            _lib = lib
    return _lib


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors passed to libhypic must be CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("tensors passed to libhypic must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(status: int, what: str):
    if status != 0:
        raise HypicError(status, what)


def _offsets(seg_offsets) -> np.ndarray:
    if isinstance(seg_offsets, torch.Tensor):
        seg_offsets = seg_offsets.cpu().numpy()
    return np.ascontiguousarray(seg_offsets, dtype=np.int64)


def make_build_args(family, k, v, seg_offsets, log_gate=None, log_gamma=None, beta=None,
                    S=None, lam=None, P=None, out_seg_stride=0, workspace=None, q=None, O=None,
                    S_init=None):
    """Fill a BuildArgs struct (and keep the host offsets array alive with it)."""
    offs = _offsets(seg_offsets)
    fam = FAMILY[family] if isinstance(family, str) else int(family)
    a = BuildArgs()
    a.family = fam
    a.dtype = DTYPE[k.dtype]
    a.n_seg = len(offs) - 1
    a.H_k, a.d_k = k.shape[1], k.shape[2]
    a.H_v, a.d_v = v.shape[1], v.shape[2]
    a.out_seg_stride = out_seg_stride
    a.seg_offsets = offs.ctypes.data
    a.k, a.v = _ptr(k), _ptr(v)
    a.log_gate, a.log_gamma, a.beta = _ptr(log_gate), _ptr(log_gamma), _ptr(beta)
    a.S, a.lam, a.P = _ptr(S), _ptr(lam), _ptr(P)
    a.q, a.O, a.S_init = _ptr(q), _ptr(O), _ptr(S_init)
    if workspace is not None:
        a.workspace, a.workspace_bytes = _ptr(workspace), workspace.numel() * workspace.element_size()
    a._keep = offs
    return a


def build_outputs(family, n_seg, H_v, d, device, out_seg_stride=0):
    units = out_seg_stride or H_v
    S = torch.empty((n_seg, units, d, d), dtype=torch.float32, device=device)
    lam = torch.empty((n_seg, units, d) if family == "diag" else (n_seg, units),
                      dtype=torch.float32, device=device)
    P = (torch.empty((n_seg, units, d, d), dtype=torch.float32, device=device)
         if family in DENSE else None)
    return S, lam, P


def _outputs(family, n_seg, v, S, lam, P, out_seg_stride):
    """The build's output tensors: allocated (with the segment stride the call writes at)
    when S is not given; checked to hold every unit the call writes when they are. Segment j
    of the call writes units j * stride .. j * stride + H_v - 1 of S, lam and P."""
    H_v, d = v.shape[1], v.shape[2]
    if S is None:
        if lam is not None or P is not None:
            raise ValueError("give S, lam (and P) together, or none of them")
        return build_outputs(family, n_seg, H_v, d, v.device, out_seg_stride)
    stride = out_seg_stride or H_v
    units = (n_seg - 1) * stride + H_v if n_seg > 0 else 0
    dense = family in DENSE or family in tuple(FAMILY[f] for f in DENSE)
    diag = family in ("diag", FAMILY["diag"])
    need = [(S, units * d * d, "S"), (lam, units * (d if diag else 1), "lam")]
    if dense:
        need.append((P, units * d * d, "P"))
    for t, n, name in need:
        if t is None:
            raise ValueError(f"{name} missing")
        if not t.is_contiguous() or t.dtype != torch.float32 or t.numel() < n:
            raise ValueError(f"{name} must be a contiguous fp32 tensor of at least {n} elements")
    return S, lam, P


def hypic_build_workspace_bytes(family, k, v, seg_offsets, **kw) -> int:
    lib = load_library()
    a = make_build_args(family, k, v, seg_offsets, **kw)
    return int(lib.hypic_build_workspace_bytes(ctypes.byref(a)))


def hypic_build_segments(family, k, v, seg_offsets, log_gate=None, log_gamma=None, beta=None,
                         S=None, lam=None, P=None, out_seg_stride=0, workspace=None,
                         stream=None, q=None, O=None, S_init=None):
    """(S(C|0), lam, P) of every segment: S [n_seg, H_v, d, d], lam [n_seg, H_v]
    ([n_seg, H_v, d] for "diag"), P [n_seg, H_v, d, d] for "gdn"/"delta"/"kda" (else None).
    With queries q [N, H_k, d] also the segment outputs O [N, H_v, d] (dtype of v; allocated
    when not given), returned fourth: (S, lam, P, O). S_init [n_seg, H_v, d, d] starts each
    segment from that state instead of zero. Outputs are allocated when not given.
    Asynchronous on `stream`."""
    lib = load_library()
    n_seg = len(_offsets(seg_offsets)) - 1
    S, lam, P = _outputs(family, n_seg, v, S, lam, P, out_seg_stride)
    if q is not None and O is None:
        O = torch.empty(v.shape, dtype=v.dtype, device=v.device)
    a = make_build_args(family, k, v, seg_offsets, log_gate, log_gamma, beta, S, lam, P,
                        out_seg_stride, q=q, O=O, S_init=S_init)
    need = int(lib.hypic_build_workspace_bytes(ctypes.byref(a)))
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=v.device)
    if workspace is not None:
        a.workspace = _ptr(workspace)
        a.workspace_bytes = workspace.numel() * workspace.element_size()
    _check(lib.hypic_build_segments(ctypes.byref(a), _stream(stream)), "hypic_build_segments")
    return (S, lam, P) if q is None else (S, lam, P, O)


def hypic_build_segments_static_ws(family, k, v, seg_offsets, log_gate=None, log_gamma=None,
                                   beta=None, S=None, lam=None, P=None, out_seg_stride=0,
                                   stream=None):
    """hypic_build_segments with the library's own device scratch (HYPIC_STATIC_WS_BYTES,
    64 MiB): no per-call allocation. Calls that overlap in time race on that scratch."""
    lib = load_library()
    n_seg = len(_offsets(seg_offsets)) - 1
    S, lam, P = _outputs(family, n_seg, v, S, lam, P, out_seg_stride)
    a = make_build_args(family, k, v, seg_offsets, log_gate, log_gamma, beta, S, lam, P,
                        out_seg_stride)
    _check(lib.hypic_build_segments_static_ws(ctypes.byref(a), _stream(stream)),
           "hypic_build_segments_static_ws")
    return S, lam, P


STATIC_WS_BYTES = 64 << 20   # HYPIC_STATIC_WS_BYTES in include/hypic.h


def make_warmup_args(family, seg_offsets, k_raw, v_raw, conv_wk, conv_wv, S_rest, lam_rest,
                     P_rest=None, log_gate=None, log_gamma=None, beta=None, S=None, lam=None,
                     P=None, workspace=None):
    """Fill a WarmupArgs struct (and keep the host offsets array alive with it)."""
    offs = _offsets(seg_offsets)
    a = WarmupArgs()
    a.family = FAMILY[family] if isinstance(family, str) else int(family)
    a.dtype = DTYPE[k_raw.dtype]
    a.n_seg = len(offs) - 1
    a.H_k, a.d_k = k_raw.shape[1], k_raw.shape[2]
    a.H_v, a.d_v = v_raw.shape[1], v_raw.shape[2]
    a.conv_k = conv_wk.shape[1]
    a.seg_offsets = offs.ctypes.data
    a.k_raw, a.v_raw = _ptr(k_raw), _ptr(v_raw)
    a.conv_wk, a.conv_wv = _ptr(conv_wk), _ptr(conv_wv)
    a.log_gate, a.log_gamma, a.beta = _ptr(log_gate), _ptr(log_gamma), _ptr(beta)
    a.S_rest, a.lam_rest, a.P_rest = _ptr(S_rest), _ptr(lam_rest), _ptr(P_rest)
    a.S, a.lam, a.P = _ptr(S), _ptr(lam), _ptr(P)
    if workspace is not None:
        a.workspace, a.workspace_bytes = _ptr(workspace), workspace.numel() * workspace.element_size()
    a._keep = offs
    return a


def hypic_warmup_workspace_bytes(family, seg_offsets, k_raw, v_raw, conv_wk, conv_wv, S_rest,
                                 lam_rest, **kw) -> int:
    lib = load_library()
    a = make_warmup_args(family, seg_offsets, k_raw, v_raw, conv_wk, conv_wv, S_rest, lam_rest, **kw)
    return int(lib.hypic_warmup_workspace_bytes(ctypes.byref(a)))


def hypic_conv_warmup(family, seg_offsets, k_raw, v_raw, conv_wk, conv_wv, S_rest, lam_rest,
                      P_rest=None, log_gate=None, log_gamma=None, beta=None, S=None, lam=None,
                      P=None, workspace=None, stream=None):
    """Entries (S, lam, P) of this prompt's segments in context, from the cached entries of
    their rests (each segment's tokens from min(K - 1, length) on) and the raw, pre-convolution
    k_raw [N, H_k, d], v_raw [N, H_v, d] of the whole prompt; conv_wk [H_k d, K] and
    conv_wv [H_v d, K] fp32 are the short convolution's taps. Outputs are allocated when not
    given (shapes of S_rest, lam_rest, P_rest). Asynchronous on `stream`."""
    lib = load_library()
    if S is None:
        S, lam = torch.empty_like(S_rest), torch.empty_like(lam_rest)
        P = None if P_rest is None else torch.empty_like(P_rest)
    a = make_warmup_args(family, seg_offsets, k_raw, v_raw, conv_wk, conv_wv, S_rest, lam_rest,
                         P_rest, log_gate, log_gamma, beta, S, lam, P)
    need = int(lib.hypic_warmup_workspace_bytes(ctypes.byref(a)))
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=S_rest.device)
    if workspace is not None:
        a.workspace = _ptr(workspace)
        a.workspace_bytes = workspace.numel() * workspace.element_size()
    _check(lib.hypic_conv_warmup(ctypes.byref(a), _stream(stream)), "hypic_conv_warmup")
    return S, lam, P


def make_compose_args(family, S, lam, P=None, S0=None, prefix=None, lam_total=None, P_total=None):
    fam = FAMILY[family] if isinstance(family, str) else int(family)
    a = ComposeArgs()
    a.family = fam
    a.n_seg, a.n_units, a.d_k, a.d_v = S.shape[0], S.shape[1], S.shape[2], S.shape[3]
    a.S, a.lam, a.P, a.S0, a.prefix = _ptr(S), _ptr(lam), _ptr(P), _ptr(S0), _ptr(prefix)
    a.lam_total, a.P_total = _ptr(lam_total), _ptr(P_total)
    return a


def hypic_compose_scan(family, S, lam, P=None, S0=None, prefix=None, lam_total=None,
                       P_total=None, stream=None):
    """Inclusive prefix scan prefix[j] = exp(lam_j) P_j prefix[j-1] + S_j over segments.
    S [n_seg, U, d, d]; returns prefix of the same shape (allocated when not given).
    Optional outputs: lam_total [U] ([U, d] for "diag") = sum_j lam_j and, for "gdn" /
    "delta", P_total [U, d, d] = P_{n-1} ... P_0 (the transition of all segments composed)."""
    lib = load_library()
    if prefix is None:
        prefix = torch.empty_like(S)
    a = make_compose_args(family, S, lam, P, S0, prefix, lam_total, P_total)
    _check(lib.hypic_compose_scan(ctypes.byref(a), _stream(stream)), "hypic_compose_scan")
    return prefix



def hypic_build_kernel_name(family, k, v, seg_offsets, **kw) -> str:
    """Name of the kernel a build with these arguments launches (host-only query)."""
    a = make_build_args(family, k, v, seg_offsets, **kw)
    r = load_library().hypic_build_kernel_name(ctypes.byref(a))
    return None if r is None else r.decode()


def hypic_compose_kernel_name(family, S, lam=None, P=None, S0=None) -> str:
    """Name of the kernel a compose scan of these arguments launches (host-only query)."""
    a = ComposeArgs()
    a.family = FAMILY[family] if isinstance(family, str) else int(family)
    a.n_seg, a.n_units, a.d_k, a.d_v = S.shape[0], S.shape[1], S.shape[2], S.shape[3]
    r = load_library().hypic_compose_kernel_name(ctypes.byref(a))
    return None if r is None else r.decode()


def hypic_get_device_status(stream=None) -> int:
    """Synchronise and read + clear the device status word (0 = HYPIC_OK)."""
    return int(load_library().hypic_get_device_status(_stream(stream)))


def hypic_probe_wait_timeout(limit_us: int, stream=None) -> None:
    """Run the library's bounded-wait failure path on every SM (a wait that nothing ends runs
    out after limit_us microseconds); hypic_get_device_status() then reports
    HYPIC_ERR_TIMEOUT. Diagnostic only: no real kernel is made to hang."""
    _check(load_library().hypic_probe_wait_timeout(int(limit_us), _stream(stream)),
           "hypic_probe_wait_timeout")


def hypic_status_string(status: int) -> str:
    return load_library().hypic_status_string(status).decode()


__all__ = ["hypic_build_segments", "hypic_build_segments_static_ws", "hypic_compose_scan",
           "hypic_build_workspace_bytes",
           "hypic_build_kernel_name", "hypic_compose_kernel_name",
           "hypic_get_device_status", "hypic_probe_wait_timeout", "hypic_status_string",
           "load_library", "HypicError",
           "build_outputs", "FAMILY"]
