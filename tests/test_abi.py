"""The C-ABI library loads, exports every symbol include/hypic.h declares, and rejects bad
arguments on the host before any launch. No test here needs a GPU: the argument checks
run before the library touches the device, and the fake pointers are never dereferenced.
"""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "hypic.h")


@pytest.fixture(scope="module")
def lib():
    from linear_attention_state_gdn_gb300 import _build, load_library
    _build.build()
    return load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(hypic_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("hypic_build_segments", "hypic_compose_scan", "hypic_build_workspace_bytes",
              "hypic_get_device_status", "hypic_status_string", "hypic_abi_version"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in hypic.h but not exported"


def test_status_strings_and_version(lib):
    assert lib.hypic_abi_version() == 5
    assert lib.hypic_status_string(0) == b"ok"
    assert lib.hypic_status_string(2) == b"misaligned tensor pointer"
    assert lib.hypic_status_string(99) == b"unknown status"


def test_python_names_match_the_abi():
    import linear_attention_state_gdn_gb300 as m
    for name in declared_functions():
        if name != "hypic_abi_version":
            assert hasattr(m, name)


# ------------------------------------------------------------------ host-side validation

from linear_attention_state_gdn_gb300 import BuildArgs, ComposeArgs, WarmupArgs  # noqa: E402

FAKE = 0x7f0000000000   # 16-byte aligned, never dereferenced


def good_build(family=4, n_seg=2, lens=(64, 64)):
    offs = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    a = BuildArgs()
    a.family, a.dtype, a.n_seg = family, 0, n_seg
    a.H_k, a.H_v, a.d_k, a.d_v = 2, 4, 128, 128
    a.seg_offsets = offs.ctypes.data
    a.k, a.v, a.S, a.lam, a.P = FAKE, FAKE + 0x1000000, FAKE + 0x2000000, FAKE + 0x3000000, \
        FAKE + 0x4000000
    a.log_gate, a.beta = FAKE + 0x5000000, FAKE + 0x6000000
    a._keep = offs
    return a


def call_build(lib, a):
    return lib.hypic_build_segments(ctypes.byref(a), None)


def test_build_rejects_null_args(lib):
    assert lib.hypic_build_segments(None, None) == 1


@pytest.mark.parametrize("field,value,status", [
    ("family", 7, 1), ("family", -1, 1), ("dtype", 5, 1), ("n_seg", -1, 1),
    ("n_seg", 1025, 1), ("H_k", 0, 1), ("H_k", 3, 1), ("d_k", 96, 3), ("d_v", 64, 3),
    ("d_k", 0, 1), ("out_seg_stride", 2, 1),
])
def test_build_rejects_bad_scalars(lib, field, value, status):
    a = good_build()
    setattr(a, field, value)
    assert call_build(lib, a) == status


def test_build_zero_segments_is_a_noop(lib):
    a = good_build()
    a.n_seg = 0
    assert call_build(lib, a) == 0


def test_build_rejects_bad_offsets(lib):
    a = good_build()
    bad = np.array([0, 70, 64], dtype=np.int64)         # decreasing
    a.seg_offsets = bad.ctypes.data
    assert call_build(lib, a) == 1
    bad2 = np.array([5, 70, 140], dtype=np.int64)       # not starting at 0
    a.seg_offsets = bad2.ctypes.data
    assert call_build(lib, a) == 1
    a.seg_offsets = None
    assert call_build(lib, a) == 1


@pytest.mark.parametrize("field", ["S", "lam", "P", "beta", "log_gate", "k", "v"])
def test_build_rejects_missing_tensors(lib, field):
    a = good_build()
    setattr(a, field, None)
    assert call_build(lib, a) == 1


def test_build_scalar_needs_exactly_one_gate_form(lib):
    a = good_build(family=1)
    a.P = None
    a.beta = None
    a.log_gamma = FAKE + 0x7000000          # both log_gate and log_gamma
    assert call_build(lib, a) == 1
    a.log_gate = None
    a.log_gamma = None                      # neither
    assert call_build(lib, a) == 1


@pytest.mark.parametrize("field", ["k", "v", "S", "P"])
def test_build_rejects_misaligned_tensors(lib, field):
    a = good_build()
    setattr(a, field, getattr(a, field) + 8)
    assert call_build(lib, a) == 2


def test_build_rejects_host_pointers(lib):
    """Fake or host addresses are refused (no GPU here: nothing is device memory)."""
    a = good_build()
    assert call_build(lib, a) == 1


def good_compose(family=4):
    a = ComposeArgs()
    a.family, a.n_seg, a.n_units, a.d_k, a.d_v = family, 3, 5, 128, 128
    a.S, a.lam, a.P, a.prefix = FAKE, FAKE + 0x1000000, FAKE + 0x2000000, FAKE + 0x3000000
    return a


@pytest.mark.parametrize("field,value,status", [
    ("family", 9, 1), ("n_seg", -2, 1), ("n_units", -1, 1), ("d_k", 48, 3), ("d_v", 32, 3)])
def test_compose_rejects_bad_scalars(lib, field, value, status):
    a = good_compose()
    setattr(a, field, value)
    assert lib.hypic_compose_scan(ctypes.byref(a), None) == status


@pytest.mark.parametrize("field", ["S", "lam", "P", "prefix"])
def test_compose_rejects_missing_tensors(lib, field):
    a = good_compose()
    setattr(a, field, None)
    assert lib.hypic_compose_scan(ctypes.byref(a), None) == 1


def test_compose_linear_needs_no_lam_or_P(lib):
    a = good_compose(family=0)
    a.lam = None
    a.P = None
    # passes the argument checks, then fails the device-pointer check (no GPU here)
    assert lib.hypic_compose_scan(ctypes.byref(a), None) == 1


def test_compose_rejects_misaligned(lib):
    a = good_compose()
    a.prefix = a.prefix + 4
    assert lib.hypic_compose_scan(ctypes.byref(a), None) == 2


@pytest.mark.parametrize("field,offset", [("P_total", 4), ("lam_total", 2)])
def test_compose_rejects_misaligned_totals(lib, field, offset):
    a = good_compose()
    a.lam_total = FAKE + 0x5000000         # P_total needs lam_total
    setattr(a, field, FAKE + 0x4000000 + offset)
    assert lib.hypic_compose_scan(ctypes.byref(a), None) == 2


def test_compose_P_total_needs_lam_total(lib):
    a = good_compose()
    a.P_total = FAKE + 0x4000000
    assert lib.hypic_compose_scan(ctypes.byref(a), None) == 1


def test_compose_args_layout():
    # int32 family, n_seg; int64 n_units; int32 d_k, d_v; seven pointers
    assert ctypes.sizeof(ComposeArgs) == 80
    assert ComposeArgs.lam_total.offset == 64 and ComposeArgs.P_total.offset == 72


def test_compose_empty_is_a_noop(lib):
    a = good_compose()
    a.n_seg = 0
    assert lib.hypic_compose_scan(ctypes.byref(a), None) == 0
    a = good_compose()
    a.n_units = 0
    assert lib.hypic_compose_scan(ctypes.byref(a), None) == 0


def test_workspace_query_is_host_only(lib):
    a = good_build()
    assert lib.hypic_build_workspace_bytes(ctypes.byref(a)) >= 0
    assert lib.hypic_build_workspace_bytes(None) == 0


def test_binding_refuses_cpu_tensors():
    import torch
    from linear_attention_state_gdn_gb300 import hypic_build_segments, _build
    _build.build()
    k = torch.zeros(8, 1, 32, dtype=torch.bfloat16)
    v = torch.zeros(8, 1, 32, dtype=torch.bfloat16)
    S = torch.zeros(1, 1, 32, 32)
    lam = torch.zeros(1, 1)
    with pytest.raises(ValueError):
        hypic_build_segments("linear", k, v, [0, 8], S=S, lam=lam)


def test_workspace_bytes_of_the_tensor_core_gdn_build(lib):
    # bf16, d = 128, DeltaNet / GDN: 8 KB per (segment, value head, 64-token chunk) and a
    # 256-byte tail (the preparation kernel's ticket counter)
    a = good_build(lens=(64, 130))
    assert lib.hypic_build_workspace_bytes(ctypes.byref(a)) == 4 * (1 + 3) * 8192 + 256
    a.d_k = a.d_v = 64                      # exact fp32-state path: no workspace
    assert lib.hypic_build_workspace_bytes(ctypes.byref(a)) == 0
    b = good_build(family=2)                # gated families: no workspace
    assert lib.hypic_build_workspace_bytes(ctypes.byref(b)) == 0


def test_build_rejects_a_short_workspace(lib):
    a = good_build()
    a.workspace, a.workspace_bytes = FAKE + 0x7000000, 100
    assert call_build(lib, a) == 1


def test_static_workspace_build_rejects_null_and_oversized_requests(lib):
    assert lib.hypic_build_segments_static_ws(None, None) == 1
    # 4 heads x 2049 chunks x 8 KB > 64 MiB: refused before any device work
    a = good_build(n_seg=1, lens=(2049 * 64,))
    assert lib.hypic_build_workspace_bytes(ctypes.byref(a)) > (64 << 20)
    assert lib.hypic_build_segments_static_ws(ctypes.byref(a), None) == 3


def test_wait_probe_rejects_limits_out_of_range(lib):
    # checked before the library touches the device
    assert lib.hypic_probe_wait_timeout(0, None) == 1
    assert lib.hypic_probe_wait_timeout(1000001, None) == 1


def test_build_args_layout():
    # eight int32 and one int64; ten pointers; size_t; then (ABI 4) q, O, S_init
    assert ctypes.sizeof(BuildArgs) == 152
    assert BuildArgs.q.offset == 128 and BuildArgs.O.offset == 136 and BuildArgs.S_init.offset == 144


def test_build_outputs_and_queries_come_together(lib):
    a = good_build()
    a.q = FAKE + 0x8000000
    assert call_build(lib, a) == 1
    a = good_build()
    a.O = FAKE + 0x8000000
    assert call_build(lib, a) == 1


def test_kda_needs_gates_beta_and_P(lib):
    for field in ("log_gate", "beta", "P"):
        a = good_build(family=5)
        setattr(a, field, None)
        assert call_build(lib, a) == 1


def test_path_of_kda_outputs_and_start_states(lib):
    a = good_build(family=5)   # bf16, d = 128: the tensor-core build of the channel-gated rule
    assert lib.hypic_build_kernel_name(ctypes.byref(a)) == b"build_kda_tc"
    # 8 records: M2 (8 KB), the ticket tail, then per record Kt, Kb (16 KB each) and 132 floats
    assert lib.hypic_build_workspace_bytes(ctypes.byref(a)) == 8 * 8192 + 256 + 8 * (2 * 16384 + 132 * 4)
    a.q, a.O = FAKE + 0x8000000, FAKE + 0x9000000   # KDA outputs: the exact path
    assert lib.hypic_build_kernel_name(ctypes.byref(a)) == b"build_seq"
    assert lib.hypic_build_workspace_bytes(ctypes.byref(a)) == 0
    a = good_build(family=5)
    a.log_gate = FAKE + 0x5000004                    # gates not 8-byte aligned: the exact path
    assert lib.hypic_build_kernel_name(ctypes.byref(a)) == b"build_seq"
    assert lib.hypic_build_workspace_bytes(ctypes.byref(a)) == 0
    a = good_build(family=5)
    a.dtype = 1                                      # fp32 inputs: the exact path
    assert lib.hypic_build_kernel_name(ctypes.byref(a)) == b"build_seq"
    a = good_build(family=4)
    assert lib.hypic_build_kernel_name(ctypes.byref(a)) == b"build_gdn_tc"
    recs = lib.hypic_build_workspace_bytes(ctypes.byref(a))
    a.q, a.O = FAKE + 0x8000000, FAKE + 0x9000000   # GDN outputs: the tensor-core build
    assert lib.hypic_build_kernel_name(ctypes.byref(a)) == b"build_gdn_tc"
    assert lib.hypic_build_workspace_bytes(ctypes.byref(a)) == recs
    a.S_init = FAKE + 0xA000000                      # start states: the exact path
    assert lib.hypic_build_kernel_name(ctypes.byref(a)) == b"build_seq"
    assert lib.hypic_build_workspace_bytes(ctypes.byref(a)) == 0
    b = good_build(family=2)                         # outputs of the other families: exact path
    b.q, b.O = FAKE + 0x8000000, FAKE + 0x9000000
    assert lib.hypic_build_kernel_name(ctypes.byref(b)) == b"build_seq"


# ------------------------------------------------------------------ convolution-state warm-up

def good_warmup(family=4, lens=(64, 2, 0, 70), K=4):
    offs = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    a = WarmupArgs()
    a.family, a.dtype, a.n_seg, a.conv_k = family, 0, len(lens), K
    a.H_k, a.H_v, a.d_k, a.d_v = 2, 4, 128, 128
    a.seg_offsets = offs.ctypes.data
    a.k_raw, a.v_raw = FAKE, FAKE + 0x1000000
    a.conv_wk, a.conv_wv = FAKE + 0x2000000, FAKE + 0x2100000
    a.log_gate, a.beta = FAKE + 0x5000000, FAKE + 0x6000000
    a.S_rest, a.lam_rest, a.P_rest = FAKE + 0x7000000, FAKE + 0x8000000, FAKE + 0x9000000
    a.S, a.lam, a.P = FAKE + 0xA000000, FAKE + 0xB000000, FAKE + 0xC000000
    a._keep = offs
    return a


def test_warmup_struct_layout():
    assert ctypes.sizeof(WarmupArgs) == 8 * 4 + 16 * 8


@pytest.mark.parametrize("field,value", [("conv_k", 0), ("conv_k", 9), ("family", 6), ("dtype", 3),
                                         ("H_k", 3), ("S_rest", None), ("lam_rest", None),
                                         ("P_rest", None), ("beta", None), ("log_gate", None),
                                         ("conv_wk", None), ("S", None)])
def test_warmup_rejects_bad_arguments(lib, field, value):
    a = good_warmup()
    setattr(a, field, value)
    assert lib.hypic_conv_warmup(ctypes.byref(a), None) == 1


def test_warmup_empty_call_and_workspace(lib):
    a = good_warmup(lens=())
    assert lib.hypic_conv_warmup(ctypes.byref(a), None) == 0
    # heads of 3, 2, 0, 3 tokens (K = 4): convolved k (2 heads) and v (4 heads), gathered gates
    # and b, then the head entries S, lam and P of 4 x 4 units (256-byte rounding); the cached
    # rests are read where they are
    a = good_warmup()
    r, U, d = 8, 16, 128
    rnd = lambda x: (x + 255) // 256 * 256
    want = (rnd(r * 2 * d * 4) + rnd(r * 4 * d * 4) + rnd(r * 4 * 4) + rnd(r * 4 * 4) +
            rnd(U * d * d * 4) + rnd(U * 4) + rnd(U * d * d * 4))
    assert lib.hypic_warmup_workspace_bytes(ctypes.byref(a)) == want
    a = good_warmup(K=1)
    assert lib.hypic_warmup_workspace_bytes(ctypes.byref(a)) == rnd(U * d * d * 4) + rnd(U * 4) + \
        rnd(U * d * d * 4)
