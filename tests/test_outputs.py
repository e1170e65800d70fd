"""Segment outputs o_t = S_t^T q_t against the fp64 oracle (needs a GPU).

The outputs of a segment's prefill, read token by token from the state after each token,
from a zero state (O(C|0)) and from a given prefix state S_init (the outputs of a segment
reused after that prefix, whose end state is then S(C|S_init) = T_C S_init + S(C|0)). Every
(segment, head) block of O, [tokens x d_v], is compared with the relative Frobenius error:
<= 1e-4 for fp32 inputs, <= 2e-2 for bf16 inputs; a build that asks for outputs must leave
S, T unchanged within the same bounds.
"""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_state_gdn_gb300 import synth
from tests.helpers import TOL, assert_close, f64, gpu_T, oracle_build, to_dev

pytestmark = pytest.mark.gpu

FAMILIES = ["linear", "scalar", "diag", "delta", "gdn", "kda"]
RAGGED = [70, 1, 0, 33, 130]


def _hy():
    import linear_attention_state_gdn_gb300 as hy
    return hy


def out_errors(inp, O_gpu, O_ref):
    """Largest relative Frobenius error over the (segment, head) blocks of O."""
    worst = 0.0
    for j in range(inp.n_seg):
        a, b = int(inp.seg_offsets[j]), int(inp.seg_offsets[j + 1])
        if b == a:
            continue
        for h in range(inp.H_v):
            g, r = O_gpu[a:b, h], O_ref[a:b, h]
            worst = max(worst, np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-300))
    return worst


def oracle_outputs(inp, S_init=None):
    return oracle.outputs(inp.family, inp.seg_offsets, f64(inp.k), f64(inp.v), f64(inp.q),
                          f64(inp.log_gate), f64(inp.log_gamma), f64(inp.beta), S_init=S_init)


def gpu_build_out(inp, S_init=None):
    hy = _hy()
    d = to_dev(inp)
    S, lam, P, O = hy.hypic_build_segments(inp.family, d["k"], d["v"], inp.seg_offsets,
                                           log_gate=d.get("log_gate"), log_gamma=d.get("log_gamma"),
                                           beta=d.get("beta"), q=d["q"],
                                           S_init=None if S_init is None else S_init.cuda())
    torch.cuda.synchronize()
    assert hy.hypic_get_device_status() == 0
    return S, lam, P, O


@pytest.mark.parametrize("family", FAMILIES)
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("d", [32, 64, 128])
def test_outputs_from_zero_state(family, dtype, d):
    inp = synth.make_inputs(family, 2, 4, d, RAGGED, dtype, seed=90 + d, with_q=True, gla_div=8.0,
                            alpha_scale=0.05)
    S, lam, P, O = gpu_build_out(inp)
    tol = TOL[dtype]
    assert out_errors(inp, f64(O), oracle_outputs(inp)) <= tol
    So, To = oracle_build(inp)
    assert_close(f64(S), So, tol, "S")
    assert_close(gpu_T(family, lam, P, d), To, tol, "T")


@pytest.mark.parametrize("family", FAMILIES)
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_outputs_from_a_prefix_state(family, dtype):
    inp = synth.make_inputs(family, 2, 4, 64, RAGGED, dtype, seed=95, with_q=True, gla_div=8.0,
                            alpha_scale=0.05)
    S_init = torch.from_numpy(np.random.default_rng(96).standard_normal((inp.n_seg, 4, 64, 64))
                              .astype(np.float32))
    S, lam, P, O = gpu_build_out(inp, S_init)
    tol = TOL[dtype]
    assert out_errors(inp, f64(O), oracle_outputs(inp, f64(S_init))) <= tol
    So, To = oracle_build(inp)
    ref = So + np.einsum("shij,shjk->shik", To, f64(S_init))   # S(C|S0) = T_C S0 + S(C|0)
    assert_close(f64(S), ref, tol, "S(C|S_init)")


def test_outputs_validation():
    hy = _hy()
    inp = synth.make_inputs("gdn", 1, 2, 64, [40], torch.bfloat16, seed=97, with_q=True)
    d = to_dev(inp)
    import ctypes
    lib = hy.load_library()
    S, lam, P = hy.build_outputs("gdn", 1, 2, 64, "cuda")
    O = torch.empty_like(d["v"])
    a = hy.make_build_args("gdn", d["k"], d["v"], inp.seg_offsets, d["log_gate"], None, d["beta"],
                           S, lam, P, O=O)     # outputs without queries
    assert lib.hypic_build_segments(ctypes.byref(a), None) == 1
    a = hy.make_build_args("gdn", d["k"], d["v"], inp.seg_offsets, d["log_gate"], None, d["beta"],
                           S, lam, P, q=d["q"], O=d["v"])   # outputs over an input
    assert lib.hypic_build_segments(ctypes.byref(a), None) == 1


def test_workload_gdn_outputs():
    """The GDN workload (32 value / 16 key heads, d = 128, 16 x 2048 tokens, bf16) with its
    queries: every (segment, head) block of O(C|0)."""
    inp = synth.make_workload("gdn", with_q=True)
    S, lam, P, O = gpu_build_out(inp)
    assert out_errors(inp, f64(O), oracle_outputs(inp)) <= TOL[inp.dtype]


@pytest.mark.parametrize("family", ["gdn", "delta"])
def test_tensor_core_outputs_over_many_units_and_key_sharing(family):
    """The tensor-core build's outputs instance over more (segment, head) units than SMs,
    ragged segments (empty, one-token, partial chunks), grouped-query keys (4 value heads per
    key head), and one long segment that is not split into pieces when outputs are asked for."""
    hy = _hy()
    lens = [int(x) for x in np.random.default_rng(98).integers(0, 300, size=60)]
    lens[:5] = [0, 1, 64, 65, 2000]
    inp = synth.make_inputs(family, 1, 4, 128, lens, torch.bfloat16, seed=99, with_q=True,
                            alpha_scale=0.05)
    d = to_dev(inp)
    assert hy.hypic_build_kernel_name(family, d["k"], d["v"], inp.seg_offsets,
                                      log_gate=d.get("log_gate"), beta=d["beta"], q=d["q"],
                                      O=torch.empty_like(d["v"])) == "build_gdn_tc"
    S, lam, P, O = gpu_build_out(inp)
    assert out_errors(inp, f64(O), oracle_outputs(inp)) <= 2e-2
    So, To = oracle_build(inp)
    assert_close(f64(S), So, 2e-2, "S")
    assert_close(gpu_T(family, lam, P, 128), To, 2e-2, "T")
