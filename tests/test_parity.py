"""CUDA path vs the fp64 oracle on identical seeded inputs (needs a GPU).

Small ragged cases span several 64-token chunks, partial chunks, 1-token and empty
segments; the named workloads run at full size in the same launch configuration as the
benchmark. Every S, every T (materialised in fp64 from the stored (lam, P)) and every
composed prefix state is compared matrix by matrix: relative Frobenius error <= 1e-4 for
fp32 inputs and <= 2e-2 for bf16 inputs.
"""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_state_gdn_gb300 import synth
from tests.helpers import (COMPOSE_TOL, TOL, assert_close, f64, gpu_T, gpu_build, oracle_build,
                           oracle_seq, slice_heads)

pytestmark = pytest.mark.gpu

RAGGED = [200, 64, 1, 0, 129, 300, 63]
FAMILIES = ["linear", "scalar", "diag", "delta", "gdn", "kda"]


def _hy():
    import linear_attention_state_gdn_gb300 as hy
    return hy


def check_build(inp, tol=None):
    tol = tol or TOL[inp.dtype]
    S, lam, P = gpu_build(inp)
    So, To = oracle_build(inp)
    eS = assert_close(f64(S), So, tol, "S")
    eT = assert_close(gpu_T(inp.family, lam, P, inp.d_k), To, tol, "T")
    return S, lam, P, eS, eT


@pytest.mark.parametrize("family", FAMILIES)
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("d", [32, 64, 128])
def test_build_parity_ragged(family, dtype, d):
    inp = synth.make_inputs(family, 2, 4, d, RAGGED, dtype, seed=40 + d, gla_div=8.0,
                            alpha_scale=0.05)
    check_build(inp)


@pytest.mark.parametrize("family", ["gdn", "delta", "kda"])
@pytest.mark.parametrize("H_k,H_v", [(3, 3), (1, 4), (2, 6)])
def test_build_key_head_sharing(family, H_k, H_v):
    """Grouped-query factors 1, 4 and 3: the tensor-core build's chunk preparation handles
    the value heads of one key head two at a time when the factor is even, one at a time
    otherwise (KDA: one at a time, its gram depends on the value head's gates)."""
    inp = synth.make_inputs(family, H_k, H_v, 128, RAGGED, torch.bfloat16, seed=47, alpha_scale=0.05)
    check_build(inp)


@pytest.mark.parametrize("family", ["gdn", "delta", "kda"])
def test_build_more_units_than_sms(family):
    """More (segment, head) units than SMs, in several rounds per SM: 180 ragged segments
    (empty, one-token, one-chunk and multi-chunk) x 2 value heads through the tensor-core
    build, whose records of many short units interleave in the workspace."""
    lens = [int(x) for x in np.random.default_rng(44).integers(0, 200, size=180)]
    lens[:6] = [0, 1, 64, 65, 0, 130]
    inp = synth.make_inputs(family, 1, 2, 128, lens, torch.bfloat16, seed=45, alpha_scale=0.05)
    check_build(inp)


@pytest.mark.parametrize("family,per_token", [("gdn", False), ("delta", False), ("kda", False), ("linear", False),
                                              ("scalar", False), ("scalar", True), ("diag", False)])
@pytest.mark.parametrize("lens", [[3000], [2500, 100, 0, 65]])
def test_build_split_segments(family, per_token, lens):
    """Few units (a long prompt as one or a few segments): the tensor-core builds cut each
    segment into up to eight chunk-aligned pieces, build them in parallel and compose them
    back into the segment's entry. The result is the entry of the whole segment."""
    hy = _hy()
    inp = synth.make_inputs(family, 1, 2, 128, lens, torch.bfloat16, seed=46, alpha_scale=0.05,
                            gla_div=8.0, per_token_scalar=per_token)
    d = {n: t.cuda() for n, t in inp.tensors().items()}
    need = hy.hypic_build_workspace_bytes(family, d["k"], d["v"], inp.seg_offsets,
                                          log_gate=d.get("log_gate"), log_gamma=d.get("log_gamma"),
                                          beta=d.get("beta"))
    chunks = sum((n + 63) // 64 for n in lens)
    records = chunks * 2 * 8192 + 256 if family in ("gdn", "delta", "kda") else 0
    assert need > records      # (records and tail, and) the pieces' scratch
    check_build(inp)


@pytest.mark.parametrize("family", ["gdn", "delta", "kda"])
def test_build_halved_trailing_segments(family):
    """A call whose units take two rounds of SMs with a nearly empty second round (80 equal
    segments x 2 heads = 160 units): its last segments are built as halves and composed back
    in one batched launch."""
    inp = synth.make_inputs(family, 1, 2, 128, [130] * 80, torch.bfloat16, seed=48, alpha_scale=0.05)
    check_build(inp)


@pytest.mark.parametrize("alpha_scale", [0.3, 0.6])
def test_build_kda_strong_channel_gates(alpha_scale):
    """The channel-gated delta rule on the tensor cores with strong per-channel decays (chunk
    log-decays of -20 to -45 per channel at 0.6): the gated keys e^{c} k and e^{-c} k of the
    chunk's gram span a wide range, and the transition is carried as exp(sum m) P."""
    inp = synth.make_inputs("kda", 2, 4, 128, RAGGED, torch.bfloat16, seed=49, alpha_scale=alpha_scale)
    lg, offs = f64(inp.log_gate), inp.seg_offsets
    sums = [lg[a:min(a + 64, offs[j + 1])].sum(0) for j in range(len(offs) - 1)
            for a in range(int(offs[j]), int(offs[j + 1]), 64)]
    assert min(float(x.min()) for x in sums) > -60   # inside the supported range
    check_build(inp)


def test_build_scalar_per_token_gate():
    inp = synth.make_inputs("scalar", 2, 2, 128, [300, 77], torch.bfloat16, seed=41,
                            per_token_scalar=True)
    check_build(inp)


def test_build_lam_closed_forms():
    """lam is the plain sum of the log gates (scalar: L * log gamma)."""
    inp = synth.make_inputs("scalar", 4, 4, 64, [100, 7, 0], torch.bfloat16, seed=42)
    _, lam, _ = gpu_build(inp)
    lg = f64(inp.log_gamma)
    ref = np.array([[L * lg[h] for h in range(4)] for L in (100, 7, 0)])
    np.testing.assert_allclose(f64(lam), ref, rtol=1e-6, atol=1e-7)
    inp = synth.make_inputs("linear", 1, 2, 32, [5, 9], torch.float32, seed=43)
    _, lam, _ = gpu_build(inp)
    assert np.all(f64(lam) == 0)


def test_build_empty_segment_is_identity():
    inp = synth.make_inputs("gdn", 1, 2, 128, [65, 0, 3], torch.bfloat16, seed=44)
    S, lam, P = gpu_build(inp)
    assert torch.all(S[1] == 0)
    assert torch.all(lam[1] == 0)
    eye = torch.eye(128, device=P.device).expand(2, 128, 128)
    assert torch.equal(P[1], eye)


def test_build_out_seg_stride_writes_a_layer_slice():
    """out_seg_stride lets two layers write interleaved into one [n_seg, 2*H_v] cache."""
    hy = _hy()
    inp = synth.make_inputs("gdn", 2, 4, 64, [70, 130], torch.bfloat16, seed=45)
    d = {n: t.cuda() for n, t in inp.tensors().items()}
    S, lam, P = hy.build_outputs("gdn", 2, 4, 64, "cuda", out_seg_stride=8)
    S.fill_(7.0)
    # a [n_seg, 8, ...] slice is not contiguous: pass the base pointers of unit 4 instead
    ref_S, ref_lam, ref_P = gpu_build(inp)
    a = hy.make_build_args("gdn", d["k"], d["v"], inp.seg_offsets, d["log_gate"], None,
                           d["beta"], None, None, None, out_seg_stride=8)
    a.S = S.data_ptr() + 4 * 64 * 64 * 4
    a.lam = lam.data_ptr() + 4 * 4
    a.P = P.data_ptr() + 4 * 64 * 64 * 4
    import ctypes
    st = hy.load_library().hypic_build_segments(ctypes.byref(a),
                                               torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    assert torch.equal(S[:, 4:], ref_S) and torch.equal(P[:, 4:], ref_P)
    assert torch.equal(lam[:, 4:], ref_lam)
    assert torch.all(S[:, :4] == 7.0)


# ------------------------------------------------------------------ compose scan

@pytest.mark.parametrize("family", FAMILIES)
@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("with_S0", [False, True])
def test_compose_parity(family, d, with_S0):
    hy = _hy()
    c = synth.make_compose_inputs(family, 9, 5, d, seed=50 + d, with_S0=with_S0)
    dev = lambda t: None if t is None else t.cuda()
    pref = hy.hypic_compose_scan(family, dev(c.S), dev(c.lam), dev(c.P), dev(c.S0))
    torch.cuda.synchronize()
    T = oracle.materialize_T(family, f64(c.lam), f64(c.P), d_k=d)
    ref = oracle.compose_scan(T, f64(c.S), f64(c.S0))
    assert_close(f64(pref), ref, COMPOSE_TOL, "prefix")
    # the carried term T_j prefix_{j-1} on its own (O(1) here, so not masked by S_j), at the
    # same bound as the prefix: the compose inputs are fp32
    assert_close(f64(pref) - f64(c.S), ref - f64(c.S), COMPOSE_TOL, "carried term")


@pytest.mark.parametrize("which,n_seg", [("two", 16), ("most", 16), ("over", 16), ("two", 1),
                                          ("two", 64), ("most", 3)])
@pytest.mark.parametrize("with_S0", [False, True])
def test_compose_few_units_column_blocks(which, n_seg, with_S0):
    """A plain d = 128 scan of few units runs four CTAs per unit, each carrying 32 state
    columns, while all of them fit on the SMs at once; one unit more and the one-CTA-per-unit
    kernel takes over. One to 64 segments (more steps than the kernel's rings have slots),
    prefix and carried term at the compose bound."""
    hy = _hy()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    units = {"two": 2, "most": sms // 4, "over": sms // 4 + 1}[which]
    c = synth.make_compose_inputs("gdn", n_seg, units, 128, seed=55 + units + n_seg, with_S0=with_S0)
    dev = lambda t: None if t is None else t.cuda()
    expect = "compose_dense_tc" if which == "over" else "compose_dense_cols"
    assert hy.hypic_compose_kernel_name("gdn", dev(c.S), dev(c.lam), dev(c.P), dev(c.S0)) == expect
    pref = hy.hypic_compose_scan("gdn", dev(c.S), dev(c.lam), dev(c.P), dev(c.S0))
    torch.cuda.synchronize()
    assert hy.hypic_get_device_status() == 0
    T = oracle.materialize_T("gdn", f64(c.lam), f64(c.P))
    ref = oracle.compose_scan(T, f64(c.S), f64(c.S0))
    assert_close(f64(pref), ref, COMPOSE_TOL, "prefix")
    assert_close(f64(pref) - f64(c.S), ref - f64(c.S), COMPOSE_TOL, "carried term")


def test_compose_single_segment_is_S_plus_carry():
    hy = _hy()
    c = synth.make_compose_inputs("gdn", 1, 3, 128, seed=51)
    pref = hy.hypic_compose_scan("gdn", c.S.cuda(), c.lam.cuda(), c.P.cuda())
    assert torch.equal(pref.cpu(), c.S)     # zero initial state: prefix_0 = S_0 exactly


# ------------------------------------------------------------------ composed entries

def compose_with_totals(family, S, lam, P, S0=None):
    hy = _hy()
    U, d = S.shape[1], S.shape[2]
    lam_t = torch.empty((U, d) if family == "diag" else (U,), dtype=torch.float32, device=S.device)
    P_t = torch.empty((U, d, d), dtype=torch.float32, device=S.device) if P is not None else None
    pref = hy.hypic_compose_scan(family, S, lam, P, S0, lam_total=lam_t, P_total=P_t)
    torch.cuda.synchronize()
    assert hy.hypic_get_device_status() == 0
    return pref, lam_t, P_t


@pytest.mark.parametrize("family", FAMILIES)
@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("with_S0", [False, True])
def test_compose_totals_parity(family, d, with_S0):
    """lam_total = sum_j lam_j and P_total = P_{n-1} ... P_0 next to the prefix scan, whose
    output must not change when the totals are requested."""
    c = synth.make_compose_inputs(family, 9, 5, d, seed=150 + d, with_S0=with_S0)
    dev = lambda t: None if t is None else t.cuda()
    pref, lam_t, P_t = compose_with_totals(family, dev(c.S), dev(c.lam), dev(c.P), dev(c.S0))
    T = oracle.materialize_T(family, f64(c.lam), f64(c.P), d_k=d)
    assert_close(f64(pref), oracle.compose_scan(T, f64(c.S), f64(c.S0)), COMPOSE_TOL, "prefix")
    lam_o, P_o = oracle.compose_transitions(family, f64(c.lam), f64(c.P), d_k=d)
    np.testing.assert_allclose(f64(lam_t), lam_o, rtol=1e-5, atol=1e-6)
    if P_o is not None:
        assert_close(f64(P_t)[None], P_o[None], COMPOSE_TOL, "P_total")


def test_compose_totals_stay_in_range_on_long_chains():
    """64 entries whose P_j have spectral norm about 0.1: the plain product (about 1e-64)
    is below the fp32 range. The d = 128 kernel carries it scaled by powers of two and
    reports the exponent in lam_total, so exp(lam_total) P_total is still the composed
    transition (compared at its own scale, in fp64)."""
    c = synth.make_compose_inputs("gdn", 64, 6, 128, seed=154, p_norm=0.1)
    pref, lam_t, P_t = compose_with_totals("gdn", c.S.cuda(), c.lam.cuda(), c.P.cuda())
    lam_o, P_o = oracle.compose_transitions("gdn", f64(c.lam), f64(c.P))
    assert np.abs(P_o).max() < 1e-50            # out of fp32's range
    E = (lam_o - f64(lam_t)) / np.log(2.0)       # the exponents applied
    assert np.all(E > 100) and np.allclose(E, np.round(E), atol=1e-3)
    got = f64(P_t) * np.exp(f64(lam_t) - lam_o)[:, None, None]
    assert_close(got[None], P_o[None], COMPOSE_TOL, "scaled P_total")


@pytest.mark.parametrize("family", FAMILIES)
def test_composed_entry_is_the_entry_of_the_concatenation(family):
    """Segments built on the GPU, composed into one entry (prefix[n-1], lam_total, P_total),
    against the oracle's entry of the same tokens built as one segment (O(1) transitions,
    so that T is compared at its own scale)."""
    inp = synth.make_inputs(family, 2, 4, 128, RAGGED, torch.bfloat16, seed=61, gla_div=64.0,
                            alpha_scale=0.002, beta_shift=-2.0)
    S, lam, P = gpu_build(inp)
    pref, lam_t, P_t = compose_with_totals(family, S, lam, P)
    N = int(inp.seg_offsets[-1])
    S_w, T_w = oracle.build_segments(family, [0, N], f64(inp.k), f64(inp.v), f64(inp.log_gate),
                                     f64(inp.log_gamma), f64(inp.beta))
    tol = TOL[inp.dtype]
    assert_close(f64(pref[-1])[None], S_w, tol, "S of the concatenation")
    assert_close(gpu_T(family, lam_t[None], None if P_t is None else P_t[None], 128), T_w, tol,
                 "T of the concatenation")


def test_compose_totals_are_validated():
    hy = _hy()
    c = synth.make_compose_inputs("scalar", 3, 2, 64, seed=152)
    S, lam = c.S.cuda(), c.lam.cuda()
    with pytest.raises(hy.HypicError):     # P_total exists for dense transitions only
        hy.hypic_compose_scan("scalar", S, lam, P_total=torch.empty(2, 64, 64, device="cuda"))
    g = synth.make_compose_inputs("gdn", 3, 2, 64, seed=153)
    S, lam, P = g.S.cuda(), g.lam.cuda(), g.P.cuda()
    prefix = torch.empty_like(S)
    lam_t = torch.empty(2, device="cuda")
    with pytest.raises(hy.HypicError):     # a total may not overlap prefix
        hy.hypic_compose_scan("gdn", S, lam, P, prefix=prefix, lam_total=lam_t, P_total=prefix[0])
    with pytest.raises(hy.HypicError):     # P_total needs lam_total (its scale)
        hy.hypic_compose_scan("gdn", S, lam, P, P_total=torch.empty(2, 64, 64, device="cuda"))
    with pytest.raises(hy.HypicError):     # nor an input
        hy.hypic_compose_scan("gdn", S, lam, P, lam_total=lam[0])


# ------------------------------------------------------------------ build -> compose chain

@pytest.mark.parametrize("family", FAMILIES)
def test_chain_matches_sequential(family):
    hy = _hy()
    inp = synth.make_inputs(family, 2, 4, 128, RAGGED, torch.bfloat16, seed=60, gla_div=64.0,
                            alpha_scale=0.002, beta_shift=-2.0)
    S, lam, P = gpu_build(inp)
    pref = hy.hypic_compose_scan(family, S, lam, P)
    torch.cuda.synchronize()
    seq = oracle_seq(inp)
    assert_close(f64(pref), seq, TOL[inp.dtype], "prefix vs sequential")


# ------------------------------------------------------------------ stress: O(1) transitions

@pytest.mark.parametrize("case", ["deltanet", "gla_slow", "retnet_slow"])
def test_stress_carried_term(case):
    """Transitions near the identity make T_j prefix_{j-1} as large as S_j, so a compose
    that dropped or transposed T would fail here (the workload gates hide it)."""
    hy = _hy()
    if case == "deltanet":
        inp = synth.make_inputs("delta", 2, 4, 128, [300, 129, 64, 200], torch.bfloat16,
                                seed=70, beta_shift=-3.0)
    elif case == "gla_slow":
        inp = synth.make_inputs("diag", 4, 4, 128, [300, 129, 64, 200], torch.bfloat16,
                                seed=71, gla_div=256.0)
    else:
        inp = synth.make_inputs("scalar", 4, 4, 128, [300, 129, 64, 200], torch.bfloat16,
                                seed=72, retnet_gammas=False)
    S, lam, P = gpu_build(inp)
    pref = hy.hypic_compose_scan(inp.family, S, lam, P)
    torch.cuda.synchronize()
    seq = oracle_seq(inp)
    So, To = oracle_build(inp)
    carried_ref = seq[1:] - So[1:]
    assert np.linalg.norm(carried_ref) > 0.3 * np.linalg.norm(So[1:])
    tol = TOL[inp.dtype]
    assert_close(f64(pref), seq, tol, "prefix")
    assert_close(f64(pref)[1:] - f64(S)[1:], carried_ref, tol, "carried term")
    assert_close(gpu_T(inp.family, lam, P, 128), To, tol, "T")


# ------------------------------------------------------------------ named workloads

def _workload_chain(name):
    hy = _hy()
    inp = synth.make_workload(name)
    S, lam, P, eS, eT = check_build(inp)
    pref = hy.hypic_compose_scan(inp.family, S, lam, P)
    torch.cuda.synchronize()
    seq = oracle_seq(inp)
    eP = assert_close(f64(pref), seq, TOL[inp.dtype], "prefix")
    return eS, eT, eP


def test_workload_gdn_tiny_fp32():
    eS, eT, eP = _workload_chain("gdn_tiny")
    assert max(eS, eT, eP) <= 1e-4


def test_workload_retnet():
    _workload_chain("retnet")


def test_workload_gla():
    _workload_chain("gla")


def test_workload_gdn():
    _workload_chain("gdn")


def test_workload_kda():
    """The channel-gated delta rule at the GDN workload's shape (32 value / 16 key heads,
    d = 128, 16 x 2048 tokens, bf16): every S, T and prefix state."""
    _workload_chain("kda")


def test_workload_gdn_compose_sampled():
    """48 layers x 32 heads x 64 ragged segments, built layer by layer into one
    [64, 1536] cache exactly as the benchmark does, then one compose launch over all 1536
    units. The oracle rebuilds and runs sequentially a sample of (layer, head) units from
    the same drawn bytes (copied back to the host)."""
    from bench import build_gdn_compose_cache
    hy = _hy()
    S, lam, P, info = build_gdn_compose_cache(layers=48)
    pref = hy.hypic_compose_scan("gdn", S, lam, P)
    torch.cuda.synchronize()
    rng = np.random.default_rng(5)
    H = info["H_v"]
    for layer in sorted(rng.choice(48, size=3, replace=False)):
        layer = int(layer)
        heads = [int(h) for h in sorted(rng.choice(H, size=2, replace=False))]
        inp = slice_heads(synth.to_host(synth.make_workload_device("gdn_compose", layer)), heads)
        seq = oracle_seq(inp)
        So, To = oracle_build(inp)
        for i, h in enumerate(heads):
            u = layer * H + h
            assert_close(f64(pref[:, u]), seq[:, i], 2e-2, f"prefix layer {layer} head {h}")
            assert_close(f64(S[:, u]), So[:, i], 2e-2, "S")
            assert_close(gpu_T("gdn", lam[:, u], P[:, u], 128), To[:, i], 2e-2, "T")


def test_workload_gdn_compose_full_size_compose_only():
    """The compose launch at full size (64 segments x 1536 units) on fp32 cached entries
    drawn directly (O(1) transitions): 1e-4 on sampled units."""
    hy = _hy()
    c = synth.make_compose_inputs("gdn", 64, 1536, 128, seed=80)
    pref = hy.hypic_compose_scan("gdn", c.S.cuda(), c.lam.cuda(), c.P.cuda())
    torch.cuda.synchronize()
    rng = np.random.default_rng(6)
    units = sorted(rng.choice(1536, size=6, replace=False))
    T = oracle.materialize_T("gdn", f64(c.lam[:, units]), f64(c.P[:, units]))
    ref = oracle.compose_scan(T, f64(c.S[:, units]))
    assert_close(f64(pref[:, units]), ref, COMPOSE_TOL, "prefix")


def test_workload_gdn_compose_full_size_with_totals():
    """The composed-entry launch the benchmark times (64 segments x 1536 units, with
    lam_total and P_total) on fp32 cached entries drawn directly: 1e-4 on sampled units."""
    c = synth.make_compose_inputs("gdn", 64, 1536, 128, seed=81)
    pref, lam_t, P_t = compose_with_totals("gdn", c.S.cuda(), c.lam.cuda(), c.P.cuda())
    rng = np.random.default_rng(7)
    units = sorted(rng.choice(1536, size=6, replace=False))
    T = oracle.materialize_T("gdn", f64(c.lam[:, units]), f64(c.P[:, units]))
    assert_close(f64(pref[:, units]), oracle.compose_scan(T, f64(c.S[:, units])), COMPOSE_TOL, "prefix")
    lam_o, P_o = oracle.compose_transitions("gdn", f64(c.lam[:, units]), f64(c.P[:, units]))
    # the composed transition exp(lam_total) P_total at its own scale: P_total carries the
    # power of two whose exponent lam_total reports
    E = (lam_o - f64(lam_t[units])) / np.log(2.0)
    assert np.allclose(E, np.round(E), atol=1e-3)
    got = f64(P_t[units]) * np.exp(f64(lam_t[units]) - lam_o)[:, None, None]
    assert_close(got[None], P_o[None], COMPOSE_TOL, "P_total")


# ------------------------------------------------------------------ kernel selection

@pytest.mark.parametrize("family,dtype,d,expect", [
    ("linear", torch.bfloat16, 128, "build_gated_tc"), ("scalar", torch.bfloat16, 128, "build_gated_tc"),
    ("diag", torch.bfloat16, 128, "build_gated_tc"), ("diag", torch.float32, 128, "build_gated_simt"),
    ("scalar", torch.bfloat16, 64, "build_gated_simt"), ("gdn", torch.float32, 32, "build_seq"),
    ("gdn", torch.bfloat16, 128, "build_gdn_tc"), ("delta", torch.bfloat16, 128, "build_gdn_tc"),
    ("gdn", torch.float32, 128, "build_seq"), ("gdn", torch.bfloat16, 64, "build_seq"),
    ("kda", torch.bfloat16, 128, "build_kda_tc"), ("kda", torch.float32, 32, "build_seq"),
    ("kda", torch.bfloat16, 64, "build_seq"),
])
def test_build_kernel_selection(family, dtype, d, expect):
    """bf16 inputs with d = 128 run on the tensor cores; fp32 inputs and smaller heads run the
    exact CUDA-core kernels (the parity cases above cover both)."""
    hy = _hy()
    inp = synth.make_inputs(family, 2, 2, d, [70, 3], dtype, seed=90)
    dd = {n: t.cuda() for n, t in inp.tensors().items()}
    name = hy.hypic_build_kernel_name(family, dd["k"], dd["v"], inp.seg_offsets,
                                      log_gate=dd.get("log_gate"), log_gamma=dd.get("log_gamma"),
                                      beta=dd.get("beta"))
    assert name == expect


@pytest.mark.parametrize("family,d,units,expect", [("gdn", 128, 2, "compose_dense_cols"),
                                                   ("gdn", 128, 200, "compose_dense_tc"),
                                                   ("delta", 64, 2, "compose_dense_simt"),
                                                   ("diag", 128, 2, "compose_scaled")])
def test_compose_kernel_selection(family, d, units, expect):
    hy = _hy()
    c = synth.make_compose_inputs(family, 2, units, d, seed=91)
    assert hy.hypic_compose_kernel_name(family, c.S) == expect


# ------------------------------------------------------------------ determinism / liveness

def test_gdn_build_is_deterministic_with_clean_status():
    """Two builds of the same 16 layers of the 64-segment workload (ragged 256-1024-token
    segments) are bitwise identical and no launch reports a timed-out wait: the build has
    no data race and no wait that can miss its phase, whatever the relative speed of its
    roles."""
    hy = _hy()
    outs = []
    for rep in range(2):
        res = []
        for layer in range(16):
            inp = synth.make_workload_device("gdn_compose", layer, "cuda")
            torch.cuda.synchronize()
            S, lam, P = hy.hypic_build_segments("gdn", inp.k, inp.v, inp.seg_offsets,
                                                log_gate=inp.log_gate, beta=inp.beta)
            assert hy.hypic_get_device_status() == 0, f"layer {layer}: device status not OK"
            res.append((S, lam, P))
        outs.append(res)
    for (S1, l1, P1), (S2, l2, P2) in zip(*outs):
        assert torch.equal(S1, S2) and torch.equal(P1, P2) and torch.equal(l1, l2)
