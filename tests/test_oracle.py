"""Pins for the fp64 oracle: each check ties it to something other than itself.

What pins what (a plausible mistake anywhere in the oracle fails at least one check):

* hand-derived fixtures under tests/golden (exact decimals, derivation in the file): GDN,
  RetNet and GLA;
* closed forms: plain linear attention (S = K^T V, T = I), scalar decay
  (T = gamma^L I, S = decayed sum), diagonal gates (T = Diag(prod g)), one-token GDN;
* delta-rule semantics: with b = 1 and |k| = 1 the last write is retrieved exactly
  (k^T S = v^T) and the last key is annihilated by T (k^T T = 0);
* invariants: det T = prod_t a_t^d (1 - b_t |k_t|^2); S(C|S0) - S(C|0) = T S0; |T|_2 <= 1
  for b |k|^2 in [0, 2]; with b_t = 2 / |k_t|^2 (Householder reflections) T is orthogonal and
  the last key is flipped by the leftmost factor;
* brute force on tiny inputs in exact rational arithmetic (sympy), with the transition
  factors formed as dense matrices and multiplied out;
* the composition theorem against the oracle's own sequential run, and the failure of
  naive end-state addition for RetNet (but not for plain linear attention);
* the composed transition of consecutive segments against the transition of the same
  tokens built as one segment.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from linear_attention_state_gdn_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f64(t):
    return None if t is None else t.double().numpy()


def run_build(inp, want_T=True):
    return oracle.build_segments(inp.family, inp.seg_offsets, f64(inp.k), f64(inp.v),
                                 f64(inp.log_gate), f64(inp.log_gamma), f64(inp.beta),
                                 want_T=want_T)


def run_seq(inp, S0=None):
    return oracle.run_sequential(inp.family, inp.seg_offsets, f64(inp.k), f64(inp.v),
                                 f64(inp.log_gate), f64(inp.log_gamma), f64(inp.beta), S0=S0)


def relF(a, b):
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


# ------------------------------------------------------------------ hand-derived fixtures

def test_golden_gdn_two_segments():
    g = json.load(open(os.path.join(GOLDEN, "gdn_d2_two_segments.json")))
    k = np.array(g["k"])[:, None, :]
    v = np.array(g["v"])[:, None, :]
    beta = np.array(g["beta"])[:, None]
    log_a = np.log(np.array(g["alpha"]))[:, None]
    offs = np.array(g["seg_offsets"])
    S, T = oracle.build_segments("gdn", offs, k, v, log_gate=log_a, beta=beta)
    np.testing.assert_allclose(S[0, 0], g["S_C1"], atol=1e-14)
    np.testing.assert_allclose(T[0, 0], g["T_C1"], atol=1e-14)
    np.testing.assert_allclose(S[1, 0], g["S_C2"], atol=1e-14)
    np.testing.assert_allclose(T[1, 0], g["T_C2"], atol=1e-14)
    pref = oracle.compose_scan(T, S)
    np.testing.assert_allclose(pref[1, 0], g["S_C1C2"], atol=1e-14)
    seq = oracle.run_sequential("gdn", offs, k, v, log_gate=log_a, beta=beta)
    np.testing.assert_allclose(seq[1, 0], g["S_C1C2"], atol=1e-14)
    np.testing.assert_allclose(S[0, 0] + S[1, 0], g["naive_add"], atol=1e-14)


def test_golden_retnet_scalar():
    g = json.load(open(os.path.join(GOLDEN, "retnet_d1_hand.json")))
    k = np.array(g["k"])[:, None, None]
    v = np.array(g["v"])[:, None, None]
    offs = np.array(g["seg_offsets"])
    log_gamma = np.array([np.log(g["gamma"])])
    S, T = oracle.build_segments("scalar", offs, k, v, log_gamma=log_gamma)
    assert S[0, 0, 0, 0] == pytest.approx(g["S_C1"], abs=1e-14)
    assert T[0, 0, 0, 0] == pytest.approx(g["T_C1"], abs=1e-14)
    assert S[1, 0, 0, 0] == pytest.approx(g["S_C2"], abs=1e-14)
    assert T[1, 0, 0, 0] == pytest.approx(g["T_C2"], abs=1e-14)
    pref = oracle.compose_scan(T, S)
    assert pref[1, 0, 0, 0] == pytest.approx(g["S_C1C2"], abs=1e-14)
    assert S[0, 0, 0, 0] + S[1, 0, 0, 0] == pytest.approx(g["naive_add"], abs=1e-14)


def test_golden_gla_diagonal():
    g = json.load(open(os.path.join(GOLDEN, "gla_d2_hand.json")))
    k = np.array(g["k"])[:, None, :]
    v = np.array(g["v"])[:, None, :]
    log_g = np.log(np.array(g["g"]))[:, None, :]
    offs = np.array(g["seg_offsets"])
    S, T = oracle.build_segments("diag", offs, k, v, log_gate=log_g)
    np.testing.assert_allclose(S[0, 0], g["S_C1"], atol=1e-14)
    np.testing.assert_allclose(T[0, 0], g["T_C1"], atol=1e-14)
    np.testing.assert_allclose(S[1, 0], g["S_C2"], atol=1e-14)
    np.testing.assert_allclose(T[1, 0], g["T_C2"], atol=1e-14)
    pref = oracle.compose_scan(T, S)
    np.testing.assert_allclose(pref[1, 0], g["S_C1C2"], atol=1e-14)
    seq = oracle.run_sequential("diag", offs, k, v, log_gate=log_g)
    np.testing.assert_allclose(seq[1, 0], g["S_C1C2"], atol=1e-14)
    np.testing.assert_allclose(S[0, 0] + S[1, 0], g["naive_add"], atol=1e-14)


# ------------------------------------------------------------------ closed forms

def _segments(inp):
    o = inp.seg_offsets
    return [(int(o[j]), int(o[j + 1])) for j in range(inp.n_seg)]


def test_linear_closed_form():
    inp = synth.make_inputs("linear", 2, 4, 8, [5, 0, 17, 3], torch.float32, seed=1)
    S, T = run_build(inp)
    k, v = f64(inp.k), f64(inp.v)
    for j, (a, b) in enumerate(_segments(inp)):
        for h in range(4):
            ref = k[a:b, h // 2].T @ v[a:b, h]
            np.testing.assert_allclose(S[j, h], ref, atol=1e-13)
            assert np.array_equal(T[j, h], np.eye(8))


@pytest.mark.parametrize("per_token", [False, True])
def test_scalar_closed_form(per_token):
    inp = synth.make_inputs("scalar", 3, 3, 8, [7, 1, 12], torch.float32, seed=2,
                            per_token_scalar=per_token, gla_div=2.0)
    S, T = run_build(inp)
    k, v = f64(inp.k), f64(inp.v)
    for j, (a, b) in enumerate(_segments(inp)):
        for h in range(3):
            if per_token:
                lg = f64(inp.log_gate)[a:b, h]
            else:
                lg = np.full(b - a, f64(inp.log_gamma)[h])
            # weight of token t = product of the gates of the tokens after it
            w = np.exp(np.concatenate([np.cumsum(lg[::-1])[::-1][1:], [0.0]]))
            ref = (k[a:b, h] * w[:, None]).T @ v[a:b, h]
            np.testing.assert_allclose(S[j, h], ref, rtol=1e-12, atol=1e-14)
            np.testing.assert_allclose(T[j, h], np.exp(lg.sum()) * np.eye(8), rtol=1e-12)


def test_diag_closed_form():
    inp = synth.make_inputs("diag", 2, 2, 6, [9, 4], torch.float32, seed=3, gla_div=1.0)
    S, T = run_build(inp)
    k, v, lg = f64(inp.k), f64(inp.v), f64(inp.log_gate)
    for j, (a, b) in enumerate(_segments(inp)):
        for h in range(2):
            g = lg[a:b, h]                                   # [L, d_k]
            after = np.concatenate([np.cumsum(g[::-1], 0)[::-1][1:], np.zeros((1, 6))], 0)
            ref = (k[a:b, h] * np.exp(after)).T @ v[a:b, h]
            np.testing.assert_allclose(S[j, h], ref, rtol=1e-12, atol=1e-14)
            np.testing.assert_allclose(T[j, h], np.diag(np.exp(g.sum(0))), rtol=1e-12)


def test_gdn_one_token_closed_form():
    inp = synth.make_inputs("gdn", 1, 2, 5, [1, 1], torch.float32, seed=4, alpha_scale=0.7)
    S, T = run_build(inp)
    k, v, b, la = f64(inp.k), f64(inp.v), f64(inp.beta), f64(inp.log_gate)
    for t in range(2):
        for h in range(2):
            kk = k[t, 0]
            np.testing.assert_allclose(
                T[t, h], np.exp(la[t, h]) * (np.eye(5) - b[t, h] * np.outer(kk, kk)), atol=1e-15)
            np.testing.assert_allclose(S[t, h], b[t, h] * np.outer(kk, v[t, h]), atol=1e-15)


def test_gdn_beta_zero_is_pure_decay():
    inp = synth.make_inputs("gdn", 2, 2, 8, [33, 10], torch.float32, seed=5)
    inp.beta.zero_()
    S, T = run_build(inp)
    assert np.all(S == 0)
    la = f64(inp.log_gate)
    for j, (a, b) in enumerate(_segments(inp)):
        for h in range(2):
            np.testing.assert_allclose(T[j, h], np.exp(la[a:b, h].sum()) * np.eye(8), rtol=1e-12)


def test_empty_segment_is_identity():
    inp = synth.make_inputs("gdn", 1, 1, 4, [3, 0, 2], torch.float32, seed=6)
    S, T = run_build(inp)
    assert np.all(S[1] == 0) and np.array_equal(T[1, 0], np.eye(4))


# ------------------------------------------------------------------ delta-rule semantics

@pytest.mark.parametrize("family", ["delta", "gdn"])
def test_delta_rule_retrieves_last_write(family):
    """b_L = 1 and |k_L| = 1 (exactly, in binary): k_L^T S = v_L^T and k_L^T T = 0."""
    inp = synth.make_inputs(family, 1, 1, 4, [6], torch.float64, seed=7)
    kl = np.array([0.6, 0.0, -0.8, 0.0])    # |kl| = 1 up to one rounding
    inp.k[-1, 0] = torch.from_numpy(kl)
    inp.beta[-1, 0] = 1.0
    S, T = run_build(inp)
    np.testing.assert_allclose(kl @ S[0, 0], f64(inp.v)[-1, 0], atol=1e-14)
    np.testing.assert_allclose(kl @ T[0, 0], np.zeros(4), atol=1e-15)


# ------------------------------------------------------------------ invariants

@pytest.mark.parametrize("family", ["delta", "gdn"])
def test_det_invariant(family):
    inp = synth.make_inputs(family, 1, 1, 6, [11], torch.float64, seed=8, l2norm_k=False,
                            k_scale=0.5, alpha_scale=0.3)
    S, T = run_build(inp)
    k, b = f64(inp.k)[:, 0], f64(inp.beta)[:, 0]
    sign, logdet = np.linalg.slogdet(T[0, 0])
    la = f64(inp.log_gate)[:, 0].sum() if family == "gdn" else 0.0
    expect = 6 * la + np.sum(np.log(np.abs(1 - b * (k * k).sum(1))))
    assert sign == np.prod(np.sign(1 - b * (k * k).sum(1)))
    assert logdet == pytest.approx(expect, rel=1e-12, abs=1e-12)


@pytest.mark.parametrize("family", ["delta", "gdn"])
def test_transition_is_a_contraction(family):
    """With b_t |k_t|^2 in [0, 2] every factor a_t (I - b_t k_t k_t^T) is symmetric with
    eigenvalues a_t and a_t (1 - b_t |k_t|^2), all in [-1, 1], so |T|_2 <= 1 (a flipped sign in
    the factor, I + b k k^T, breaks it)."""
    inp = synth.make_inputs(family, 1, 2, 8, [64], torch.float64, seed=13)
    S, T = run_build(inp)
    for h in range(2):
        assert np.linalg.norm(T[0, h], 2) <= 1 + 1e-12


def test_reflection_product_is_orthogonal():
    """With b_t = 2 / |k_t|^2 every DeltaNet factor is the Householder reflection through the
    plane orthogonal to k_t: T is orthogonal with det (-1)^L, and each k_t is flipped by its own
    factor, so the last key satisfies k_L^T T = -k_L^T F_{L-1} ... F_1."""
    L, d = 9, 5
    inp = synth.make_inputs("delta", 1, 1, d, [L], torch.float64, seed=12, l2norm_k=False)
    k = f64(inp.k)[:, 0]
    inp.beta = torch.from_numpy((2.0 / (k * k).sum(1))[:, None])
    S, T = run_build(inp)
    Tm = T[0, 0]
    np.testing.assert_allclose(Tm.T @ Tm, np.eye(d), atol=1e-12)
    assert np.linalg.det(Tm) == pytest.approx((-1.0) ** L, abs=1e-10)
    inp_head = synth.make_inputs("delta", 1, 1, d, [L - 1], torch.float64, seed=12, l2norm_k=False)
    inp_head.k, inp_head.v = inp.k[: L - 1], inp.v[: L - 1]
    inp_head.beta = inp.beta[: L - 1]
    _, T_head = run_build(inp_head)
    np.testing.assert_allclose(k[-1] @ Tm, -(k[-1] @ T_head[0, 0]), atol=1e-12)


@pytest.mark.parametrize("family", ["linear", "scalar", "diag", "delta", "gdn"])
def test_T_is_the_jacobian_of_the_end_state(family):
    inp = synth.make_inputs(family, 2, 4, 8, [40], torch.float32, seed=9, gla_div=4.0)
    S, T = run_build(inp)
    S0 = np.random.default_rng(0).standard_normal((4, 8, 8))
    with_s0 = run_seq(inp, S0=S0)
    for h in range(4):
        np.testing.assert_allclose(with_s0[0, h] - S[0, h], T[0, h] @ S0[h], rtol=1e-11,
                                   atol=1e-12)


# ------------------------------------------------------------------ brute force (exact)

def _exact_affine(k, v, a, b):
    """Exact rationals: S_t = F_t S_{t-1} + b_t k_t v_t^T with F_t = a_t (I - b_t k_t k_t^T)
    formed as a dense matrix; T = F_L ... F_1 multiplied out one dense product at a time."""
    import sympy
    d = len(k[0])
    S = sympy.zeros(d, d)
    T = sympy.eye(d)
    for kt, vt, at, bt in zip(k, v, a, b):
        K = sympy.Matrix(kt)
        F = at * (sympy.eye(d) - bt * K * K.T)
        S = F * S + bt * K * sympy.Matrix(vt).T
        T = F * T
    return S, T


def test_bruteforce_exact_rational_gdn():
    sympy = pytest.importorskip("sympy")
    rng = np.random.default_rng(11)
    d, L = 4, 9
    # dyadic rationals are exact in binary floating point
    k = rng.integers(-8, 9, size=(L, d)) / 8.0
    v = rng.integers(-8, 9, size=(L, d)) / 4.0
    b = rng.integers(1, 9, size=L) / 16.0
    a = rng.integers(8, 17, size=L) / 16.0
    S_ex, T_ex = _exact_affine([[Fraction(x) for x in r] for r in k],
                               [[Fraction(x) for x in r] for r in v],
                               [Fraction(x) for x in a], [Fraction(x) for x in b])
    S, T = oracle.build_segments("gdn", [0, L], k[:, None], v[:, None],
                                 log_gate=np.log(a)[:, None], beta=b[:, None])
    S_ex = np.array(S_ex.tolist(), dtype=np.float64)
    T_ex = np.array(T_ex.tolist(), dtype=np.float64)
    assert relF(S[0, 0], S_ex) < 1e-13
    assert relF(T[0, 0], T_ex) < 1e-13


def test_bruteforce_dense_products_random():
    for L in (1, 2, 7, 16):
        inp = synth.make_inputs("gdn", 1, 1, 4, [L], torch.float64, seed=100 + L,
                                alpha_scale=0.5)
        S, T = run_build(inp)
        k, v = f64(inp.k)[:, 0], f64(inp.v)[:, 0]
        a, b = np.exp(f64(inp.log_gate)[:, 0]), f64(inp.beta)[:, 0]
        Tb, Sb = np.eye(4), np.zeros((4, 4))
        for t in range(L):
            F = a[t] * (np.eye(4) - b[t] * np.outer(k[t], k[t]))
            Sb = F @ Sb + b[t] * np.outer(k[t], v[t])
            Tb = F @ Tb
        assert relF(T[0, 0], Tb) < 1e-13 and relF(S[0, 0], Sb) < 1e-13


# ------------------------------------------------------------------ composition theorem

@pytest.mark.parametrize("family", ["linear", "scalar", "diag", "delta", "gdn"])
def test_composition_equals_sequential(family):
    inp = synth.make_inputs(family, 2, 4, 16, [70, 1, 0, 129, 64, 33], torch.bfloat16,
                            seed=20, gla_div=8.0, alpha_scale=0.02)
    S, T = run_build(inp)
    pref = oracle.compose_scan(T.reshape(inp.n_seg, 4, 16, 16), S)
    seq = run_seq(inp)
    for j in range(inp.n_seg):
        for h in range(4):
            if np.linalg.norm(seq[j, h]) == 0:
                assert np.linalg.norm(pref[j, h]) == 0
            else:
                assert relF(pref[j, h], seq[j, h]) < 1e-12


def test_compose_scan_with_initial_state_matches_matmul_chain():
    c = synth.make_compose_inputs("gdn", 5, 3, 8, seed=21, with_S0=True)
    T = oracle.materialize_T("gdn", c.lam.double().numpy(), c.P.double().numpy())
    S, S0 = c.S.double().numpy(), c.S0.double().numpy()
    pref = oracle.compose_scan(T, S, S0)
    for u in range(3):
        cur = S0[u]
        for j in range(5):
            cur = np.matmul(T[j, u], cur) + S[j, u]
            assert relF(pref[j, u], cur) < 1e-13


def test_composition_is_associative():
    c = synth.make_compose_inputs("gdn", 3, 1, 6, seed=22)
    T = oracle.materialize_T("gdn", c.lam.double().numpy(), c.P.double().numpy())[:, 0]
    S = c.S.double().numpy()[:, 0]
    # ((3 o 2) o 1) and (3 o (2 o 1)) as pairs (T, S), then applied to zero
    T32, S32 = T[2] @ T[1], T[2] @ S[1] + S[2]
    S21 = T[1] @ S[0] + S[1]
    left = T32 @ S[0] + S32
    right = T[2] @ S21 + S[2]
    pref = oracle.compose_scan(T[:, None], S[:, None])[2, 0]
    assert relF(left, right) < 1e-13 and relF(pref, right) < 1e-13


def test_materialize_T_forms():
    lam = np.array([[-0.5, 0.0]])
    np.testing.assert_allclose(oracle.materialize_T("scalar", lam, d_k=3)[0, 0],
                               np.exp(-0.5) * np.eye(3))
    np.testing.assert_array_equal(oracle.materialize_T("linear", lam, d_k=3)[0, 1], np.eye(3))
    lv = np.array([[[-1.0, 0.25]]])
    np.testing.assert_allclose(oracle.materialize_T("diag", lv)[0, 0], np.diag(np.exp([-1, .25])))
    P = np.arange(4.0).reshape(1, 1, 2, 2)
    np.testing.assert_allclose(oracle.materialize_T("gdn", np.array([[np.log(2.0)]]), P)[0, 0],
                               2 * P[0, 0])


# ------------------------------------------------------------------ composed entries

def segment_log_scale(inp):
    """lam of every (segment, value head) from the gates alone: the sum of the log-gates
    over the segment (L log gamma for a constant decay, 0 without gates)."""
    offs = inp.seg_offsets
    n, H, d = inp.n_seg, inp.H_v, inp.d_k
    lam = np.zeros((n, H, d) if inp.family == "diag" else (n, H))
    for j in range(n):
        a, b = offs[j], offs[j + 1]
        if inp.log_gate is not None:
            lam[j] = f64(inp.log_gate)[a:b].sum(0)
        elif inp.log_gamma is not None:
            lam[j] = (b - a) * f64(inp.log_gamma)
    return lam


@pytest.mark.parametrize("family,per_token", [("linear", False), ("scalar", False), ("scalar", True),
                                              ("diag", False), ("delta", False), ("gdn", False)])
def test_composed_transition_is_the_transition_of_the_concatenation(family, per_token):
    # segments built one by one, their transitions composed, against the same tokens built
    # as one segment: T(C_0 ... C_4) = T_4 ... T_0, through the log-scaled storage
    inp = synth.make_inputs(family, 2, 4, 8, [9, 0, 13, 1, 6], torch.float32, seed=23,
                            gla_div=8.0, alpha_scale=0.1, per_token_scalar=per_token)
    _, T = run_build(inp)
    lam = segment_log_scale(inp)
    dense = family in ("delta", "gdn")
    P = T * np.exp(-lam)[..., None, None] if dense else None
    lam_t, P_t = oracle.compose_transitions(family, lam, P, d_k=8)
    T_t = oracle.materialize_T(family, lam_t, P_t, d_k=8)
    N = int(inp.seg_offsets[-1])
    _, T_whole = oracle.build_segments(family, [0, N], f64(inp.k), f64(inp.v), f64(inp.log_gate),
                                       f64(inp.log_gamma), f64(inp.beta))
    for h in range(4):
        assert relF(T_t[h], T_whole[0, h]) < 1e-12
    if dense:
        # the order is what the check above fixes: the reversed product is far off
        rev = P[0, 0]
        for j in range(1, inp.n_seg):
            rev = rev @ P[j, 0]
        assert relF(np.exp(lam_t[0]) * rev, T_whole[0, 0]) > 1e-3


def test_composed_transition_of_one_segment_is_that_segment():
    c = synth.make_compose_inputs("gdn", 1, 3, 8, seed=24)
    lam, P = c.lam.double().numpy(), c.P.double().numpy()
    lam_t, P_t = oracle.compose_transitions("gdn", lam, P)
    np.testing.assert_array_equal(lam_t, lam[0])
    np.testing.assert_array_equal(P_t, P[0])
    lam_l, P_l = oracle.compose_transitions("linear", lam, None, d_k=8)
    assert P_l is None and not lam_l.any()


# ------------------------------------------------------------------ naive addition

def test_naive_add_exact_for_linear_only():
    inp = synth.make_inputs("linear", 1, 1, 8, [50, 60, 70], torch.float32, seed=30)
    S, _ = run_build(inp, want_T=False)
    seq = run_seq(inp)
    np.testing.assert_allclose(S.sum(0), seq[-1], rtol=1e-12, atol=1e-13)


def test_naive_add_fails_for_retnet_by_the_predicted_amount():
    inp = synth.make_inputs("scalar", 1, 1, 8, [50, 60], torch.float32, seed=31)
    S, T = run_build(inp)
    seq = run_seq(inp)
    g = np.exp(f64(inp.log_gamma)[0])
    naive = S[0, 0] + S[1, 0]
    np.testing.assert_allclose(naive - seq[1, 0], (1 - g ** 60) * S[0, 0], rtol=1e-11, atol=1e-13)
    assert relF(naive, seq[1, 0]) > 1e-2


# ------------------------------------------------------------------ KDA (channel-gated delta rule)

def _kda_inputs(L, d, seed, **kw):
    return synth.make_inputs("kda", 1, 2, d, [L], torch.float64, seed=seed, alpha_scale=0.3, **kw)


def test_golden_kda_outputs():
    g = json.load(open(os.path.join(GOLDEN, "kda_d2_outputs.json")))
    k = np.array(g["k"])[:, None, :]
    v = np.array(g["v"])[:, None, :]
    q = np.array(g["q"])[:, None, :]
    beta = np.array(g["beta"])[:, None]
    lg = np.log(np.array(g["alpha"]))[:, None, :]
    S, T = oracle.build_segments("kda", g["seg_offsets"], k, v, lg, None, beta)
    np.testing.assert_allclose(S[0, 0], g["S_C"], atol=1e-14)
    np.testing.assert_allclose(T[0, 0], g["T_C"], atol=1e-14)
    O = oracle.outputs("kda", g["seg_offsets"], k, v, q, lg, None, beta)
    np.testing.assert_allclose(O[:, 0], g["O"], atol=1e-14)


def test_kda_with_equal_channel_gates_is_gdn():
    """A per-channel decay that is the same on every channel is the GDN scalar gate."""
    inp = _kda_inputs(37, 6, seed=160)
    a = f64(inp.log_gate)[:, :, 0]
    inp.log_gate = torch.from_numpy(np.repeat(a[:, :, None], 6, axis=2))
    gdn = synth.make_inputs("gdn", 1, 2, 6, [37], torch.float64, seed=160)
    gdn.k, gdn.v, gdn.beta, gdn.log_gate = inp.k, inp.v, inp.beta, torch.from_numpy(a)
    S1, T1 = run_build(inp)
    S2, T2 = run_build(gdn)
    assert relF(S1, S2) < 1e-13 and relF(T1, T2) < 1e-13


def test_kda_with_beta_zero_is_the_diagonal_decay():
    """b = 0 removes the delta update and the write: S = 0 and T = Diag(prod_t a_t), the GLA
    transition of the same gates."""
    inp = _kda_inputs(23, 5, seed=161)
    inp.beta = torch.zeros_like(inp.beta)
    S, T = run_build(inp)
    assert np.all(S == 0)
    diag = synth.make_inputs("diag", 1, 2, 5, [23], torch.float64, seed=161)
    diag.log_gate = inp.log_gate
    _, T_diag = run_build(diag)
    np.testing.assert_allclose(T, T_diag, rtol=1e-13, atol=0)


def test_kda_retrieves_last_write_so_the_gate_comes_first():
    """b_L = 1, |k_L| = 1: k_L^T S = v_L^T and k_L^T T = 0 whatever the decays, which holds only
    with the decay applied before the delta update, (I - k k^T) Diag(a), not after it."""
    inp = _kda_inputs(6, 4, seed=162)
    kl = np.array([0.6, 0.0, -0.8, 0.0])
    inp.k[-1, 0] = torch.from_numpy(kl)
    inp.beta[-1, :] = 1.0
    S, T = run_build(inp)
    for h in range(2):
        np.testing.assert_allclose(kl @ S[0, h], f64(inp.v)[-1, h], atol=1e-14)
        np.testing.assert_allclose(kl @ T[0, h], np.zeros(4), atol=1e-15)


def test_kda_det_invariant():
    """det T = prod_t (1 - b_t |k_t|^2) prod_i a_t[i]."""
    inp = synth.make_inputs("kda", 1, 1, 6, [11], torch.float64, seed=163, l2norm_k=False,
                            k_scale=0.5, alpha_scale=0.3)
    S, T = run_build(inp)
    k, b = f64(inp.k)[:, 0], f64(inp.beta)[:, 0]
    sign, logdet = np.linalg.slogdet(T[0, 0])
    expect = f64(inp.log_gate)[:, 0].sum() + np.sum(np.log(np.abs(1 - b * (k * k).sum(1))))
    assert sign == np.prod(np.sign(1 - b * (k * k).sum(1)))
    assert logdet == pytest.approx(expect, rel=1e-12, abs=1e-12)


def test_kda_T_is_the_jacobian_and_segments_compose():
    inp = synth.make_inputs("kda", 1, 2, 8, [30, 0, 17], torch.float64, seed=164, alpha_scale=0.3)
    S, T = run_build(inp)
    seq = run_seq(inp)
    np.testing.assert_allclose(oracle.compose_scan(T, S), seq, rtol=1e-11, atol=1e-12)
    S0 = np.random.default_rng(1).standard_normal((2, 8, 8))
    with_s0 = run_seq(inp, S0=S0)
    np.testing.assert_allclose(with_s0[-1] - seq[-1], np.einsum("hij,hjk->hik", T[2] @ T[1] @ T[0], S0),
                               rtol=1e-10, atol=1e-12)


# ------------------------------------------------------------------ segment outputs o_t = S_t^T q_t

def _with_q(family, lens, d=6, seed=170, **kw):
    return synth.make_inputs(family, 2, 4, d, lens, torch.float64, seed=seed, with_q=True, **kw)


def run_out(inp, S_init=None):
    return oracle.outputs(inp.family, inp.seg_offsets, f64(inp.k), f64(inp.v), f64(inp.q),
                          f64(inp.log_gate), f64(inp.log_gamma), f64(inp.beta), S_init=S_init)


def test_outputs_linear_closed_form():
    """Plain linear attention: o_t = sum_{s <= t in the segment} (q_t . k_s) v_s."""
    inp = _with_q("linear", [9, 0, 5])
    O = run_out(inp)
    k, v, q = f64(inp.k), f64(inp.v), f64(inp.q)
    for j in range(inp.n_seg):
        a, b = inp.seg_offsets[j], inp.seg_offsets[j + 1]
        for t in range(a, b):
            for h in range(4):
                hk = h // 2
                ref = sum((q[t, hk] @ k[s, hk]) * v[s, h] for s in range(a, t + 1))
                np.testing.assert_allclose(O[t, h], ref, rtol=1e-12, atol=1e-14)


def test_outputs_scalar_decay_closed_form():
    """RetNet: o_t = sum_{s <= t} gamma^(t - s) (q_t . k_s) v_s within the segment."""
    inp = _with_q("scalar", [12, 7])
    O = run_out(inp)
    k, v, q, lg = f64(inp.k), f64(inp.v), f64(inp.q), f64(inp.log_gamma)
    for j in range(inp.n_seg):
        a, b = inp.seg_offsets[j], inp.seg_offsets[j + 1]
        for t in range(a, b):
            for h in range(4):
                ref = sum(np.exp((t - s) * lg[h]) * (q[t, h // 2] @ k[s, h // 2]) * v[s, h]
                          for s in range(a, t + 1))
                np.testing.assert_allclose(O[t, h], ref, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("family", ["linear", "scalar", "diag", "delta", "gdn", "kda"])
def test_last_output_reads_the_end_state(family):
    """The output of a segment's last token is S(C|0)^T q_L, with S(C|0) from the build."""
    inp = _with_q(family, [13, 1, 8], alpha_scale=0.3, gla_div=4.0)
    O = run_out(inp)
    S, _ = run_build(inp, want_T=False)
    q = f64(inp.q)
    for j in range(inp.n_seg):
        t = inp.seg_offsets[j + 1] - 1
        for h in range(4):
            np.testing.assert_allclose(O[t, h], S[j, h].T @ q[t, h // 2], rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("family", ["linear", "scalar", "diag", "delta", "gdn", "kda"])
def test_outputs_after_a_prefix_state_are_corrected_by_the_transition(family):
    """Starting a segment from a prefix state S0 adds (T_{<=t} S0)^T q_t to every output,
    T_{<=t} the transition of the segment's tokens up to t (the build's T of the prefix of the
    segment that ends at t)."""
    L = 10
    inp = _with_q(family, [L], alpha_scale=0.3, gla_div=4.0)
    S0 = np.random.default_rng(2).standard_normal((1, 4, 6, 6))
    dO = run_out(inp, S_init=S0) - run_out(inp)
    q = f64(inp.q)
    for t in range(L):
        part = synth.make_inputs(family, 2, 4, 6, [t + 1], torch.float64, seed=170, with_q=True,
                                 alpha_scale=0.3, gla_div=4.0)
        for n in ("k", "v", "q", "log_gate", "beta"):
            if getattr(inp, n) is not None:
                setattr(part, n, getattr(inp, n)[: t + 1])
        part.log_gamma = inp.log_gamma
        _, T = run_build(part)
        for h in range(4):
            np.testing.assert_allclose(dO[t, h], (T[0, h] @ S0[0, h]).T @ q[t, h // 2],
                                       rtol=1e-10, atol=1e-12)


# ------------------------------------------------------------------ convolution-state warm-up

def _conv_case(family, lens, K, seed, d=6, H_k=1, H_v=2):
    rng = np.random.default_rng(seed)
    inp = synth.make_inputs(family, H_k, H_v, d, lens, torch.float64, seed=seed, alpha_scale=0.3,
                            gla_div=4.0, k_scale=0.7)
    k_raw, v_raw = inp.k.numpy(), inp.v.numpy()
    wk = rng.standard_normal((H_k * d, K)) * 0.6
    wv = rng.standard_normal((H_v * d, K)) * 0.6
    f = lambda t: None if t is None else t.numpy()
    return inp, k_raw, v_raw, wk, wv, f(inp.log_gate), f(inp.log_gamma), f(inp.beta)


def _segment_local_conv(x, w, offs, normalize):
    """Each segment convolved on its own (zeros before its first token): the values a cached
    segment was built from."""
    return np.concatenate([oracle.short_conv(x[offs[j]:offs[j + 1]], w, normalize=normalize)
                           for j in range(len(offs) - 1)])


def test_short_conv_is_numpy_convolve_then_silu():
    rng = np.random.default_rng(170)
    x = rng.standard_normal((11, 2, 3))
    w = rng.standard_normal((6, 4))
    y = oracle.short_conv(x, w)
    for h in range(2):
        for c in range(3):
            ref = np.convolve(x[:, h, c], w[h * 3 + c, ::-1])[:11]
            np.testing.assert_allclose(y[:, h, c], ref / (1 + np.exp(-ref)), rtol=1e-13, atol=1e-14)
    yn = oracle.short_conv(x, w, normalize=True)
    np.testing.assert_allclose(np.linalg.norm(yn, axis=2), 1.0, rtol=1e-13)
    np.testing.assert_allclose(oracle.short_conv(x, w, 4, 9), y[4:9], rtol=0, atol=0)


@pytest.mark.parametrize("family", ["linear", "scalar", "diag", "delta", "gdn", "kda"])
@pytest.mark.parametrize("K", [2, 4])
def test_conv_warmup_is_recomputation_of_the_whole_prompt(family, K):
    """The defining property: each segment's entry from its cached rest plus the head rebuilt
    in context equals the entry built from the whole prompt convolved in one pass (segments of
    length 0, 1 and below K - 1 included)."""
    lens = [9, 1, 0, 2, 7, 12]
    inp, k_raw, v_raw, wk, wv, lg, lgam, beta = _conv_case(family, lens, K, seed=171 + K)
    offs = inp.seg_offsets
    delta = family in oracle.DELTA_FAMILIES
    # the cached rests: each segment convolved alone, its tokens from the head length on
    kl = _segment_local_conv(k_raw, wk, offs, delta)
    vl = _segment_local_conv(v_raw, wv, offs, False)
    hl = oracle.head_lengths(offs, K)
    rest = [(int(offs[j] + hl[j]), int(offs[j + 1])) for j in range(len(lens))]
    keep = np.concatenate([np.arange(a, b) for a, b in rest]).astype(np.int64)
    r_offs = np.concatenate([[0], np.cumsum([b - a for a, b in rest])]).astype(np.int64)
    g = lambda a: None if a is None else a[keep]
    S_r, T_r = oracle.build_segments(family, r_offs, kl[keep], vl[keep], g(lg), lgam, g(beta))
    # (lam, P) of the rests as the library stores them: here lam = 0 and P = T (any pair with
    # exp(lam) P = T is an entry)
    d = v_raw.shape[2]
    if family in ("delta", "gdn", "kda"):
        lam_r, P_r = np.zeros(S_r.shape[:2]), T_r
    elif family == "diag":
        lam_r, P_r = np.log(np.diagonal(T_r, axis1=2, axis2=3)), None
    elif family == "scalar":
        lam_r, P_r = np.log(T_r[:, :, 0, 0]), None
    else:
        lam_r, P_r = np.zeros(S_r.shape[:2]), None
    S, T = oracle.conv_warmup(family, offs, k_raw, v_raw, wk, wv, K, S_r, lam_r, P_r, lg, lgam, beta)
    kf = oracle.short_conv(k_raw, wk, normalize=delta)
    vf = oracle.short_conv(v_raw, wv)
    S_w, T_w = oracle.build_segments(family, offs, kf, vf, lg, lgam, beta)
    np.testing.assert_allclose(S, S_w, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(T, T_w, rtol=1e-10, atol=1e-12)
    # the pin is sensitive to the window: segment-local heads (a zero convolution state) differ
    S_0, _ = oracle.build_segments(family, offs, kl, vl, lg, lgam, beta)
    assert max(np.abs(S_0[j] - S_w[j]).max() for j in (3, 4, 5)) > 1e-3


def test_conv_warmup_without_window_is_the_rest():
    """K = 1: no token sees another, the heads are empty and the entry is the cached one."""
    inp, k_raw, v_raw, wk, wv, lg, lgam, beta = _conv_case("gdn", [5, 3], 1, seed=175)
    S_r = np.random.default_rng(1).standard_normal((2, 2, 6, 6))
    P_r = np.random.default_rng(2).standard_normal((2, 2, 6, 6))
    lam_r = np.full((2, 2), -0.5)
    S, T = oracle.conv_warmup("gdn", inp.seg_offsets, k_raw, v_raw, wk, wv, 1, S_r, lam_r, P_r, lg,
                              lgam, beta)
    np.testing.assert_allclose(S, S_r, rtol=0, atol=0)
    np.testing.assert_allclose(T, np.exp(-0.5) * P_r, rtol=1e-15)
