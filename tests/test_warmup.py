"""Convolution-state warm-up on the GPU against the oracle's recomputation of the whole prompt
(needs a GPU).

Each case draws a prompt's raw keys and values and the short convolution's taps, builds every
segment's rest (its tokens from min(K - 1, length) on, convolved within the segment, as a cache
of a convolutional layer holds them) with the library's build, runs the warm-up, and compares
each segment's entry in context with the oracle's entry of the same segment built from the
whole prompt convolved in one pass: relative Frobenius error <= 1e-4 (fp32 inputs), 2e-2 (bf16
inputs), on S and on T = exp(lam) P. The cached rests, which the composition reads in place,
must come back bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_state_gdn_gb300 import synth
from tests.helpers import TOL, assert_close, f64, gpu_T

pytestmark = pytest.mark.gpu

LENS = [200, 1, 0, 3, 129, 70, 2]


def _hy():
    import linear_attention_state_gdn_gb300 as hy
    return hy


def _case(family, dtype, d, K, lens, seed):
    hy = _hy()
    inp = synth.make_inputs(family, 2, 4, d, lens, dtype, seed=seed, alpha_scale=0.05, gla_div=8.0)
    rng = np.random.default_rng(seed)
    wk = (rng.standard_normal((2 * d, K)) * 0.5).astype(np.float32)
    wv = (rng.standard_normal((4 * d, K)) * 0.5).astype(np.float32)
    offs = inp.seg_offsets
    delta = family in oracle.DELTA_FAMILIES
    k_raw, v_raw = f64(inp.k), f64(inp.v)
    lg = f64(inp.log_gate)
    lgam = f64(inp.log_gamma)
    beta = f64(inp.beta)
    # the rests: each segment convolved alone, its tokens from the head length on
    hl = oracle.head_lengths(offs, K)
    kl = np.concatenate([oracle.short_conv(k_raw[offs[j]:offs[j + 1]], wk, normalize=delta)
                         for j in range(len(lens))])
    vl = np.concatenate([oracle.short_conv(v_raw[offs[j]:offs[j + 1]], wv) for j in range(len(lens))])
    keep = np.concatenate([np.arange(offs[j] + hl[j], offs[j + 1]) for j in range(len(lens))]).astype(np.int64)
    r_offs = np.concatenate([[0], np.cumsum([offs[j + 1] - offs[j] - hl[j] for j in range(len(lens))])])
    dev = lambda a, dt=torch.float32: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(dt).cuda()
    S_r, lam_r, P_r = hy.hypic_build_segments(
        family, dev(kl[keep], dtype), dev(vl[keep], dtype), r_offs,
        log_gate=None if lg is None else dev(lg[keep]), log_gamma=dev(lgam),
        beta=None if beta is None else dev(beta[keep]))
    rests = [None if t is None else t.clone() for t in (S_r, lam_r, P_r)]
    S, lam, P = hy.hypic_conv_warmup(
        family, offs, inp.k.cuda(), inp.v.cuda(), dev(wk), dev(wv), S_r, lam_r, P_r,
        log_gate=dev(lg), log_gamma=dev(lgam), beta=dev(beta))
    torch.cuda.synchronize()
    assert hy.hypic_get_device_status() == 0
    # the cached rests are read where they are and left as they were
    for before, after in zip(rests, (S_r, lam_r, P_r)):
        assert before is None or torch.equal(before, after)
    # the oracle: the whole prompt convolved in one pass, every segment built from it
    kf = oracle.short_conv(k_raw, wk, normalize=delta)
    vf = oracle.short_conv(v_raw, wv)
    S_w, T_w = oracle.build_segments(family, offs, kf, vf, lg, lgam, beta)
    tol = TOL[dtype]
    assert_close(f64(S), S_w, tol, "S in context")
    assert_close(gpu_T(family, lam, P, d), T_w, tol, "T in context")
    return S, lam, P


@pytest.mark.parametrize("family", ["linear", "scalar", "diag", "delta", "gdn", "kda"])
@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.float32, 64)])
def test_conv_warmup_matches_whole_prompt_recomputation(family, dtype, d):
    _case(family, dtype, d, 4, LENS, seed=180 + d)


@pytest.mark.parametrize("K", [1, 2, 8])
def test_conv_warmup_widths(K):
    """K = 1 (empty heads: the entries are the rests), 2 and the widest supported, 8 (heads of
    up to seven tokens, longer than some segments)."""
    _case("gdn", torch.float32, 32, K, LENS, seed=190 + K)


def test_conv_warmup_many_segments_one_launch():
    """Sixteen equal segments of 256 tokens in one call (every head of three tokens reaches
    into the segment before)."""
    _case("gdn", torch.bfloat16, 128, 4, [256] * 16, seed=195)
