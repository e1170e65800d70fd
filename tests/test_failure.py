"""The device-detected failures reach the host as a status, and the library stays usable
after them (needs a GPU). Neither case faults, traps or leaves a kernel waiting:

- a gate outside the supported range is plain input data (a GDN chunk whose log-decay sum is
  below -60): the tensor-core build reports HYPIC_ERR_RANGE;
- a bounded wait that runs out is made by the library's wait probe, whose CTAs wait on a
  barrier that nothing arrives at for a few microseconds, with the same wait and abort code
  as the kernels: the status is HYPIC_ERR_TIMEOUT, and the CTAs free their tensor memory.

After each, the next build of a reference input is bitwise identical to the build taken
before, with a clean status.
"""
import time

import numpy as np
import pytest
import torch

from linear_attention_state_gdn_gb300 import synth
from tests.helpers import to_dev

pytestmark = pytest.mark.gpu

HYPIC_ERR_RANGE = 4
HYPIC_ERR_TIMEOUT = 6


def _hy():
    import linear_attention_state_gdn_gb300 as hy
    return hy


def _reference_build():
    """A build over more (segment, head) units than SMs, so that its CTAs run on every SM
    (each allocates all of an SM's tensor memory)."""
    hy = _hy()
    lens = [int(x) for x in np.random.default_rng(81).integers(64, 257, size=96)]
    inp = synth.make_inputs("gdn", 2, 4, 128, lens, torch.bfloat16, seed=82, alpha_scale=0.05)
    d = to_dev(inp)

    def run():
        out = hy.hypic_build_segments("gdn", d["k"], d["v"], inp.seg_offsets,
                                      log_gate=d["log_gate"], beta=d["beta"])
        st = hy.hypic_get_device_status()
        return out, st
    return run


def test_gate_out_of_range_reports_range_status():
    hy = _hy()
    ref_run = _reference_build()
    (S0, l0, P0), st = ref_run()
    assert st == 0
    inp = synth.make_inputs("gdn", 1, 2, 128, [200, 64, 130], torch.bfloat16, seed=83, alpha_scale=0.05)
    lg = inp.log_gate.clone()
    lg[200:264] = -1.25          # the second segment's only chunk: log-decay sum -80 < -60
    d = to_dev(inp)
    hy.hypic_build_segments("gdn", d["k"], d["v"], inp.seg_offsets, log_gate=lg.cuda(),
                            beta=d["beta"])
    assert hy.hypic_get_device_status() == HYPIC_ERR_RANGE
    assert hy.hypic_get_device_status() == 0      # read and cleared
    (S1, l1, P1), st = ref_run()
    assert st == 0
    assert torch.equal(S0, S1) and torch.equal(P0, P1) and torch.equal(l0, l1)


def test_kda_channel_gate_out_of_range_reports_range_status():
    """KDA: one key channel of one chunk decays below -60 (the others stay in range)."""
    hy = _hy()
    inp = synth.make_inputs("kda", 1, 2, 128, [200, 64, 130], torch.bfloat16, seed=85, alpha_scale=0.05)
    lg = inp.log_gate.clone()
    lg[200:264, 1, 17] = -1.25
    d = to_dev(inp)
    hy.hypic_build_segments("kda", d["k"], d["v"], inp.seg_offsets, log_gate=lg.cuda(), beta=d["beta"])
    assert hy.hypic_get_device_status() == HYPIC_ERR_RANGE
    hy.hypic_build_segments("kda", d["k"], d["v"], inp.seg_offsets, log_gate=d["log_gate"], beta=d["beta"])
    assert hy.hypic_get_device_status() == 0


def test_exact_path_has_no_gate_range_limit():
    """The exact fp32 path steps token by token in fp32 and has no chunk log-decay limit."""
    hy = _hy()
    inp = synth.make_inputs("gdn", 1, 2, 64, [200, 64], torch.float32, seed=84, alpha_scale=0.05)
    lg = inp.log_gate.clone()
    lg[200:264] = -1.25
    d = to_dev(inp)
    hy.hypic_build_segments("gdn", d["k"], d["v"], inp.seg_offsets, log_gate=lg.cuda(),
                            beta=d["beta"])
    assert hy.hypic_get_device_status() == 0


def test_bounded_wait_runs_out_and_reports_timeout():
    hy = _hy()
    ref_run = _reference_build()
    (S0, l0, P0), st = ref_run()
    assert st == 0
    t0 = time.perf_counter()
    hy.hypic_probe_wait_timeout(20)
    st = hy.hypic_get_device_status()
    dt = time.perf_counter() - t0
    assert st == HYPIC_ERR_TIMEOUT
    # the second wait gave up on the abort flag instead of sitting out its own 2 s limit
    assert dt < 1.5, dt
    assert hy.hypic_get_device_status() == 0      # read and cleared
    # every SM's tensor memory was freed: the reference build allocates all of it again
    (S1, l1, P1), st = ref_run()
    assert st == 0
    assert torch.equal(S0, S1) and torch.equal(P0, P1) and torch.equal(l0, l1)
