"""The debug-bounds build (HYPIC_DEBUG_BOUNDS: index checks compiled into the kernels, in place
of a memory checker) runs the tensor-core and exact builds and the composes of small ragged
cases with a clean device status and the same results as the release library (needs a GPU).

The debug library runs in a child process (the binding loads one library per process); both
processes draw the same seeded inputs."""
import os
import subprocess
import sys

import pytest
import torch

from linear_attention_state_gdn_gb300 import synth

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CASES = [("gdn", torch.bfloat16, 128), ("kda", torch.bfloat16, 128), ("scalar", torch.bfloat16, 128),
         ("diag", torch.bfloat16, 128), ("gdn", torch.float32, 64), ("kda", torch.float32, 32)]
LENS = [200, 64, 1, 0, 129, 300, 63]


def run_cases(out_path):
    """Every case through the library this process loaded: (S, lam, P, prefix) and the status."""
    import linear_attention_state_gdn_gb300 as hy
    res = {}
    for fam, dt, d in CASES:
        inp = synth.make_inputs(fam, 2, 4, d, LENS, dt, seed=70 + d, alpha_scale=0.05, gla_div=8.0)
        dev = {n: t.cuda() for n, t in inp.tensors().items()}
        S, lam, P = hy.hypic_build_segments(fam, dev["k"], dev["v"], inp.seg_offsets,
                                            log_gate=dev.get("log_gate"), log_gamma=dev.get("log_gamma"),
                                            beta=dev.get("beta"))
        pref = hy.hypic_compose_scan(fam, S, lam, P)
        st = hy.hypic_get_device_status()
        res[f"{fam}_{d}_{dt}"] = (st, S.cpu(), lam.cpu(), None if P is None else P.cpu(), pref.cpu())
    torch.save(res, out_path)


def test_debug_bounds_build_matches_release(tmp_path):
    from linear_attention_state_gdn_gb300 import _build
    lib = _build.build(debug_bounds=True)
    rel = tmp_path / "release.pt"
    dbg = tmp_path / "debug.pt"
    run_cases(rel)
    code = (f"import sys; sys.path.insert(0, {ROOT!r}); "
            f"from tests.test_debug_bounds import run_cases; run_cases({str(dbg)!r})")
    env = dict(os.environ, HYPIC_LIBRARY=lib)
    subprocess.run([sys.executable, "-c", code], env=env, check=True, cwd=ROOT, timeout=600)
    a, b = torch.load(rel), torch.load(dbg)
    for key in a:
        assert a[key][0] == 0 and b[key][0] == 0, (key, a[key][0], b[key][0])
        for x, y in zip(a[key][1:], b[key][1:]):
            if x is not None:
                assert torch.equal(x, y), key
