"""hypic_build_segments_static_ws (library-owned device scratch, no per-call allocation)
against hypic_build_segments with a caller workspace: two calls in a row, bit for bit.

Kept in its own module, collected last, so it also runs after every other GPU test has
used the library in the same process."""
import pytest
import torch

from linear_attention_state_gdn_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("family", ["gdn", "delta"])
def test_static_workspace_build_matches_the_workspace_build(family):
    import linear_attention_state_gdn_gb300 as hy
    inp = synth.make_inputs(family, 2, 4, 128, [300, 70, 130], torch.bfloat16, seed=77)
    d = {n: t.cuda() for n, t in inp.tensors().items()}
    kw = dict(log_gate=d.get("log_gate"), beta=d.get("beta"))
    assert hy.hypic_build_workspace_bytes(family, d["k"], d["v"], inp.seg_offsets, **kw) > 0
    ref = hy.hypic_build_segments(family, d["k"], d["v"], inp.seg_offsets, **kw)
    torch.cuda.synchronize()
    assert hy.hypic_get_device_status() == 0
    for _ in range(2):
        got = hy.hypic_build_segments_static_ws(family, d["k"], d["v"], inp.seg_offsets, **kw)
        torch.cuda.synchronize()
        assert hy.hypic_get_device_status() == 0
        for r, g in zip(ref, got):
            assert torch.equal(r, g)
