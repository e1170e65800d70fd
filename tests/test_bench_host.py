"""Host arithmetic of bench.py on CPU: the algorithmic work every roofline fraction divides by,
pinned to the workloads' shapes counted independently here, and the helpers the JSON line is
built from (relative Frobenius error, whole-job throughput, the traffic record's source hash).

The figures: the chunked GDN build does, per token and value head with chunks of C = 64 and
d = 128, the gram, W and U products (2 C d flop each) and the two state products X = W [S | P]
and the update (2 d (2 d) flop each); the GDN workload (32768 tokens as 16 x 2048, 16 key and 32
value heads) moves k and v in bf16, log a and b in fp32, and S, P (fp32) and lam out; the
48-layer compose (1536 units, 64 segments) reads S_j and P_j (j >= 1) and lam_j and writes the
prefix states.
"""
import os

import numpy as np
import pytest

import bench

C, D = 64, 128


def test_gdn_flop_per_token_and_value_head():
    gram = w = u = 2 * C * D
    state = 2 * D * (2 * D) + 2 * D * (2 * D)
    assert bench.GDN_FLOP_PER_TOKEN_HEAD == gram + w + u + state == 180_224


def test_gdn_workload_bytes():
    n_tok, H_k, H_v, n_seg = 32768, 16, 32, 16
    k = n_tok * H_k * D * 2
    v = n_tok * H_v * D * 2
    gates_beta = n_tok * H_v * (4 + 4)
    s_p_lam = n_seg * H_v * (D * D * 4 * 2 + 4)
    assert bench.gdn_algorithmic_bytes(n_tok, H_k, H_v, D, n_seg) == k + v + gates_beta + s_p_lam == 478_152_704


def test_compose_bytes_of_the_48_layer_workload():
    units, n_seg = 48 * 32, 64
    tile = D * D * 4
    want = units * (n_seg * tile          # S_j
                    + (n_seg - 1) * tile  # P_j, j >= 1
                    + n_seg * tile        # prefix_j
                    + n_seg * 4)          # lam_j
    assert bench.compose_algorithmic_bytes(n_seg, units, D, dense=True) == want == 19_227_082_752


def test_compose_bytes_scalar_diagonal_and_start_state():
    tile = D * D * 4
    assert bench.compose_algorithmic_bytes(8, 16, D, dense=False) == 16 * 8 * (2 * tile + 4)
    assert bench.compose_algorithmic_bytes(16, 16, D, dense=False, diag=True) == 16 * 16 * (2 * tile + 4 * D)
    # a start state S0 is read once, and with it P_0 too
    assert (bench.compose_algorithmic_bytes(4, 2, D, dense=True, s0=True)
            == 2 * (4 * (2 * tile + 4) + 4 * tile + tile))


def test_rel_frob_max():
    rng = np.random.default_rng(0)
    ref = rng.standard_normal((3, 4, 5, 5))
    got = ref.copy()
    got[2, 1] *= 1.01                       # one matrix off by 1%
    assert bench.rel_frob_max(got, ref) == pytest.approx(0.01, rel=1e-9)
    z = np.zeros((2, 3, 3))
    g = z.copy()
    g[1, 0, 0] = 0.5                        # an exactly-zero reference counts the absolute norm
    assert bench.rel_frob_max(g, z) == pytest.approx(0.5)
    assert bench.rel_frob_max(np.zeros((0, 2, 2)), np.zeros((0, 2, 2))) == 0.0


def test_aggregate_throughput_counts_every_rank_over_the_slowest_time():
    assert bench.aggregate_throughput(1000.0, 2.0, 4) == pytest.approx(2000.0)


def test_src_hash_ignores_comments_and_blank_lines(tmp_path, monkeypatch):
    csrc = tmp_path / "linear_attention_state_gdn_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "a.cu").write_text("int x = 1;  // one\n\n/* block\n comment */int y = 2;\n")
    (csrc / "b.cu").write_text("int x = 1;\nint y = 2;\n")
    (csrc / "c.cu").write_text("int x = 1;\nint y = 3;\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.src_hash("a.cu") == bench.src_hash("b.cu")
    assert bench.src_hash("b.cu") != bench.src_hash("c.cu")


def test_recorded_traffic_is_none_for_other_sources(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    csrc = tmp_path / "linear_attention_state_gdn_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text("int k;\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    import json
    h = bench.src_hash("k.cu")
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({"kern": {"src": h, "bytes_per_launch": 7}}))
    assert bench.recorded_traffic("kern", ["k.cu"]) == 7
    (csrc / "k.cu").write_text("int k2;\n")           # the kernel changed since the capture
    assert bench.recorded_traffic("kern", ["k.cu"]) is None
    assert bench.recorded_traffic("other", ["k.cu"]) is None
    os.remove(tmp_path / "profiles" / "traffic.json")
    assert bench.recorded_traffic("kern", ["k.cu"]) is None
