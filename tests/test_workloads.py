"""The synthetic workload recipes (CPU only): shapes, tree constraints, and the
planted acceptance depth, which the oracle's greedy acceptance must recover."""
import numpy as np
import pytest

import workloads as W


def depths(par):
    d = np.zeros(len(par), int)
    for i in range(1, len(par)):
        d[i] = d[par[i]] + 1
    return d


@pytest.mark.parametrize("name", list(W.SPECS))
def test_tree_shapes(name):
    spec = W.SPECS[name]
    w = W.make(name, parts=(), B=min(spec.B, 8))
    par = w["parents"]
    assert par.shape == (min(spec.B, 8), spec.N)
    for row in par:
        assert row[0] == -1 and all(0 <= row[i] < i for i in range(1, spec.N))
        dep = depths(row)
        if spec.tree in ("random", "eagle2"):
            assert dep.max() <= spec.depth
            assert np.bincount(row[1:]).max() <= spec.branch
        assert all(dep[i] >= dep[i - 1] for i in range(1, spec.N))   # breadth-first labels
    if spec.tree == "chain":
        assert (par == np.arange(-1, spec.N - 1)).all()
    bt = w["block_table"]
    used = bt[bt >= 0]
    assert len(np.unique(used)) == len(used) == w["num_blocks"]


@pytest.mark.parametrize("name", ["tiny_fp32", "llama3_8b_tree60", "llama3_8b_b32_tree26",
                                  "qwen2_7b_32k_tree63"])
def test_planted_acceptance_is_recovered(orc, name):
    spec = W.SPECS[name]
    w = W.make(name, parts=("accept",), B=min(spec.B, 6), V=min(spec.V, 4096))
    mp = W.max_path_len(w["parents"])
    acc, path, out, st = orc.accept_greedy(w["parents"], w["draft_tokens"], w["logits"], mp)
    assert (st == 0).all()
    assert (acc == w["planted_accept_len"]).all()


def test_stochastic_inputs_are_distributions():
    w = W.make("llama3_8b_b128_chain5", parts=("accept",), B=3, V=2000)
    for x in (w["p"], w["q_probs"]):
        assert x.dtype == np.float32 and (x >= 0).all()
        np.testing.assert_allclose(x.sum(-1), 1.0, rtol=1e-4)
    tok = w["draft_tokens"]
    assert (w["q_probs"][np.arange(3)[:, None], np.arange(1, 6)[None], tok[:, 1:]] > 0).all()


def test_bf16_rounding_round_trip():
    x = np.array([1.0, 1.00390625, 1.0078125, -2.5, 3.1415927, 1e-30], np.float32)
    b = W.f32_to_bf16_bits(x)
    y = W.bf16_bits_to_f32(b)
    assert y[0] == 1.0 and y[1] == 1.0 and y[2] == 1.0078125 and y[3] == -2.5
    assert abs(y[4] - 3.140625) < 1e-7
    assert (W.f32_to_bf16_bits(y) == b).all()
