"""Oracle pins for batches whose trees have fewer nodes than the batch's N
(ragged node counts; "P-EAGLE in vLLM", practice 5: shapes are kept fixed so
that CUDA graphs stay valid, and a smaller tree occupies the first counts[b]
of the N node slots).

A ragged batch is B independent problems: sequence b with counts[b] = c must
give exactly what the dense oracle gives on the batch cut to its first c
nodes (so every sequence keeps its batch index, and with it its random draw
keys), and its absent nodes must get the defined outputs (no mask bits,
depth -1, zero attention output, never accepted, nothing appended).  The
dense functions are pinned independently (test_oracle_*.py); these pins
catch a count that is ignored, or that one step reads N where it should read
counts[b] (key range, chain length, draw index, token checks).  Anything
written into the absent slots (bad parents, out-of-range tokens, NaN logits)
must change nothing.
"""
import numpy as np
import pytest

import workloads as W

N = 12


def ragged_trees(rng, B, counts):
    """Random trees filling counts[b] slots; absent slots hold junk."""
    par = np.full((B, N), 99, np.int32)                 # junk in absent slots
    for b in range(B):
        par[b, 0] = -1
        for i in range(1, counts[b]):
            par[b, i] = int(rng.integers(0, i))
    return par


def batch(seed=0, B=9):
    rng = np.random.default_rng(seed)
    counts = np.array([1, 2, 3, 5, 7, N, 4, 7, N][:B], np.int32)
    return rng, counts, ragged_trees(rng, B, counts)


def test_mask_ragged_equals_dense_cut(orc):
    rng, counts, par = batch()
    mask, depth, st = orc.tree_mask(par, counts)
    assert (st == 0).all()
    for c in np.unique(counts):
        rows = counts == c
        m, d, s = orc.tree_mask(par[rows, :c])
        assert (s == 0).all()
        assert np.array_equal(mask[rows, :c], m) and np.array_equal(depth[rows, :c], d)
        assert (mask[rows, c:] == 0).all() and (depth[rows, c:] == -1).all()
    # a present node's bits never reach the absent slots
    for b in range(len(counts)):
        assert (mask[b, :counts[b]] >> np.uint64(counts[b]) == 0).all()


def test_counts_outside_range_are_out_of_range(orc):
    rng, counts, par = batch()
    bad = counts.copy()
    bad[1], bad[4] = 0, N + 1
    mask, depth, st = orc.tree_mask(par, bad)
    assert st[1] == orc.OUT_OF_RANGE and st[4] == orc.OUT_OF_RANGE
    assert (mask[[1, 4]] == 0).all() and (depth[[1, 4]] == -1).all()
    others = np.ones(len(counts), bool)
    others[[1, 4]] = False
    assert (st[others] == 0).all()


def test_attention_ragged_equals_dense_cut(orc):
    rng, counts, par = batch(1)
    spec = W.Spec("ragged", B=len(counts), P_lo=0, P_hi=90, Hq=4, Hkv=2, d=16, V=8, N=N,
                  tree="random", depth=3, branch=2, bs=16, bf16=False, seed=3)
    w = W.make(spec, parts=("attn",))
    w["parents"] = par
    mask, _, _ = orc.tree_mask(par, counts)
    out, st = orc.attention(w["q"], w["k_cache"], w["v_cache"], w["block_table"],
                            w["prefix_lens"], mask, bf16=False, counts=counts)
    assert (st == 0).all()
    out = out.reshape(len(counts), N, spec.Hq, spec.d)
    for c in np.unique(counts):
        rows = np.flatnonzero(counts == c)
        m, _, _ = orc.tree_mask(par[rows, :c])
        ref, rst = orc.attention(w["q"][rows, :c], w["k_cache"], w["v_cache"],
                                 w["block_table"][rows], w["prefix_lens"][rows], m, bf16=False)
        assert (rst == 0).all()
        assert np.array_equal(out[rows, :c], ref.reshape(len(rows), c, spec.Hq, spec.d))
        assert (out[rows, c:] == 0).all()


def test_attention_ragged_reads_only_present_keys(orc):
    """K/V rows of absent tree slots (positions P + c .. P + N - 1) may hold
    anything, and their blocks need not exist: both change nothing."""
    rng, counts, par = batch(2)
    spec = W.Spec("ragged2", B=len(counts), P_lo=5, P_hi=70, Hq=2, Hkv=1, d=16, V=8, N=N,
                  tree="random", depth=3, branch=2, bs=16, bf16=False, seed=4)
    w = W.make(spec, parts=("attn",))
    mask, _, _ = orc.tree_mask(par, counts)
    kw = dict(bf16=False, counts=counts)
    base, _ = orc.attention(w["q"], w["k_cache"], w["v_cache"], w["block_table"],
                            w["prefix_lens"], mask, **kw)
    k2, v2, bt2 = w["k_cache"].copy(), w["v_cache"].copy(), w["block_table"].copy()
    for b in range(len(counts)):
        P = int(w["prefix_lens"][b])
        for t in range(P + counts[b], P + N):
            blk = bt2[b, t // spec.bs]
            k2[blk, :, t % spec.bs] = np.nan
            v2[blk, :, t % spec.bs] = np.nan
        first_absent_block = (P + counts[b] + spec.bs - 1) // spec.bs
        bt2[b, first_absent_block:] = -1                 # blocks past the tree: none
    got, st = orc.attention(w["q"], k2, v2, bt2, w["prefix_lens"], mask, **kw)
    assert (st == 0).all()
    assert np.array_equal(got, base)
    # mask bits at or above counts[b] (absent slots) are never read
    junk = mask.copy()
    for b in range(len(counts)):
        high = np.uint64(((1 << N) - 1) & ~((1 << int(counts[b])) - 1))
        junk[b] |= high
    got, st = orc.attention(w["q"], w["k_cache"], w["v_cache"], w["block_table"],
                            w["prefix_lens"], junk, **kw)
    assert (st == 0).all()
    assert np.array_equal(got, base)


def _greedy_inputs(rng, counts, par, V=50):
    B = len(counts)
    logits = rng.integers(-3, 3, size=(B, N, V)).astype(np.float32)
    tok = rng.integers(0, V, size=(B, N)).astype(np.int32)
    am = np.argmax(logits, axis=2)
    for b in range(B):
        for c in range(1, counts[b]):
            if rng.random() < 0.7:
                tok[b, c] = am[b, par[b, c]]
    return logits, tok


def test_greedy_ragged_equals_dense_cut_and_ignores_absent_slots(orc):
    rng, counts, par = batch(3)
    logits, tok = _greedy_inputs(rng, counts, par)
    mp = N
    got = orc.accept_greedy(par, tok, logits, mp, counts=counts)
    assert (got[3] == 0).all() and got[0].max() > 0
    for c in np.unique(counts):
        rows = counts == c
        ref = orc.accept_greedy(par[rows, :c], tok[rows, :c], logits[rows, :c], mp)
        for g, r in zip(got, ref):
            assert np.array_equal(g[rows], r)
    # junk in the absent slots: out-of-range tokens, NaN rows, bad parents
    tok2, lg2, par2 = tok.copy(), logits.copy(), par.copy()
    for b in range(len(counts)):
        tok2[b, counts[b]:] = -5
        lg2[b, counts[b]:] = np.nan
        par2[b, counts[b]:] = 1000
    again = orc.accept_greedy(par2, tok2, lg2, mp, counts=counts)
    for g, r in zip(again, got):
        assert np.array_equal(g, r)


@pytest.mark.parametrize("chain", [True, False])
def test_stochastic_ragged_equals_dense_cut(orc, chain):
    """Chains (the chain rule: K = counts[b] - 1 tests, then a draw keyed by
    counts[b]) and branching trees (their rule, with counts[b] in place of N
    in the draw indices)."""
    rng = np.random.default_rng(4)
    counts = np.array([1, 2, 4, 7, N, 3, N, 6], np.int32)
    B, V = len(counts), 16
    if chain:
        par = np.tile(np.arange(-1, N - 1, dtype=np.int32), (B, 1))
    else:
        par = ragged_trees(rng, B, counts)
        for b in range(B):
            par[b, counts[b]:] = np.arange(counts[b] - 1, N - 1)   # any junk
    p = rng.dirichlet(np.ones(V) * 0.7, size=(B, N)).astype(np.float32)
    q = rng.dirichlet(np.ones(V) * 0.7, size=(B, N)).astype(np.float32)
    q[:, 1:] = 0.5 * q[:, 1:] + 0.5 * p[:, :-1]                       # frequent acceptance
    tok = rng.integers(0, V, size=(B, N)).astype(np.int32)
    for seed, off in ((5, 0), (5, 9)):
        got = orc.accept_stochastic(par, tok, p, q, seed, off, N, counts=counts)
        assert (got[3] == 0).all()
        for c in np.unique(counts):
            rows = counts == c
            # the dense batch cut to c nodes keeps every sequence's index (draw key)
            ref = orc.accept_stochastic(par[:, :c], tok[:, :c], p[:, :c], q[:, :c], seed, off, N)
            for g, r in zip(got, ref):
                assert np.array_equal(g[rows], r[rows])


def test_append_ragged_writes_only_present_nodes(orc):
    rng, counts, par = batch(5)
    B, Hkv, d, bs = len(counts), 2, 8, 16
    P = rng.integers(0, 40, size=B).astype(np.int32)
    nb = [(int(x) + N + bs - 1) // bs for x in P]
    bt = np.full((B, max(nb)), -1, np.int32)
    perm = rng.permutation(sum(nb))
    o = 0
    for b in range(B):
        bt[b, :nb[b]] = perm[o:o + nb[b]]
        o += nb[b]
    kn = rng.standard_normal((B, N, Hkv, d)).astype(np.float32)
    vn = rng.standard_normal((B, N, Hkv, d)).astype(np.float32)
    _, depth, _ = orc.tree_mask(par, counts)
    kc = rng.standard_normal((sum(nb), Hkv, bs, d)).astype(np.float32)
    vc = rng.standard_normal((sum(nb), Hkv, bs, d)).astype(np.float32)
    k0, v0 = kc.copy(), vc.copy()
    st = orc.tree_kv_append(kn, vn, depth, kc, vc, bt, P, rope_theta=10000.0, counts=counts)
    assert (st == 0).all()
    for c in np.unique(counts):
        rows = np.flatnonzero(counts == c)
        kr, vr = k0.copy(), v0.copy()
        _, dc, _ = orc.tree_mask(par[rows, :c])
        s = orc.tree_kv_append(kn[rows, :c], vn[rows, :c], dc, kr, vr, bt[rows], P[rows],
                               rope_theta=10000.0)
        assert (s == 0).all()
        for b in rows:
            for t in range(P[b], P[b] + N):
                blk, r = bt[b, t // bs], t % bs
                if t < P[b] + c:
                    assert np.array_equal(kc[blk, :, r], kr[blk, :, r])
                    assert np.array_equal(vc[blk, :, r], vr[blk, :, r])
                else:
                    assert np.array_equal(kc[blk, :, r], k0[blk, :, r])   # untouched
                    assert np.array_equal(vc[blk, :, r], v0[blk, :, r])
