"""Pins for the oracle's acceptance step (CPU only).

Greedy ("P-EAGLE in vLLM", 技术原理和实现方式 step 4: keep drafts while they
verify, truncate at the first rejection; "vLLM EAGLE in practice", 无损性保障:
greedy speculative decoding equals greedy decoding).  Pinned by enumerating
every root path with numpy's nanargmax (lowest index on ties, NaN skipped)
and by a hand-worked fixture.

Stochastic (same sections: rejection sampling converges to the target
distribution).  Pinned by the Philox4x32-10 known-answer vectors of its
published definition, by the empirical distribution of the emitted tokens, by
degenerate draft/target pairs, and by an exhaustive check of the integer CDF
sampler's interval boundaries.
"""
import os

import numpy as np
import pytest
from scipy import stats

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------
# greedy
# ---------------------------------------------------------------------------

def brute_force_greedy(par, tok, logits, max_path):
    N = len(par)
    best = []
    for r in range(N):
        row = logits[r]
        best.append(-1 if np.isnan(row).all() else int(np.nanargmax(row)))
    # enumerate each node's root path; accepted iff every edge matches
    candidates = []
    for c in range(N):
        chain = [c]
        while par[chain[-1]] >= 0:
            chain.append(par[chain[-1]])
        chain = chain[::-1]
        if all(tok[chain[k]] == best[chain[k - 1]] for k in range(1, len(chain))):
            candidates.append((-(len(chain) - 1), c, chain))
    _, c, chain = min(candidates)
    if best[c] < 0:
        return None
    toks = [int(tok[n]) for n in chain[1:]] + [best[c]]
    return len(chain) - 1, chain, toks


def random_tree(rng, N):
    return [-1] + [int(rng.integers(i)) for i in range(1, N)]


@pytest.mark.parametrize("seed", range(6))
def test_greedy_matches_path_enumeration(orc, seed):
    rng = np.random.default_rng(seed)
    B, N, V = 200, 9, 4
    par = np.array([random_tree(rng, N) for _ in range(B)], np.int32)
    # integer-valued logits: many ties; a few NaNs
    logits = rng.integers(0, 3, size=(B, N, V)).astype(np.float32)
    logits[rng.random((B, N, V)) < 0.05] = np.nan
    tok = rng.integers(0, V, size=(B, N)).astype(np.int32)
    acc, path, out, st = orc.accept_greedy(par, tok, logits, N)
    for b in range(B):
        ref = brute_force_greedy(list(par[b]), tok[b], logits[b], N)
        if ref is None:
            assert st[b] == orc.BAD_VALUES
            continue
        A, chain, toks = ref
        assert st[b] == 0
        assert acc[b] == A
        assert list(path[b, :A + 1]) == chain and (path[b, A + 1:] == -1).all()
        assert list(out[b, :A + 1]) == toks and (out[b, A + 1:] == -1).all()


def test_greedy_golden_fixed7(orc):
    lines = [l.strip() for l in open(os.path.join(GOLDEN, "greedy_fixed7.txt"))
             if l.strip() and not l.startswith("#")]
    rows = [list(map(float, l.split(":")[1].split())) for l in lines if l.startswith("row")]
    tokens = [int(x) for x in next(l for l in lines if l.startswith("tokens")).split(":")[1].split()]
    exp = {l.split(":")[0][len("expect "):]: [int(x) for x in l.split(":")[1].split()]
           for l in lines if l.startswith("expect")}
    par = np.array([[-1, 0, 0, 1, 1, 2, 2]], np.int32)
    acc, path, out, st = orc.accept_greedy(par, np.array([tokens], np.int32),
                                           np.array([rows], np.float32), 4)
    assert st[0] == 0
    assert acc[0] == exp["accept_len"][0]
    assert list(path[0, :3]) == exp["path"] and path[0, 3] == -1
    assert list(out[0, :3]) == exp["out_tokens"] and out[0, 3] == -1


def test_greedy_chain_all_accepted_equals_greedy_decode(orc):
    """On a chain whose drafts are each row's argmax, every draft is accepted and
    the emitted tokens are exactly the target's greedy continuation."""
    rng = np.random.default_rng(1)
    N, V = 7, 50
    logits = rng.standard_normal((1, N, V)).astype(np.float32)
    tok = np.zeros((1, N), np.int32)
    for k in range(1, N):
        tok[0, k] = int(np.argmax(logits[0, k - 1]))
    par = np.arange(-1, N - 1, dtype=np.int32)[None]
    acc, path, out, st = orc.accept_greedy(par, tok, logits, N)
    assert acc[0] == N - 1 and list(path[0]) == list(range(N))
    assert list(out[0]) == [int(np.argmax(logits[0, k])) for k in range(N)]


def test_greedy_errors(orc):
    par = np.array([[-1, 0, 0], [-1, 0, 0], [-1, 2, 0], [-1, 0, 1]], np.int32)
    tok = np.array([[0, 1, 2], [0, 9, 1], [0, 1, 1], [0, 1, 1]], np.int32)
    logits = np.zeros((4, 3, 4), np.float32)
    logits[0, 0, 1] = 1
    logits[0, 1, :] = np.nan           # the accepted leaf has an all-NaN row
    logits[3, 0, 1] = 1
    logits[3, 1, 1] = 1
    acc, path, out, st = orc.accept_greedy(par, tok, logits, 3)
    assert list(st) == [orc.BAD_VALUES, orc.OUT_OF_RANGE, orc.BAD_TREE, 0]
    for b in range(3):
        assert acc[b] == 0 and list(path[b]) == [0, -1, -1] and list(out[b]) == [-1, -1, -1]
    # path of length 3 does not fit in max_path 2
    acc, path, out, st = orc.accept_greedy(par[3:], tok[3:], logits[3:], 2)
    assert st[0] == orc.OUT_OF_RANGE


# ---------------------------------------------------------------------------
# Philox4x32-10 known-answer vectors (Salmon et al., SC'11, and the
# known-answer file distributed with its reference implementation)
# ---------------------------------------------------------------------------

KAT = [
    ((0, 0, 0, 0), (0, 0), (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
    ((0xFFFFFFFF,) * 4, (0xFFFFFFFF,) * 2, (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
    ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
     (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)),
]


@pytest.mark.parametrize("ctr,key,expect", KAT)
def test_philox_known_answers(orc, ctr, key, expect):
    assert tuple(int(x) for x in orc.philox4x32_10(ctr, key)) == expect


# ---------------------------------------------------------------------------
# integer CDF sampler
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("w", [[3, 0, 5, 2], [1], [0, 0, 7], [2**40, 1, 2**40 - 1, 0, 9],
                               [5, 5, 5, 5, 5, 5, 5]])
def test_integer_cdf_interval_boundaries(orc, w):
    """x maps to t exactly for x in [ceil(2^32 C_{t-1} / S), ceil(2^32 C_t / S)),
    so index t is drawn with probability (interval length) / 2^32 = w_t / S to
    within 2^-32."""
    S = sum(w)
    C = [0]
    for x in w:
        C.append(C[-1] + x)           # Python integers: no overflow
    for t in range(len(w)):
        lo = -(-(C[t] << 32) // S)
        hi = -(-(C[t + 1] << 32) // S)
        if w[t] == 0:
            assert lo == hi
            continue
        for x in {lo, hi - 1, (lo + hi) // 2}:
            if lo <= x < hi and 0 <= x < 2**32:   # empty when w_t / S < 2^-32
                assert orc.sample_weights(w, x) == t
        assert abs((hi - lo) / 2**32 - w[t] / S) <= 2**-32
    assert orc.sample_weights([0, 0], 123) == -1


# ---------------------------------------------------------------------------
# rejection sampling
# ---------------------------------------------------------------------------

def draft_from_q(rng, q, B):
    N = q.shape[0]
    tok = np.zeros((B, N), np.int32)
    for k in range(1, N):
        tok[:, k] = rng.choice(q.shape[1], size=B, p=q[k] / q[k].sum())
    return tok


def test_rejection_sampling_reproduces_target_distribution(orc):
    """First emitted token ~ p_0; given the first draft was accepted, the second
    emitted token ~ p_1 (the target distributions of those positions)."""
    rng = np.random.default_rng(2024)
    V, N, B = 8, 4, 250_000
    p = rng.dirichlet(np.ones(V) * 0.7, size=N).astype(np.float32)
    q = rng.dirichlet(np.ones(V) * 0.7, size=N).astype(np.float32)
    par = np.tile(np.arange(-1, N - 1, dtype=np.int32), (B, 1))
    P = np.broadcast_to(p, (B, N, V))
    Q = np.broadcast_to(q, (B, N, V))
    first, second = [], []
    acc_hits = 0
    for offset in range(4):
        tok = draft_from_q(rng, q, B)
        acc, path, out, st = orc.accept_stochastic(par, tok, P, Q, seed=99, offset=offset,
                                                   max_path=N)
        assert (st == 0).all()
        first.append(out[:, 0])
        second.append(out[acc >= 1, 1])
        acc_hits += int((acc >= 1).sum())
    first = np.concatenate(first)
    second = np.concatenate(second)
    for sample, target in ((first, p[0]), (second, p[1])):
        counts = np.bincount(sample, minlength=V)
        expect = target.astype(np.float64) / target.sum() * len(sample)
        keep = expect > 5
        chi2 = ((counts[keep] - expect[keep]) ** 2 / expect[keep]).sum()
        pval = stats.chi2.sf(chi2, keep.sum() - 1)
        assert pval > 1e-4, (counts, expect)
        tv = 0.5 * np.abs(counts / len(sample) - target / target.sum()).sum()
        assert tv < 5e-3
    # acceptance rate of the first draft = sum_x min(p_0(x), q_1(x))
    rate = acc_hits / (4 * B)
    assert abs(rate - np.minimum(p[0], q[1]).sum()) < 5e-3


def test_identical_draft_and_target_always_accepts(orc):
    """q row k (draft for node k) equal to p row k-1 (target at that position)."""
    rng = np.random.default_rng(5)
    V, N, B = 16, 6, 4000
    p = rng.dirichlet(np.ones(V), size=(B, N)).astype(np.float32)
    q = np.zeros_like(p)
    q[:, 1:] = p[:, :-1]
    par = np.tile(np.arange(-1, N - 1, dtype=np.int32), (B, 1))
    tok = np.zeros((B, N), np.int32)
    for b in range(B):
        for k in range(1, N):
            tok[b, k] = rng.choice(V, p=q[b, k] / q[b, k].sum())
    acc, path, out, st = orc.accept_stochastic(par, tok, p, q, seed=1, offset=0, max_path=N)
    assert (st == 0).all() and (acc == N - 1).all()
    assert (out[:, :N - 1] == tok[:, 1:]).all()
    # the bonus token follows p_{N-1}
    assert (p[np.arange(B), N - 1, out[:, N - 1]] > 0).all()


def test_disjoint_supports_always_reject_and_resample_from_target(orc):
    V, N, B = 8, 3, 20000
    p = np.zeros((B, N, V), np.float32)
    q = np.zeros((B, N, V), np.float32)
    p[:, :, :4] = [0.1, 0.2, 0.3, 0.4]
    q[:, :, 4:] = 0.25
    par = np.tile(np.arange(-1, N - 1, dtype=np.int32), (B, 1))
    tok = np.tile(np.array([0, 5, 6], np.int32), (B, 1))
    acc, path, out, st = orc.accept_stochastic(par, tok, p, q, seed=3, offset=11, max_path=N)
    assert (st == 0).all() and (acc == 0).all()
    freq = np.bincount(out[:, 0], minlength=V) / B
    np.testing.assert_allclose(freq[:4], [0.1, 0.2, 0.3, 0.4], atol=0.015)
    assert (freq[4:] == 0).all() and (out[:, 1:] == -1).all()


def test_stochastic_takes_branching_trees_and_rejects_bad_tokens(orc):
    p = np.full((3, 3, 4), 0.25, np.float32)
    par = np.array([[-1, 0, 0], [-1, 0, 1], [-1, 0, 1]], np.int32)
    tok = np.array([[0, 1, 2], [0, 4, 1], [0, 1, 2]], np.int32)
    acc, path, out, st = orc.accept_stochastic(par, tok, p, p, seed=0, offset=0, max_path=3)
    assert list(st) == [0, orc.OUT_OF_RANGE, 0]
    # p == q: the first child of the root is accepted, then node 1 is a leaf
    assert acc[0] == 1 and list(path[0]) == [0, 1, -1] and out[0, 0] == 1


# ---- branching trees: multi-candidate rejection sampling ------------------------

TREE = np.array([-1, 0, 0, 0, 1, 1, 2], np.int32)  # root: 3 children; node 1: 2; node 2: 1


def tree_inputs(rng, B, V, seed_rows):
    """Target rows p[node] and draft rows q[node] = Q[parent(node)] (siblings are
    drawn i.i.d. from their parent's draft distribution), tokens sampled from q."""
    N = len(TREE)
    pr = np.random.default_rng(seed_rows)
    p = pr.dirichlet(np.ones(V) * 0.7, size=N).astype(np.float32)
    Qp = pr.dirichlet(np.ones(V) * 0.7, size=N).astype(np.float32)
    q = np.zeros((N, V), np.float32)
    for c in range(1, N):
        q[c] = Qp[TREE[c]]
    tok = np.zeros((B, N), np.int32)
    for c in range(1, N):
        cdf = np.cumsum(q[c].astype(np.float64))
        tok[:, c] = np.minimum(np.searchsorted(cdf / cdf[-1], rng.random(B)), V - 1)
    return p, q, tok


def test_tree_rejection_sampling_reproduces_target_distribution(orc):
    """Whatever the tree's branching, the first emitted token follows the root's
    target row, and given that node 1 was accepted the next one follows p[1]
    (lossless speculative sampling, "vLLM EAGLE in practice", 无损性保障)."""
    rng = np.random.default_rng(77)
    V, B = 8, 250_000
    p, q, _ = tree_inputs(rng, B, V, 3)
    N = len(TREE)
    par = np.tile(TREE, (B, 1))
    P = np.broadcast_to(p, (B, N, V))
    Qb = np.broadcast_to(q, (B, N, V))
    first, second = [], []
    for offset in range(4):
        _, _, tok = tree_inputs(rng, B, V, 3)
        acc, path, out, st = orc.accept_stochastic(par, tok, P, Qb, seed=5, offset=offset,
                                                   max_path=4)
        assert (st == 0).all()
        first.append(out[:, 0])
        via1 = (acc >= 1) & (path[:, 1] == 1)
        second.append(out[via1, 1])
    for sample, target in ((np.concatenate(first), p[0]), (np.concatenate(second), p[1])):
        counts = np.bincount(sample, minlength=V)
        expect = target.astype(np.float64) / target.sum() * len(sample)
        keep = expect > 5
        chi2 = ((counts[keep] - expect[keep]) ** 2 / expect[keep]).sum()
        assert stats.chi2.sf(chi2, keep.sum() - 1) > 1e-4, (counts, expect)
        tv = 0.5 * np.abs(counts / len(sample) - target / target.sum()).sum()
        assert tv < 5e-3


def test_tree_rule_reduces_to_the_chain_rule_on_chains(orc):
    """The branching-tree routine run on chains gives exactly the chain routine's
    accept lengths, paths and tokens (same draws, same integer CDF)."""
    rng = np.random.default_rng(8)
    B, N, V = 3000, 6, 64
    p = rng.dirichlet(np.ones(V) * 0.5, size=(B, N)).astype(np.float32)
    q = rng.dirichlet(np.ones(V) * 0.5, size=(B, N)).astype(np.float32)
    par = np.tile(np.arange(-1, N - 1, dtype=np.int32), (B, 1))
    tok = rng.integers(0, V, size=(B, N)).astype(np.int32)
    a = orc.accept_stochastic(par, tok, p, q, seed=11, offset=3, max_path=N)
    t = orc.accept_stochastic_tree(par, tok, p, q, seed=11, offset=3, max_path=N)
    for x, y in zip(a, t):
        assert np.array_equal(x, y)
    assert 0 < (a[0] > 0).mean() < 1  # both outcomes occur


def test_tree_identical_draft_and_target_takes_first_children(orc):
    """q of every child equal to its parent's target row: the first child is
    always accepted, so the path follows first children to a leaf."""
    rng = np.random.default_rng(9)
    V, B = 16, 2000
    N = len(TREE)
    p = rng.dirichlet(np.ones(V), size=(B, N)).astype(np.float32)
    q = np.zeros_like(p)
    for c in range(1, N):
        q[:, c] = p[:, TREE[c]]
    tok = rng.integers(0, V, size=(B, N)).astype(np.int32)
    acc, path, out, st = orc.accept_stochastic(np.tile(TREE, (B, 1)), tok, p, q, seed=2,
                                               offset=0, max_path=4)
    # first children: 0 -> 1 -> 4 (a leaf); tokens with p = 0 never occur here
    ok = p[np.arange(B), 0, tok[:, 1]] > 0
    ok &= p[np.arange(B), 1, tok[:, 4]] > 0
    assert (st == 0).all()
    assert (acc[ok] == 2).all() and (path[ok, :3] == [0, 1, 4]).all()


def test_tree_disjoint_supports_reject_every_child_and_resample_from_target(orc):
    """Drafts only where the target is zero: every child of the root is tried and
    rejected, and the emitted token follows the target row."""
    V, B = 8, 20000
    N = len(TREE)
    p = np.zeros((B, N, V), np.float32)
    q = np.zeros((B, N, V), np.float32)
    p[:, :, :4] = [0.1, 0.2, 0.3, 0.4]
    q[:, :, 4:] = 0.25
    tok = np.tile(np.array([0, 5, 6, 7, 4, 5, 6], np.int32), (B, 1))
    acc, path, out, st = orc.accept_stochastic(np.tile(TREE, (B, 1)), tok, p, q, seed=4,
                                               offset=1, max_path=4)
    assert (st == 0).all() and (acc == 0).all()
    freq = np.bincount(out[:, 0], minlength=V) / B
    np.testing.assert_allclose(freq[:4], [0.1, 0.2, 0.3, 0.4], atol=0.015)
    assert (freq[4:] == 0).all()


def test_tree_second_child_acceptance_matches_the_residual(orc):
    """Root with two children, both drafted from q: after the first is rejected,
    the second is accepted with probability sum_x q(x) min(1, r(x)/q(x)) =
    sum_x min(q(x), r(x)), r = norm(max(0, p - q)) (the residual's overlap)."""
    rng = np.random.default_rng(12)
    V, B = 6, 400_000
    par2 = np.array([-1, 0, 0], np.int32)
    p0 = np.array([0.05, 0.3, 0.1, 0.25, 0.2, 0.1], np.float32)
    qd = np.array([0.3, 0.1, 0.2, 0.1, 0.2, 0.1], np.float32)
    p = np.broadcast_to(np.stack([p0, p0, p0]), (B, 3, V))
    q = np.broadcast_to(np.stack([qd, qd, qd]), (B, 3, V))
    cdf = np.cumsum(qd.astype(np.float64))
    tok = np.zeros((B, 3), np.int32)
    for c in (1, 2):
        tok[:, c] = np.minimum(np.searchsorted(cdf, rng.random(B)), V - 1)
    acc, path, out, st = orc.accept_stochastic(np.tile(par2, (B, 1)), tok, p, q, seed=6,
                                               offset=0, max_path=2)
    assert (st == 0).all()
    r = np.maximum(0.0, p0.astype(np.float64) - qd)
    r /= r.sum()
    first_rej = ~((acc == 1) & (path[:, 1] == 1))
    second_acc = (acc == 1) & (path[:, 1] == 2)
    rate = second_acc.sum() / first_rej.sum()
    assert abs(rate - np.minimum(qd, r).sum()) < 4e-3
    assert abs((1 - first_rej.mean()) - np.minimum(p0, qd).sum()) < 3e-3


def test_stochastic_draws_depend_on_seed_offset_and_sequence(orc):
    V, N, B = 64, 2, 512
    rng = np.random.default_rng(0)
    p = rng.dirichlet(np.ones(V), size=(1, N)).astype(np.float32)
    q = rng.dirichlet(np.ones(V), size=(1, N)).astype(np.float32)
    P = np.broadcast_to(p, (B, N, V))
    Q = np.broadcast_to(q, (B, N, V))
    par = np.tile(np.array([-1, 0], np.int32), (B, 1))
    tok = np.tile(np.array([0, int(np.argmax(q[0, 1]))], np.int32), (B, 1))
    r1 = orc.accept_stochastic(par, tok, P, Q, 1, 0, 2)[2]
    r2 = orc.accept_stochastic(par, tok, P, Q, 1, 0, 2)[2]
    r3 = orc.accept_stochastic(par, tok, P, Q, 1, 1, 2)[2]
    r4 = orc.accept_stochastic(par, tok, P, Q, 2, 0, 2)[2]
    assert np.array_equal(r1, r2)
    assert not np.array_equal(r1, r3) and not np.array_equal(r1, r4)
    assert len(np.unique(r1[:, 0])) > 10          # sequences draw independently
