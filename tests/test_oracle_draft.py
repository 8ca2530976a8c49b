"""Pins for the oracle's draft-tree construction (CPU only).

The pages give the outline ("vLLM-TreeEagle", 核心组件 / 3.
EnhancedEagleProposer: multi-level candidate generation with path pruning;
"EAGLE code principles", 树结构缓冲: precompute likely paths, keep the
high-probability ones, prune the rest); the oracle fills it in EAGLE-2 style
(top-k children per expanded node, the k best new nodes expanded next, the
N - 1 best nodes kept, breadth-first labels).  These tests check it against
things fixed independently of its code:

Scores are formed in binary32, the precision of the draft logits (the pages
fix none for the ranking, an integer result decided by comparing scores), so
they are compared with the double-precision recomputations within 5e-5.

* exhaustive enumeration: when k >= N - 1 no pruning step can drop a node of
  the best N - 1 root paths (each of them has fewer than k better nodes at its
  own depth and among its siblings), so the tree must be exactly the N - 1
  best of ALL token paths up to the depth, scored with scipy's log_softmax;
* closed forms: k = 1 is the greedy argmax chain, one layer is the root row's
  stable argsort;
* with pruning active, every property the construction promises, recomputed
  with numpy / scipy from a path-keyed synthetic draft model;
* a hand-worked fixture, the tie rule, the breadth-first labelling and the
  error cases.
"""
import itertools
import os

import numpy as np
import pytest
from scipy.special import log_softmax

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def draft_row(seed, path, V, sigma=2.0):
    """Synthetic draft model: the logits after a token path, keyed by the path."""
    rng = np.random.default_rng([seed, len(path), *path])
    return (sigma * rng.standard_normal(V)).astype(np.float32)


def run(orc, seed, V, k, L, N, root=0):
    t = orc.DraftTree(root, V, k, L)
    fronts = []
    for _ in range(L):
        paths = t.front_paths()
        rows = np.stack([draft_row(seed, p, V) for p in paths])
        ft, fs = t.expand(rows)
        fronts.append((paths, ft, fs))
    par, tok, sc, st = t.finalize(N)
    return t, fronts, par, tok, sc, st


def node_paths(par, tok):
    paths = [()]
    for i in range(1, len(par)):
        paths.append(paths[par[i]] + (int(tok[i]),))
    return paths


def path_score(seed, path, V):
    s = 0.0
    for j in range(len(path)):
        s += float(log_softmax(draft_row(seed, path[:j], V).astype(np.float64))[path[j]])
    return s


@pytest.mark.parametrize("seed,V,k,L,N", [(1, 5, 4, 3, 5), (2, 5, 5, 3, 6), (3, 4, 4, 4, 5),
                                          (4, 6, 3, 3, 4), (5, 3, 3, 4, 4)])
def test_equals_best_paths_of_exhaustive_enumeration(orc, seed, V, k, L, N):
    _, _, par, tok, sc, st = run(orc, seed, V, k, L, N)
    assert st == orc.OK
    allp = [p for d in range(1, L + 1) for p in itertools.product(range(V), repeat=d)]
    scores = {p: path_score(seed, p, V) for p in allp}
    best = sorted(allp, key=lambda p: -scores[p])[:N - 1]
    got = node_paths(par, tok)
    assert got[0] == () and set(got[1:]) == set(best)
    for p, s in zip(got[1:], sc[1:]):
        assert abs(s - scores[p]) < 5e-5


def test_chain_when_k_is_one(orc):
    seed, V, L = 7, 40, 6
    _, _, par, tok, sc, st = run(orc, seed, V, 1, L, L + 1, root=11)
    assert st == orc.OK
    assert list(par) == [-1] + list(range(L))
    path, s = [], 0.0
    for i in range(1, L + 1):
        row = draft_row(seed, tuple(path), V)
        t = int(np.argmax(row))
        s += float(log_softmax(row.astype(np.float64))[t])
        path.append(t)
        assert tok[i] == t and abs(sc[i] - s) < 5e-5
    assert tok[0] == 11


def test_one_layer_is_the_root_rows_stable_argsort(orc):
    seed, V, k, N = 8, 30, 12, 9
    row = draft_row(seed, (), V)
    row[[3, 17, 25]] = row.max()               # a three-way tie at the top
    t = orc.DraftTree(4, V, k, 1)
    t.expand(row[None])
    par, tok, sc, st = t.finalize(N)
    assert st == orc.OK
    order = np.argsort(-row, kind="stable")
    assert list(tok[1:]) == list(order[:N - 1]) and list(tok[1:4]) == [3, 17, 25]
    assert (par[1:] == 0).all()
    assert np.allclose(sc[1:], log_softmax(row.astype(np.float64))[order[:N - 1]], atol=1e-6)


@pytest.mark.parametrize("seed,V,k,L,N", [(11, 9, 2, 4, 8), (12, 7, 3, 4, 12), (13, 12, 4, 3, 20),
                                          (14, 6, 2, 6, 10)])
def test_pruned_construction_properties(orc, seed, V, k, L, N):
    t, fronts, par, tok, sc, st = run(orc, seed, V, k, L, N)
    assert st == orc.OK
    # every node the construction created: each frontier path's top-k children
    created = {}
    prev = [()]
    for layer, (paths, ft, fs) in enumerate(fronts):
        assert paths == prev
        cand = []
        for p in paths:
            row = draft_row(seed, p, V).astype(np.float64)
            for tkn in np.argsort(-row, kind="stable")[:k]:
                q = p + (int(tkn),)
                created[q] = created.get(p, 0.0) + float(log_softmax(row)[tkn])
                cand.append(q)
        # the next frontier: the k best children of this layer, best first
        want = sorted(cand, key=lambda q: -created[q])[:k]
        got = [paths[fs[r]] + (int(ft[r]),) for r in range(len(ft))]
        assert got == want
        prev = got
    # the tree: the root and the N - 1 best created nodes
    got = node_paths(par, tok)
    best = sorted(created, key=lambda q: -created[q])[:N - 1]
    assert set(got[1:]) == set(best)
    for p, s in zip(got[1:], sc[1:]):
        assert abs(s - created[p]) < 5e-5
    # breadth-first labels: parents never decrease, siblings keep creation
    # (= draft-probability) order, depth never decreases
    assert all(par[i] <= par[i + 1] for i in range(1, N - 1))
    assert all(0 <= par[i] < i for i in range(1, N))
    for i in range(1, N - 1):
        if par[i] == par[i + 1]:
            assert sc[i] >= sc[i + 1]
    dep = [len(p) for p in got]
    assert dep == sorted(dep)


def test_golden_hand_worked_v4(orc):
    lines = [l.strip() for l in open(os.path.join(GOLDEN, "draft_tree_v4.txt"))
             if l.strip() and not l.startswith("#")]
    rows = {}
    exp = {}
    root = None
    for l in lines:
        key, val = l.split(":")
        if key.startswith("row"):
            _, layer, f = key.split()
            rows.setdefault(int(layer), {})[int(f)] = np.log(np.array(val.split(), np.float64))
        elif key == "root":
            root = int(val)
        else:
            exp[key[len("expect "):]] = [float(x) for x in val.split()]
    for N in (4, 5):
        t = orc.DraftTree(root, 4, 2, 2)
        for layer in (0, 1):
            r = np.stack([rows[layer][f] for f in sorted(rows[layer])]).astype(np.float32)
            ft, fs = t.expand(r)
            assert list(ft) == exp[f"front {layer} tokens"]
            assert list(fs) == exp[f"front {layer} src"]
        par, tok, sc, st = t.finalize(N)
        assert st == orc.OK
        assert list(par) == exp[f"N{N} parents"] and list(tok) == exp[f"N{N} tokens"]
        assert np.allclose(np.exp(sc), exp[f"N{N} probs"], rtol=1e-6)


def test_full_tree_and_root_only(orc):
    seed, V, k, L = 21, 10, 3, 3
    C = 1 + k + (L - 1) * k * k
    t, _, par, tok, sc, st = run(orc, seed, V, k, L, C)
    assert st == orc.OK and t.count == C
    assert sorted(len(p) for p in node_paths(par, tok)) == [0] + [1] * k + [2] * k * k + [3] * k * k
    _, _, par1, tok1, sc1, st1 = run(orc, seed, V, k, L, 1, root=9)
    assert st1 == orc.OK and list(par1) == [-1] and list(tok1) == [9] and sc1[0] == 0.0


def test_minus_infinity_logits_are_never_preferred(orc):
    V = 8
    row = np.full(V, -np.inf, np.float32)
    row[[2, 5]] = [0.0, 1.0]
    t = orc.DraftTree(0, V, 3, 1)
    t.expand(row[None])
    par, tok, sc, st = t.finalize(4)
    assert st == orc.OK
    assert list(tok[1:]) == [5, 2, 0]           # then the lowest-id -inf token
    assert sc[3] == -np.inf


@pytest.mark.parametrize("bad", [np.nan, np.inf, "all-minus-inf"])
def test_bad_rows_fail_the_sequence(orc, bad):
    V, k = 6, 2
    rows0 = np.zeros((2, 1, V), np.float32)
    rows1 = np.zeros((2, k, V), np.float32)
    if bad == "all-minus-inf":
        rows1[1, 1, :] = -np.inf
    else:
        rows1[1, 1, 4] = bad
    par, tok, sc, fronts, st, _ = orc.draft_tree([rows0, rows1], [1, 2], k, 4)
    assert list(st) == [orc.OK, orc.BAD_VALUES]
    assert (par[1] == -1).all() and (tok[1] == -1).all() and (sc[1] == -np.inf).all()
    assert (fronts[1][0][1] == -1).all()
    assert list(par[0]) == [-1, 0, 0, 1]


def test_equal_scores_rank_by_creation_order(orc):
    """Exact score ties: the node created first ranks first, at the final cut
    and inside the frontier (a stable order, like the token tie rule)."""
    V = 6
    row = np.log(np.array([0.1, 0.3, 0.1, 0.3, 0.1, 0.1], np.float64)).astype(np.float32)
    t = orc.DraftTree(0, V, 3, 1)
    t.expand(row[None])
    par, tok, _, st = t.finalize(3)               # tokens 1 and 3 tie; 0, 2, 4 tie below
    assert st == orc.OK and list(tok) == [0, 1, 3]
    t = orc.DraftTree(0, V, 3, 1)
    t.expand(row[None])
    par, tok, _, st = t.finalize(4)               # the cut falls inside the tie at 0.1
    assert st == orc.OK and list(tok) == [0, 1, 3, 0]
    # two tied parents with identical rows: their children tie pairwise and the
    # frontier lists the first parent's child before the second's
    row1 = np.log(np.array([0.1, 0.5, 0.1, 0.2, 0.05, 0.05], np.float64)).astype(np.float32)
    for N, want_par, want_tok in ((5, [-1, 0, 0, 1, 2], [0, 1, 3, 1, 1]),
                                  (4, [-1, 0, 0, 1], [0, 1, 3, 1])):
        t = orc.DraftTree(0, V, 2, 2)
        ft, fs = t.expand(row[None])
        assert list(ft) == [1, 3] and list(fs) == [0, 0]
        ft, fs = t.expand(np.stack([row1, row1]))
        assert list(ft) == [1, 1] and list(fs) == [0, 1]
        par, tok, _, st = t.finalize(N)
        assert st == orc.OK and list(par) == want_par and list(tok) == want_tok


def test_breadth_first_labels_on_deep_trees(orc):
    """Breadth-first labels, characterised without the creation order: node 0
    is the root, parents never decrease along the labels, and siblings appear
    in draft-probability order.  Deep trees with a frontier whose rank order
    differs from the label order (the case a level-by-creation-id labelling
    gets wrong)."""
    seen_inversion = False
    for seed in range(30):
        V, k, L, N = 16, 3, 6, 40
        t, fronts, par, tok, sc, st = run(orc, 100 + seed, V, k, L, N)
        assert st == orc.OK
        assert par[0] == -1 and all(par[i] <= par[i + 1] for i in range(1, N - 1))
        for i in range(1, N - 1):
            if par[i] == par[i + 1]:
                assert sc[i] >= sc[i + 1]
        label = {p: i for i, p in enumerate(node_paths(par, tok))}
        for paths, ft, fs in fronts:
            # the frontier chosen at this layer, best first, and its labels
            ranked = [paths[s] + (int(x),) for x, s in zip(ft, fs)]
            labs = [label[p] for p in ranked if p in label]
            seen_inversion |= labs != sorted(labs)
    assert seen_inversion
