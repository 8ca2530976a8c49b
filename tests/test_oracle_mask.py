"""Pins for the oracle's tree mask (CPU only).

The rule ("vLLM-TreeEagle", 核心组件 / TreeAttentionLayer): the mask is built
dynamically from the tree so that each draft node attends to its own root
path.  The oracle walks parent links upward; these tests derive the same
relation independently as the reflexive-transitive closure of the parent
relation (Warshall's algorithm) and the depth by a breadth-first search from
the root, over every valid tree with up to 7 nodes.
"""
import itertools
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def all_trees(N):
    """Every parent array with parents[0] = -1 and 0 <= parents[i] < i."""
    for rest in itertools.product(*[range(i) for i in range(1, N)]):
        yield [-1, *rest]


def closure_mask(par):
    N = len(par)
    R = np.eye(N, dtype=bool)
    for i in range(1, N):
        R[i, par[i]] = True          # i -> parent
    for k in range(N):               # Warshall
        R = R | (R[:, [k]] & R[[k], :])
    return [sum(1 << j for j in range(N) if R[i, j]) for i in range(N)]


def bfs_depth(par):
    N = len(par)
    kids = {u: [] for u in range(N)}
    for i in range(1, N):
        kids[par[i]].append(i)
    dep = [-1] * N
    dep[0] = 0
    frontier = [0]
    while frontier:
        nxt = []
        for u in frontier:
            for c in kids[u]:
                dep[c] = dep[u] + 1
                nxt.append(c)
        frontier = nxt
    return dep


@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 6, 7])
def test_mask_every_tree_matches_closure(orc, N):
    trees = list(all_trees(N))
    parents = np.array(trees, np.int32)
    mask, depth, status = orc.tree_mask(parents)
    assert (status == 0).all()
    for b, par in enumerate(trees):
        assert [int(m) for m in mask[b]] == closure_mask(par)
        assert list(depth[b]) == bfs_depth(par)


def test_mask_golden_fixed7(orc):
    rows = [l.split() for l in open(os.path.join(GOLDEN, "tree_mask_fixed7.txt"))
            if l.strip() and not l.startswith("#")]
    exp_mask = [int(r[1], 2) for r in rows]
    exp_depth = [int(r[2]) for r in rows]
    mask, depth, status = orc.tree_mask(np.array([[-1, 0, 0, 1, 1, 2, 2]], np.int32))
    assert status[0] == 0
    assert [int(m) for m in mask[0]] == exp_mask
    assert list(depth[0]) == exp_depth


def test_mask_chain_and_star_closed_forms(orc):
    N = 64
    chain = np.arange(-1, N - 1, dtype=np.int32)[None]
    star = np.array([[-1] + [0] * (N - 1)], np.int32)
    m, d, s = orc.tree_mask(np.concatenate([chain, star]))
    assert (s == 0).all()
    for i in range(N):
        assert int(m[0, i]) == (1 << (i + 1)) - 1 if i < 63 else int(m[0, i]) == 2**64 - 1
        assert int(m[1, i]) == (1 | (1 << i))
        assert d[0, i] == i and d[1, i] == (0 if i == 0 else 1)


def test_mask_popcount_is_depth_plus_one(orc):
    rng = np.random.default_rng(0)
    N = 40
    par = np.array([[-1] + [int(rng.integers(i)) for i in range(1, N)] for _ in range(50)],
                   np.int32)
    m, d, s = orc.tree_mask(par)
    pc = np.array([[bin(int(x)).count("1") for x in row] for row in m])
    assert (pc == d + 1).all()


@pytest.mark.parametrize("bad", [
    [0, 0, 1],          # root has a parent
    [-1, 1, 0],         # self parent
    [-1, 0, 3, 1],      # forward parent
    [-1, -1, 0],        # second root
    [-1, 0, -5],        # negative parent
])
def test_mask_invalid_trees(orc, bad):
    m, d, s = orc.tree_mask(np.array([bad], np.int32))
    assert s[0] == orc.BAD_TREE
    assert (m == 0).all() and (d == -1).all()
