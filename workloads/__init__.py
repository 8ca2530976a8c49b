"""Seeded synthetic workloads for EAGLE draft-tree verification.

This module is shared by the tests, the benchmark and the smoke check, and
holds none of the verification arithmetic: it only draws random numbers and
lays them out.  It imports neither the oracle nor the CUDA library.

The five named workloads follow the shapes the pages' setting implies
(Llama-3-8B and Qwen2-7B attention geometry, EAGLE-style trees of 7 to 63
nodes, a chain draft of five tokens).  The pages' own evaluation data (chat
and coding prompts, trained draft heads) is not available, so every tensor is
random with the stated distribution:

* Q and the paged K/V caches ~ N(0, 1), rounded to bfloat16 (kept in float32
  for the tiny workload).
* Physical KV blocks: a seeded random permutation of the blocks each sequence
  needs (identity order for the "contiguous" tiny workload); unused block
  table entries are -1.
* Trees: the fixed 7-node tree; an EAGLE-2-style tree (top-4 expansion of the
  four best nodes per layer by cumulative draft log-probability, then the
  global best N-1 candidates, relabelled breadth first); or random trees
  (each new node picks a uniform parent among nodes of depth < D with fewer
  than `branch` children, then breadth-first relabelling); or a chain.
* Greedy workloads plant an accepted path: per sequence a depth A is drawn
  uniformly from 0..max depth and a uniform node at that depth is the planted
  end point.  Every internal node u gets a designated token z_u whose logit is
  set to 10 sigma (far above any N(0, sigma) draw over the vocabulary, so the
  row's maximum is known without computing it); the planted path's children
  carry z_parent, every other child carries a different token, and siblings
  are distinct.
* The stochastic chain workload: p and q rows are softmax(N(0, 3) / 0.8)
  (float32), drawn independently; draft token k is drawn from q row k.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

__all__ = ["Spec", "SPECS", "DEFAULT_BENCH", "make", "f32_to_bf16_bits", "bf16_bits_to_f32"]


@dataclasses.dataclass(frozen=True)
class Spec:
    name: str
    B: int
    P_lo: int
    P_hi: int
    Hq: int
    Hkv: int
    d: int
    V: int
    N: int
    tree: str            # "fixed" | "eagle2" | "random" | "chain"
    depth: int = 0       # maximum tree depth (random / eagle2 trees)
    branch: int = 0      # maximum children per node (random trees) / top-k (eagle2)
    bs: int = 16
    bf16: bool = True
    mode: str = "greedy"  # "greedy" | "stochastic"
    sigma: float = 3.0   # logit standard deviation
    temperature: float = 1.0
    seed: int = 0
    contiguous: bool = False
    fixed_parents: tuple = ()


SPECS = {
    s.name: s for s in [
        Spec("tiny_fp32", B=1, P_lo=64, P_hi=64, Hq=2, Hkv=1, d=64, V=1000, N=7, tree="fixed",
             fixed_parents=(-1, 0, 0, 1, 1, 2, 2), bf16=False, sigma=2.0, seed=0,
             contiguous=True),
        Spec("llama3_8b_tree60", B=1, P_lo=2048, P_hi=2048, Hq=32, Hkv=8, d=128, V=128256,
             N=60, tree="eagle2", depth=6, branch=4, sigma=3.0, seed=2),
        Spec("llama3_8b_b32_tree26", B=32, P_lo=512, P_hi=8192, Hq=32, Hkv=8, d=128, V=128256,
             N=26, tree="random", depth=6, branch=4, sigma=3.0, seed=3),
        Spec("llama3_8b_b128_chain5", B=128, P_lo=1024, P_hi=4096, Hq=32, Hkv=8, d=128,
             V=128256, N=6, tree="chain", mode="stochastic", sigma=3.0, temperature=0.8,
             seed=7),
        Spec("qwen2_7b_32k_tree63", B=8, P_lo=32768, P_hi=32768, Hq=28, Hkv=4, d=128,
             V=152064, N=63, tree="random", depth=8, branch=3, sigma=3.0, seed=5),
    ]
}

# the workload the benchmark times by default: the largest KV-read-bound one
# (batch 128, chain drafts of five tokens, stochastic acceptance)
DEFAULT_BENCH = "llama3_8b_b128_chain5"


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round finite float32 to bfloat16 (nearest, ties to even); returns uint16 bit patterns."""
    flat = np.ascontiguousarray(x, np.float32).reshape(-1).view(np.uint32)
    out = np.empty(flat.shape, np.uint16)
    step = 1 << 24
    for s in range(0, flat.size, step):       # bounded temporaries for large caches
        u = flat[s:s + step]
        out[s:s + step] = ((u + (0x7FFF + ((u >> 16) & 1))) >> 16).astype(np.uint16)
    return out.reshape(np.shape(x))


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns (uint16) to float32 exactly."""
    return (np.ascontiguousarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------------------
# trees
# ---------------------------------------------------------------------------

def _bfs_relabel(par_old: list, depth_old: list) -> np.ndarray:
    """Relabel nodes by (depth, creation order); returns the new parent array."""
    order = sorted(range(len(par_old)), key=lambda u: (depth_old[u], u))
    new_id = {u: i for i, u in enumerate(order)}
    out = np.empty(len(order), np.int32)
    for u in order:
        out[new_id[u]] = -1 if par_old[u] < 0 else new_id[par_old[u]]
    return out


def _random_tree(rng, N: int, max_depth: int, branch: int) -> np.ndarray:
    par, dep, nch = [-1], [0], [0]
    while len(par) < N:
        cand = [u for u in range(len(par)) if dep[u] < max_depth and nch[u] < branch]
        u = cand[int(rng.integers(len(cand)))]
        par.append(u)
        dep.append(dep[u] + 1)
        nch.append(0)
        nch[u] += 1
    return _bfs_relabel(par, dep)


def _eagle2_tree(rng, N: int, layers: int, topk: int) -> np.ndarray:
    """EAGLE-2-style expansion: per layer the top-k nodes (by cumulative draft
    log-probability) each get top-k children; then the N-1 best candidates."""
    par, dep, score = [-1], [0], [0.0]
    frontier = [0]
    for _ in range(layers):
        new = []
        for u in frontier:
            # top-k draft log-probabilities of this node: sorted Dirichlet mass
            mass = np.sort(rng.dirichlet(np.ones(topk + 1)))[::-1][:topk]
            for m in mass:
                par.append(u)
                dep.append(dep[u] + 1)
                score.append(score[u] + math.log(float(m)))
                new.append(len(par) - 1)
        new.sort(key=lambda v: (-score[v], v))
        frontier = new[:topk]
    cand = sorted(range(1, len(par)), key=lambda v: (-score[v], v))[: N - 1]
    keep = [0] + sorted(cand)
    idx = {u: i for i, u in enumerate(keep)}
    par_k = [-1 if par[u] < 0 else idx[par[u]] for u in keep]
    dep_k = [dep[u] for u in keep]
    return _bfs_relabel(par_k, dep_k)


def _make_tree(spec: Spec, rng) -> np.ndarray:
    if spec.tree == "fixed":
        return np.asarray(spec.fixed_parents, np.int32)
    if spec.tree == "chain":
        return np.arange(-1, spec.N - 1, dtype=np.int32)
    if spec.tree == "random":
        return _random_tree(rng, spec.N, spec.depth, spec.branch)
    if spec.tree == "eagle2":
        return _eagle2_tree(rng, spec.N, spec.depth, spec.branch)
    raise ValueError(spec.tree)


def _depths(par: np.ndarray) -> np.ndarray:
    dep = np.zeros(len(par), np.int32)
    for i in range(1, len(par)):
        dep[i] = dep[par[i]] + 1
    return dep


# ---------------------------------------------------------------------------
# workload
# ---------------------------------------------------------------------------

def make(name_or_spec, *, parts=("attn", "accept"), **overrides) -> dict:
    """Build a workload.

    ``overrides`` replace Spec fields (e.g. a smaller B, V or prefix range for
    parity tests).  ``parts`` selects what to generate: "attn" (q, caches,
    block table) and/or "accept" (tokens and logits, or p and q).
    Returns a dict of numpy arrays plus the spec under "spec".
    """
    spec = SPECS[name_or_spec] if isinstance(name_or_spec, str) else name_or_spec
    if overrides:
        spec = dataclasses.replace(spec, **overrides)
    seed = spec.seed
    rs = lambda tag: np.random.default_rng([seed, tag])  # noqa: E731

    B, N, bs = spec.B, spec.N, spec.bs
    rng_tree = rs(1)
    parents = np.stack([_make_tree(spec, rng_tree) for _ in range(B)]).astype(np.int32)
    assert parents.shape == (B, N)
    P = rs(2).integers(spec.P_lo, spec.P_hi + 1, size=B).astype(np.int32)
    w = {"spec": spec, "parents": parents, "prefix_lens": P}

    nb = [(int(p) + N + bs - 1) // bs for p in P]
    max_blocks = max(nb)
    total = sum(nb)
    perm = np.arange(total) if spec.contiguous else rs(3).permutation(total)
    bt = np.full((B, max_blocks), -1, np.int32)
    off = 0
    for b in range(B):
        bt[b, : nb[b]] = perm[off: off + nb[b]]
        off += nb[b]
    w["block_table"] = bt
    w["num_blocks"] = total

    if "attn" in parts:
        def normal(tag, shape):
            x = rs(tag).standard_normal(size=shape, dtype=np.float32)
            return f32_to_bf16_bits(x) if spec.bf16 else x
        w["q"] = normal(4, (B, N, spec.Hq, spec.d))
        w["k_cache"] = normal(5, (total, spec.Hkv, bs, spec.d))
        w["v_cache"] = normal(6, (total, spec.Hkv, bs, spec.d))

    if "accept" in parts:
        if spec.mode == "greedy":
            _greedy_inputs(spec, parents, rs, w)
        else:
            _stochastic_inputs(spec, parents, rs, w)
    return w


def _greedy_inputs(spec: Spec, parents: np.ndarray, rs, w: dict) -> None:
    B, N, V = spec.B, spec.N, spec.V
    rng = rs(7)
    logits = rs(8).standard_normal(size=(B, N, V), dtype=np.float32) * np.float32(spec.sigma)
    tokens = np.zeros((B, N), np.int32)
    planted = np.zeros(B, np.int32)
    spike = np.float32(10.0 * spec.sigma)
    for b in range(B):
        par = parents[b]
        dep = _depths(par)
        A = int(rng.integers(0, int(dep.max()) + 1))
        ends = np.flatnonzero(dep == A)
        end = int(ends[int(rng.integers(len(ends)))])
        on_path = set()
        j = end
        while j >= 0:
            on_path.add(j)
            j = int(par[j])
        planted[b] = A
        tokens[b, 0] = int(rng.integers(V))
        children = {u: [] for u in range(N)}
        for c in range(1, N):
            children[int(par[c])].append(c)
        for u in range(N):
            ch = children[u]
            if not ch:
                continue
            z = int(rng.integers(V))
            logits[b, u, z] = spike
            used = {z}
            for c in ch:
                if c in on_path:
                    tokens[b, c] = z
                    continue
                while True:
                    t = int(rng.integers(V))
                    if t not in used:
                        break
                used.add(t)
                tokens[b, c] = t
    w["draft_tokens"] = tokens
    w["logits"] = logits
    w["planted_accept_len"] = planted


def _softmax_rows(x: np.ndarray) -> np.ndarray:
    x = x - x.max(axis=-1, keepdims=True)
    np.exp(x, out=x)
    x /= x.sum(axis=-1, keepdims=True)
    return x


def _stochastic_inputs(spec: Spec, parents: np.ndarray, rs, w: dict) -> None:
    B, N, V = spec.B, spec.N, spec.V
    scale = np.float32(spec.sigma / spec.temperature)
    p = _softmax_rows(rs(9).standard_normal(size=(B, N, V), dtype=np.float32) * scale)
    q = _softmax_rows(rs(10).standard_normal(size=(B, N, V), dtype=np.float32) * scale)
    rng = rs(11)
    tokens = np.zeros((B, N), np.int32)
    for b in range(B):
        tokens[b, 0] = int(rng.integers(V))
        for k in range(1, N):
            row = q[b, k].astype(np.float64)
            tokens[b, k] = int(rng.choice(V, p=row / row.sum()))
    w["draft_tokens"] = tokens
    w["p"] = p.astype(np.float32)
    w["q_probs"] = q.astype(np.float32)
    w["seed"] = int(spec.seed)
    w["offset"] = 0


def max_path_len(parents: np.ndarray) -> int:
    """Capacity for path / out_tokens rows: the deepest node's depth + 1."""
    return int(max(_depths(p).max() for p in parents)) + 1
