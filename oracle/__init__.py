"""CPU oracle for EAGLE draft-tree verification — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never does, and
this package imports nothing from the product.

The arithmetic lives in ``oracle.c`` (plain C, double precision); this module
only marshals numpy arrays into it.  ``build()`` compiles it with gcc.

Parity status of each function (the pins are in ``tests/test_oracle_*.py``):
  tree_mask         pinned (brute-force ancestor walks over every tree N <= 7,
                    hand-worked golden fixture)
  attention         pinned (torch SDPA with an explicit boolean mask, chain ==
                    sequential causal decode, closed forms, block permutation)
  accept_greedy     pinned (enumeration of root paths with numpy nanargmax,
                    golden fixture)
  accept_stochastic pinned (Philox4x32-10 known-answer vectors, empirical
                    target-distribution test, degenerate cases, exhaustive
                    integer-CDF check)
  kv_compact        pinned (torch index_select + narrow + copy_, the operation
                    the KVCache.copy passage describes)
  tree_kv_append    pinned (closed-form rotations, plain copies, error cases)
  ragged node counts (counts= on tree_mask, attention, accept_*, tree_kv_append)
                    pinned (a ragged batch equals the dense functions on the
                    batch cut to each count, sequence indices kept; junk in
                    absent slots, absent K/V rows and blocks, and mask bits
                    above a count change nothing)
  draft_tree        pinned (exhaustive enumeration of every token path when no
                    pruning can bite, greedy-chain and one-layer closed forms,
                    per-layer frontier / final cut recomputed with numpy and
                    scipy on a path-keyed draft model, hand-worked fixture,
                    tie and breadth-first-label cases)
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None

OK, BAD_TREE, OUT_OF_RANGE, UNSUPPORTED, BAD_VALUES = 0, 2, 3, 4, 7


def build(force: bool = False) -> str:
    """Compile oracle.c into _build/liboracle.so (gcc, OpenMP, no fast-math)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
           "-ffp-contract=off", "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = ctypes.CDLL(build())
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


I64 = ctypes.c_int64


def _counts(counts, B):
    return None if counts is None else _c(counts, np.int32).reshape(B)


def tree_mask(parents, counts=None):
    """parents int32 [B, N] -> (mask uint64 [B, N], depth int32 [B, N], status int32 [B]).
    counts int32 [B] (optional): node count of each tree; the rest are absent."""
    lib = _load()
    parents = _c(parents, np.int32)
    B, N = parents.shape
    mask = np.zeros((B, N), np.uint64)
    depth = np.zeros((B, N), np.int32)
    status = np.zeros(B, np.int32)
    cnt = _counts(counts, B)
    lib.orc_tree_mask(_p(parents), I64(B), I64(N), _p(mask), _p(depth), _p(status), _p(cnt))
    return mask, depth, status


def attention(q, k_cache, v_cache, block_table, prefix_lens, mask, *, bf16: bool,
              scale: float = 0.0, sel=None, nthreads: int = 1, counts=None):
    """Tree-masked paged GQA attention in double precision.

    q: [B, N, Hq, d]; k_cache/v_cache: [num_blocks, Hkv, bs, d]; both float32,
    or uint16 bfloat16 bit patterns when ``bf16``.  ``sel``: flat node indices
    b*N+i to evaluate (None: all).  Returns (out float64 [n, Hq, d], status).
    """
    lib = _load()
    dt = np.uint16 if bf16 else np.float32
    q = _c(q, dt)
    k_cache = _c(k_cache, dt)
    v_cache = _c(v_cache, dt)
    block_table = _c(block_table, np.int32)
    prefix_lens = _c(prefix_lens, np.int32)
    mask = _c(mask, np.uint64)
    B, N, Hq, d = q.shape
    num_blocks, Hkv, bs, d2 = k_cache.shape
    assert d2 == d and v_cache.shape == k_cache.shape
    sel_arr = None if sel is None else _c(sel, np.int64)
    n = B * N if sel is None else len(sel_arr)
    out = np.zeros((n, Hq, d), np.float64)
    status = np.zeros(B, np.int32)
    lib.orc_attention(ctypes.c_int(1 if bf16 else 0), _p(q), _p(k_cache), _p(v_cache),
                      _p(block_table), I64(block_table.shape[1]), _p(prefix_lens), _p(mask),
                      I64(B), I64(N), I64(Hq), I64(Hkv), I64(d), I64(bs), I64(num_blocks),
                      ctypes.c_double(scale), _p(sel_arr), I64(0 if sel is None else n),
                      _p(out), _p(status), ctypes.c_int(nthreads), _p(_counts(counts, B)))
    return out, status


def accept_greedy(parents, tokens, logits, max_path, counts=None):
    """Greedy acceptance -> (accept_len [B], path [B, max_path], out_tokens, status)."""
    lib = _load()
    parents = _c(parents, np.int32)
    tokens = _c(tokens, np.int32)
    logits = _c(logits, np.float32)
    B, N, V = logits.shape
    acc = np.zeros(B, np.int32)
    path = np.zeros((B, max_path), np.int32)
    out = np.zeros((B, max_path), np.int32)
    status = np.zeros(B, np.int32)
    lib.orc_accept_greedy(_p(parents), _p(tokens), _p(logits), I64(B), I64(N), I64(V),
                          I64(max_path), _p(acc), _p(path), _p(out), _p(status),
                          _p(_counts(counts, B)))
    return acc, path, out, status


def accept_stochastic(parents, tokens, p, q, seed, offset, max_path, counts=None):
    """Chain rejection sampling -> (accept_len, path, out_tokens, status)."""
    lib = _load()
    parents = _c(parents, np.int32)
    tokens = _c(tokens, np.int32)
    p = _c(p, np.float32)
    q = _c(q, np.float32)
    B, N, V = p.shape
    acc = np.zeros(B, np.int32)
    path = np.zeros((B, max_path), np.int32)
    out = np.zeros((B, max_path), np.int32)
    status = np.zeros(B, np.int32)
    lib.orc_accept_stochastic(_p(parents), _p(tokens), _p(p), _p(q), I64(B), I64(N), I64(V),
                              ctypes.c_uint64(seed), ctypes.c_uint64(offset), I64(max_path),
                              _p(acc), _p(path), _p(out), _p(status), _p(_counts(counts, B)))
    return acc, path, out, status


def accept_stochastic_tree(parents, tokens, p, q, seed, offset, max_path):
    """The branching-tree rule applied to every sequence, chains included (the
    public accept_stochastic takes the chain rule for chains) -> same outputs."""
    lib = _load()
    parents = _c(parents, np.int32)
    tokens = _c(tokens, np.int32)
    p = _c(p, np.float32)
    q = _c(q, np.float32)
    B, N, V = p.shape
    acc = np.zeros(B, np.int32)
    path = np.zeros((B, max_path), np.int32)
    out = np.zeros((B, max_path), np.int32)
    status = np.zeros(B, np.int32)
    for b in range(B):
        lib.orc_accept_stochastic_tree(
            _p(parents[b]), _p(tokens[b]), _p(p[b]), _p(q[b]), I64(1), I64(N), I64(V),
            ctypes.c_uint64(seed), ctypes.c_uint64(offset), I64(max_path), _p(acc[b:]),
            _p(path[b]), _p(out[b]), _p(status[b:]), I64(b))
    return acc, path, out, status


def tree_kv_append(k_new, v_new, depth, k_cache, v_cache, block_table, prefix_lens,
                   rope_theta=0.0, counts=None):
    """In-place append of the tree's K/V rows into numpy caches -> status.

    k_new / v_new [B][N][Hkv][d] and the caches [num_blocks][Hkv][bs][d] are
    float32 arrays or bfloat16 bit patterns (uint16)."""
    lib = _load()
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    elem = 1 if k_cache.dtype == np.uint16 else 0
    k_new = np.ascontiguousarray(k_new)
    v_new = np.ascontiguousarray(v_new)
    B, N, Hkv, d = k_new.shape
    num_blocks, _, bs, _ = k_cache.shape
    block_table = _c(block_table, np.int32)
    prefix_lens = _c(prefix_lens, np.int32)
    dep = _c(depth, np.int32) if depth is not None else np.zeros((B, N), np.int32)
    status = np.zeros(B, np.int32)
    lib.orc_tree_kv_append(I64(elem), _p(k_new), _p(v_new), _p(dep), I64(B), I64(N), I64(Hkv),
                           I64(d), ctypes.c_double(rope_theta), _p(k_cache), _p(v_cache),
                           _p(block_table), I64(block_table.shape[1]), _p(prefix_lens), I64(bs),
                           I64(num_blocks), _p(status), _p(_counts(counts, B)))
    return status


def philox4x32_10(counter, key):
    """One Philox4x32-10 block: counter 4 x uint32, key 2 x uint32 -> 4 x uint32."""
    lib = _load()
    c = np.asarray(counter, np.uint32)
    k = np.asarray(key, np.uint32)
    o = np.zeros(4, np.uint32)
    lib.orc_philox4x32_10(_p(c), _p(k), _p(o))
    return o


def sample_weights(w, x):
    """Integer-CDF sampler: index t with probability w_t / sum(w) for uniform 32-bit x."""
    lib = _load()
    w = _c(w, np.uint64)
    lib.orc_sample_weights_u32.restype = ctypes.c_int64
    return int(lib.orc_sample_weights_u32(_p(w), I64(len(w)), ctypes.c_uint32(x)))


def kv_compact(k_cache, v_cache, block_table, prefix_lens, path, accept_len, *,
               num_layers=1, layer_stride=0):
    """In-place compaction of the numpy caches -> (new_lens, src_slots, dst_slots, status).

    Caches are [num_layers?][num_blocks, Hkv, bs, d] arrays of any 2- or
    4-byte element type; with num_layers > 1 the caches hold the layers back to
    back with ``layer_stride`` elements between them.
    """
    lib = _load()
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    block_table = _c(block_table, np.int32)
    prefix_lens = _c(prefix_lens, np.int32)
    path = _c(path, np.int32)
    accept_len = _c(accept_len, np.int32)
    num_blocks, Hkv, bs, d = k_cache.shape[-4:]
    B, max_path = path.shape
    new_lens = np.zeros(B, np.int32)
    src = np.zeros((B, max_path), np.int64)
    dst = np.zeros((B, max_path), np.int64)
    status = np.zeros(B, np.int32)
    lib.orc_kv_compact(I64(k_cache.itemsize), _p(k_cache), _p(v_cache), I64(num_layers),
                       I64(layer_stride), _p(block_table), I64(block_table.shape[1]),
                       _p(prefix_lens), _p(path), _p(accept_len), I64(max_path), I64(B),
                       I64(Hkv), I64(d), I64(bs), I64(num_blocks), _p(new_lens), _p(src),
                       _p(dst), _p(status))
    return new_lens, src, dst, status


class DraftTree:
    """Draft-tree construction for one sequence, one layer per ``expand`` call
    (the draft model runs between layers on the frontier the call returns).

    Node 0 is the root (``root_token``, score 0).  ``expand(rows)`` takes the
    draft logits float32 [F, V] of the current frontier (F = 1 at the first
    layer, the root) and returns (front_tokens, front_src): the next frontier
    best first, and for each entry the row it was drawn from.  ``finalize(N)``
    returns (parents int32 [N], tokens int32 [N], scores float64 [N], status).
    ``margin`` is the smallest score gap behind any ranking decision so far.
    """

    def __init__(self, root_token: int, V: int, k: int, layers: int):
        self.V, self.k, self.layers = V, k, layers
        cap = 1 + k + max(0, layers - 1) * k * k
        self.tok = np.zeros(cap, np.int32)
        self.par = np.full(cap, -1, np.int32)
        self.score = np.zeros(cap, np.float64)
        self.tok[0] = root_token
        self.count = 1
        self.front = np.zeros(1, np.int32)
        self.margin = np.inf
        self.status = OK

    def front_paths(self):
        """Token path (root token excluded) of every frontier node."""
        out = []
        for u in self.front:
            p = []
            while u > 0:
                p.append(int(self.tok[u]))
                u = self.par[u]
            out.append(tuple(reversed(p)))
        return out

    def expand(self, rows):
        lib = _load()
        rows = _c(rows, np.float32)
        F = len(self.front)
        assert rows.shape == (F, self.V)
        nf = min(self.k, F * self.k)
        new_front = np.zeros(nf, np.int32)
        new_src = np.zeros(nf, np.int32)
        m = ctypes.c_double(self.margin)
        st = lib.orc_draft_expand(I64(self.V), I64(self.k), I64(F), _p(rows), _p(self.front),
                                  _p(self.tok), _p(self.par), _p(self.score),
                                  I64(self.count), _p(new_front), _p(new_src), ctypes.byref(m))
        if st != OK:
            self.status = st
            return None, None
        self.margin = m.value
        self.count += F * self.k
        self.front = new_front
        return self.tok[new_front].copy(), new_src

    def finalize(self, N: int):
        lib = _load()
        parents = np.full(N, -1, np.int32)
        tokens = np.full(N, -1, np.int32)
        scores = np.full(N, -np.inf, np.float64)
        if self.status != OK:
            return parents, tokens, scores, self.status
        m = ctypes.c_double(self.margin)
        st = lib.orc_draft_finalize(I64(self.count), _p(self.tok), _p(self.par), _p(self.score),
                                    I64(N), _p(parents), _p(tokens), _p(scores), ctypes.byref(m))
        self.margin = m.value
        return parents, tokens, scores, st


def draft_tree(rows_per_layer, root_tokens, k: int, N: int):
    """Batch driver: rows_per_layer[l] float32 [B, F_l, V] (F_0 = 1, then k),
    rows in the order of the previous layer's frontier.  Returns (parents
    [B, N], tokens [B, N], scores [B, N] float64, fronts, status [B], margin [B])
    with fronts[l] = (front_tokens [B, k], front_src [B, k]), -1 where a
    sequence failed."""
    B = len(root_tokens)
    L = len(rows_per_layer)
    V = rows_per_layer[0].shape[-1]
    trees = [DraftTree(int(root_tokens[b]), V, k, L) for b in range(B)]
    fronts = []
    for rows in rows_per_layer:
        ft = np.full((B, k), -1, np.int32)
        fs = np.full((B, k), -1, np.int32)
        for b, t in enumerate(trees):
            if t.status != OK:
                continue
            a, s = t.expand(rows[b])
            if a is not None:
                ft[b, :len(a)], fs[b, :len(s)] = a, s
        fronts.append((ft, fs))
    out = [t.finalize(N) for t in trees]
    parents = np.stack([o[0] for o in out])
    tokens = np.stack([o[1] for o in out])
    scores = np.stack([o[2] for o in out])
    status = np.array([o[3] for o in out], np.int32)
    margin = np.array([t.margin for t in trees])
    return parents, tokens, scores, fronts, status, margin
