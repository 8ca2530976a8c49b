"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle.

Integer and index outputs must be bit-exact; attention must be within
max-abs 2e-2 and mean-abs 2e-3 of the double-precision oracle for bfloat16,
and within 1e-5 for float32.  Small cases span several 64-key tiles, several
split-KV chunks, ragged tails, every warp arrangement of the bf16 kernel and
both head sizes; the full-size workloads are checked on every node (the
oracle runs on all host cores) in the launch configuration the benchmark
uses, and the Qwen2-7B-shaped one under both attention schedules.
"""
import os

import numpy as np
import pytest
import torch

import workloads as W
from gpu_util import dev, host_f32, to_device

pytestmark = pytest.mark.gpu

BF16_MAX, BF16_MEAN, F32_MAX = 2e-2, 2e-3, 1e-5


@pytest.fixture(scope="module")
def tv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import eagle_speculative_decoding_parent_gb300 as m
    return m


def random_trees(rng, B, N, max_depth=None):
    out = []
    for _ in range(B):
        par = [-1]
        dep = [0]
        for i in range(1, N):
            cand = [u for u in range(i) if max_depth is None or dep[u] < max_depth]
            u = cand[int(rng.integers(len(cand)))]
            par.append(u)
            dep.append(dep[u] + 1)
        out.append(par)
    return np.array(out, np.int32)


# ------------------------------------------------------------------ mask

@pytest.mark.parametrize("N", [1, 2, 7, 31, 32, 33, 63, 64])
def test_mask_bit_exact(tv, orc, N):
    rng = np.random.default_rng(N)
    par = random_trees(rng, 257, N)
    par[3, N - 1] = N - 1 if N > 1 else 5       # invalid: self / forward parent
    par[7, 0] = 0                                 # invalid root
    mask, depth, status = orc.tree_mask(par)
    m = torch.zeros((257, N), dtype=torch.int64, device="cuda")
    d = torch.zeros((257, N), dtype=torch.int32, device="cuda")
    s = torch.full((257,), -9, dtype=torch.int32, device="cuda")
    tv.tree_mask_build(dev(par), m, d, s)
    assert np.array_equal(m.cpu().numpy().view(np.uint64), mask)
    assert np.array_equal(d.cpu().numpy(), depth)
    assert np.array_equal(s.cpu().numpy(), status)
    assert status[7] == orc.BAD_TREE


def test_mask_host_errors(tv):
    par = torch.zeros((2, 65), dtype=torch.int32, device="cuda")
    m = torch.zeros((2, 65), dtype=torch.int64, device="cuda")
    s = torch.zeros(2, dtype=torch.int32, device="cuda")
    with pytest.raises(tv.TreeVerifyError):
        tv.tree_mask_build(par, m, None, s)


# ------------------------------------------------------------------ attention

def run_attention(tv, w, mask_np=None, scale=0.0, ws_bytes=None):
    """ws_bytes: workspace size (default: the size the library asks for; 256
    selects the schedule without partial results in global memory)."""
    spec = w["spec"]
    d = to_device(w)
    B, N = w["parents"].shape
    mask = torch.from_numpy((mask_np if mask_np is not None else w["_mask"]).view(np.int64)).cuda()
    out = torch.empty_like(d["q"])
    status = torch.full((B,), -9, dtype=torch.int32, device="cuda")
    ws = tv.tree_verify_attention_workspace(B, N, spec.Hq, spec.Hkv, spec.d,
                                            w["block_table"].shape[1], spec.bs, d["q"].dtype)
    if ws_bytes is not None:
        ws = ws_bytes
    wsb = torch.zeros(max(ws, 256), dtype=torch.uint8, device="cuda")
    tv.tree_verify_attention(d["q"], d["k_cache"], d["v_cache"], d["block_table"],
                             d["prefix_lens"], mask, out, status, wsb, scale=scale)
    torch.cuda.synchronize()
    return host_f32(out), status.cpu().numpy(), wsb


def oracle_attention(orc, w, sel=None, scale=0.0):
    spec = w["spec"]
    out, st = orc.attention(w["q"], w["k_cache"], w["v_cache"], w["block_table"],
                            w["prefix_lens"], w["_mask"], bf16=spec.bf16, scale=scale, sel=sel,
                            nthreads=os.cpu_count() or 8)
    return out, st


def small(name, **kw):
    w = W.make(name, parts=("attn",), **kw)
    return w


def with_mask(orc, w):
    w["_mask"] = orc.tree_mask(w["parents"])[0]
    return w


def assert_close_bf16(got, ref):
    err = np.abs(got.astype(np.float64) - ref)
    assert err.max() <= BF16_MAX, err.max()
    assert err.mean() <= BF16_MEAN, err.mean()


def test_attention_f32_tiny_workload(tv, orc):
    w = with_mask(orc, W.make("tiny_fp32", parts=("attn",)))
    got, st, _ = run_attention(tv, w)
    ref, rst = oracle_attention(orc, w)
    assert (st == 0).all() and (rst == 0).all()
    np.testing.assert_allclose(got.reshape(ref.shape), ref, atol=F32_MAX, rtol=0)


@pytest.mark.parametrize("case", [
    # (N, Hq, Hkv, d, bs, P_lo, P_hi, B)  -> packed rows M = N * Hq / Hkv
    # head size 128: tensor-memory kernel (row tiles padded to 128 rows)
    (4, 8, 2, 128, 16, 0, 300, 3),       # M = 16
    (6, 32, 8, 128, 16, 900, 2100, 5),   # M = 24   chain-like
    (13, 8, 2, 128, 32, 64, 700, 4),     # M = 52   block size 32
    (26, 32, 8, 128, 16, 1, 1500, 4),    # M = 104
    (60, 32, 8, 128, 16, 2000, 2100, 1), # M = 240  (two row tiles)
    (63, 28, 4, 128, 16, 700, 1000, 2),  # M = 441  (four row tiles)
    # head size 64: warp-MMA kernel (row warps x key groups)
    (7, 2, 1, 64, 16, 0, 130, 3),        # M = 14   (1 x 8 warps)
    (33, 16, 4, 64, 16, 50, 333, 3),     # M = 132  (several row tiles)
    (6, 32, 8, 64, 16, 900, 2100, 5),    # M = 24   (2 x 4)  chain-like
    (1, 4, 4, 128, 16, 0, 65, 4),        # root only, empty prefix possible
])
def test_attention_bf16_small(tv, orc, case):
    N, Hq, Hkv, d, bs, plo, phi, B = case
    spec = W.Spec("case", B=B, P_lo=plo, P_hi=phi, Hq=Hq, Hkv=Hkv, d=d, V=16, N=N,
                  tree="random", depth=8, branch=4, bs=bs, seed=sum(case))
    w = with_mask(orc, small(spec))
    got, st, wsb = run_attention(tv, w)
    ref, rst = oracle_attention(orc, w)
    assert (st == 0).all() and (rst == 0).all()
    assert_close_bf16(got.reshape(ref.shape), ref)
    # arrival counters are left at zero for the next call
    got2, _, _ = run_attention(tv, w)
    assert np.array_equal(got, got2)


@pytest.mark.parametrize("case", [
    # tensor-core row tiles (M > 64) under both schedules
    (26, 32, 8, 128, 16, 1, 1500, 4),    # M = 104
    (60, 32, 8, 128, 16, 2000, 2100, 1), # M = 240, one sequence over many SMs
    (63, 28, 4, 128, 16, 700, 1000, 2),  # M = 441
    (20, 16, 4, 128, 16, 0, 5000, 9),    # M = 80, very uneven prefixes
    (20, 16, 4, 128, 16, 4000, 5000, 1), # one sequence cut into ~38 pieces per group
    (2, 64, 64, 128, 16, 0, 60, 256),    # G = 1: 16k one-tile groups, ~100 pieces per run
])
@pytest.mark.parametrize("schedule", ["balanced", "clusters", "clusters-small-ws"])
def test_attention_tc_schedules(tv, orc, case, schedule, monkeypatch):
    """The balanced split (forced on, whatever the group count) and the cluster
    schedule (forced, or chosen because the workspace is too small for partial
    results) give the same attention."""
    monkeypatch.setenv("TV_SPLIT", "0" if schedule == "clusters" else "1")
    ws_bytes = 256 if schedule == "clusters-small-ws" else None
    N, Hq, Hkv, d, bs, plo, phi, B = case
    spec = W.Spec("sched", B=B, P_lo=plo, P_hi=phi, Hq=Hq, Hkv=Hkv, d=d, V=16, N=N,
                  tree="random", depth=8, branch=4, bs=bs, seed=7 + sum(case))
    w = with_mask(orc, small(spec))
    got, st, _ = run_attention(tv, w, ws_bytes=ws_bytes)
    ref, rst = oracle_attention(orc, w)
    assert (st == 0).all() and (rst == 0).all()
    assert_close_bf16(got.reshape(ref.shape), ref)
    got2, _, _ = run_attention(tv, w, ws_bytes=ws_bytes)
    assert np.array_equal(got, got2)


def test_attention_tc_balanced_flags_bad_sequences(tv, orc, monkeypatch):
    """Balanced schedule: a sequence with a block id outside the cache and one
    with a negative prefix length get status 3 and zero outputs; the others,
    whose groups are cut into pieces around them, stay exact."""
    monkeypatch.setenv("TV_SPLIT", "1")
    spec = W.Spec("badtc", B=5, P_lo=600, P_hi=3000, Hq=32, Hkv=8, d=128, V=16, N=26,
                  tree="random", depth=6, branch=4, seed=21)
    w = with_mask(orc, small(spec))
    ref, _ = oracle_attention(orc, w)
    w["block_table"] = w["block_table"].copy()
    w["block_table"][1, 3] = w["k_cache"].shape[0] + 1
    w["prefix_lens"] = w["prefix_lens"].copy()
    w["prefix_lens"][3] = -5
    got, st, _ = run_attention(tv, w)
    assert list(st) == [0, orc.OUT_OF_RANGE, 0, orc.OUT_OF_RANGE, 0]
    g = got.reshape(5, spec.N, spec.Hq, spec.d)
    r = ref.reshape(5, spec.N, spec.Hq, spec.d)
    assert (g[1] == 0).all() and (g[3] == 0).all()
    for b in (0, 2, 4):
        assert_close_bf16(g[b], r[b])


def test_attention_kernel_count(tv):
    """The launch count the library reports: the balanced schedule (row tiles
    too few for the SMs, full workspace) adds a merge kernel."""
    bf = torch.bfloat16
    full = tv.tree_verify_attention_workspace(8, 63, 28, 4, 128, 2100, 16, bf)
    assert tv.tree_verify_attention_kernels(8, 63, 28, 4, 128, 2100, 16, bf, full) == 2
    assert tv.tree_verify_attention_kernels(8, 63, 28, 4, 128, 2100, 16, bf, 256) == 1
    assert tv.tree_verify_attention_kernels(1, 60, 32, 8, 128, 200, 16, bf, 1 << 30) == 1
    assert tv.tree_verify_attention_kernels(128, 6, 32, 8, 128, 300, 16, bf, 1 << 30) == 1
    assert tv.tree_verify_attention_kernels(0, 6, 32, 8, 128, 300, 16, bf, 0) == 0


FULL = ["llama3_8b_tree60", "llama3_8b_b32_tree26", "llama3_8b_b128_chain5",
        "qwen2_7b_32k_tree63"]


@pytest.mark.parametrize("name,split", [(n, None) for n in FULL] +
                         [("qwen2_7b_32k_tree63", "0"), ("llama3_8b_b32_tree26", "1")])
def test_attention_full_size_every_node(tv, orc, name, split, monkeypatch):
    """Every node and head of the full-size workloads against the oracle.  The
    Qwen2-7B-shaped batch takes the balanced split by default and is also run
    on the cluster schedule; the batch of 32 is also run on the balanced
    split (so both merges are checked on full outputs)."""
    if split is not None:
        monkeypatch.setenv("TV_SPLIT", split)
    spec = W.SPECS[name]
    w = with_mask(orc, W.make(name, parts=("attn",)))
    got, st, _ = run_attention(tv, w)
    assert (st == 0).all()
    ref, rst = oracle_attention(orc, w)
    assert (rst == 0).all()
    assert_close_bf16(got.reshape(ref.shape), ref)


def test_attention_block_permutation_and_non_ancestor_invariance(tv, orc):
    spec = W.Spec("perm", B=3, P_lo=100, P_hi=700, Hq=16, Hkv=4, d=128, V=16, N=20,
                  tree="random", depth=5, branch=3, seed=11)
    w = with_mask(orc, small(spec))
    base, _, _ = run_attention(tv, w)
    # relocate every physical block
    perm = np.random.default_rng(5).permutation(w["k_cache"].shape[0])
    w2 = dict(w)
    for k in ("k_cache", "v_cache"):
        c = np.empty_like(w[k])
        c[perm] = w[k]
        w2[k] = c
    bt = w["block_table"]
    w2["block_table"] = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1).astype(np.int32)
    moved, _, _ = run_attention(tv, w2)
    assert np.array_equal(base, moved)
    # perturb K/V of tree nodes that are not ancestors of node 5 of sequence 0
    w3 = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in w.items()}
    P = int(w["prefix_lens"][0])
    anc = int(w["_mask"][0, 5])
    bs = spec.bs
    for a in range(spec.N):
        if (anc >> a) & 1:
            continue
        t = P + a
        blk = w["block_table"][0, t // bs]
        for k in ("k_cache", "v_cache"):
            w3[k][blk, :, t % bs, :] = W.f32_to_bf16_bits(
                np.full(spec.d, 3.0 + a, np.float32))
    pert, _, _ = run_attention(tv, w3)
    Hq = spec.Hq
    assert np.array_equal(base.reshape(3, spec.N, Hq, -1)[0, 5], pert.reshape(3, spec.N, Hq, -1)[0, 5])


def test_attention_ignores_nan_past_sequence_end_and_flags_bad_blocks(tv, orc):
    spec = W.Spec("nan", B=3, P_lo=40, P_hi=200, Hq=8, Hkv=2, d=128, V=16, N=9,
                  tree="random", depth=4, branch=3, seed=3)
    w = with_mask(orc, small(spec))
    # cache rows past P+N-1 in each sequence's last block: NaN
    nan_bits = np.uint16(0x7FC0)
    for b in range(3):
        L = int(w["prefix_lens"][b]) + spec.N
        last = w["block_table"][b, (L - 1) // spec.bs]
        for r in range(L % spec.bs if L % spec.bs else spec.bs, spec.bs):
            w["k_cache"][last, :, r, :] = nan_bits
            w["v_cache"][last, :, r, :] = nan_bits
    got, st, _ = run_attention(tv, w)
    ref, _ = oracle_attention(orc, w)
    assert np.isfinite(got).all()
    assert_close_bf16(got.reshape(ref.shape), ref)
    # a block id outside the cache -> status 3, zero output for that sequence only
    w["block_table"] = w["block_table"].copy()
    w["block_table"][1, 0] = w["k_cache"].shape[0] + 7
    got, st, _ = run_attention(tv, w)
    assert list(st) == [0, orc.OUT_OF_RANGE, 0]
    g = got.reshape(3, spec.N, spec.Hq, spec.d)
    assert (g[1] == 0).all() and np.abs(g[0]).sum() > 0


def test_attention_scale_argument(tv, orc):
    spec = W.Spec("scale", B=2, P_lo=10, P_hi=300, Hq=8, Hkv=2, d=128, V=16, N=5,
                  tree="random", depth=3, branch=2, seed=4)
    w = with_mask(orc, small(spec))
    got, _, _ = run_attention(tv, w, scale=0.3)
    ref, _ = oracle_attention(orc, w, scale=0.3)
    assert_close_bf16(got.reshape(ref.shape), ref)


# ------------------------------------------------------------------ acceptance

def run_accept(tv, w, mode, max_path, seed=0, offset=0):
    B, N = w["parents"].shape
    target = dev(w["logits"] if mode == 0 else w["p"])
    draft = None if mode == 0 else dev(w["q_probs"])
    acc = torch.full((B,), -9, dtype=torch.int32, device="cuda")
    path = torch.full((B, max_path), -9, dtype=torch.int32, device="cuda")
    out = torch.full((B, max_path), -9, dtype=torch.int32, device="cuda")
    st = torch.full((B,), -9, dtype=torch.int32, device="cuda")
    V = target.shape[2]
    aws = tv.tree_accept_workspace(mode, B, N, V)
    ws = torch.zeros(max(aws, 256), dtype=torch.uint8, device="cuda")
    tv.tree_accept(mode, dev(w["parents"]), dev(w["draft_tokens"]), target, draft, acc, path,
                   out, st, seed=seed, offset=offset, workspace=ws)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), path.cpu().numpy(), out.cpu().numpy(), st.cpu().numpy()


def assert_same(a, b):
    for x, y in zip(a, b):
        assert np.array_equal(x, y), (x, y)


@pytest.mark.parametrize("name", ["tiny_fp32", "llama3_8b_tree60", "llama3_8b_b32_tree26",
                                  "qwen2_7b_32k_tree63"])
def test_greedy_full_size_bit_exact(tv, orc, name):
    w = W.make(name, parts=("accept",))
    mp = W.max_path_len(w["parents"])
    got = run_accept(tv, w, 0, mp)
    ref = orc.accept_greedy(w["parents"], w["draft_tokens"], w["logits"], mp)
    assert_same(got, ref)
    assert (got[0] == w["planted_accept_len"]).all()


@pytest.mark.parametrize("V", [1, 3, 4, 37, 1000, 4096])
def test_greedy_ties_nans_small_vocab(tv, orc, V):
    rng = np.random.default_rng(V)
    B, N = 300, 12
    par = random_trees(rng, B, N, max_depth=5)
    logits = rng.integers(0, 3, size=(B, N, V)).astype(np.float32)
    logits[rng.random((B, N, V)) < 0.08] = np.nan
    logits[5] = np.nan                                    # every row NaN -> BAD_VALUES
    logits[6, :, :] = -np.inf                             # all -inf: argmax 0
    tok = rng.integers(0, V, size=(B, N)).astype(np.int32)
    tok[9, 3] = V                                          # out of range
    par[11, 4] = 7                                         # bad tree
    w = {"parents": par, "draft_tokens": tok, "logits": logits}
    for mp in (N, 2):
        got = run_accept(tv, w, 0, mp)
        ref = orc.accept_greedy(par, tok, logits, mp)
        assert_same(got, ref)


def test_stochastic_chain_full_size_bit_exact(tv, orc):
    w = W.make("llama3_8b_b128_chain5", parts=("accept",))
    N = w["parents"].shape[1]
    for seed, offset in ((7, 0), (7, 1), (123456789012345, 2**40 + 3)):
        got = run_accept(tv, w, 1, N, seed=seed, offset=offset)
        ref = orc.accept_stochastic(w["parents"], w["draft_tokens"], w["p"], w["q_probs"],
                                    seed, offset, N)
        assert_same(got, ref)


def _chunk_len(V, ch):
    per = -(-V // ch)
    return (per + 3) & ~3


@pytest.mark.parametrize("V", [128256, 152064])
@pytest.mark.parametrize("B,N", [(1, 60), (32, 26)])
def test_greedy_ties_full_vocab(tv, orc, V, B, N):
    """Integer logits at the full vocabularies, so every row's maximum is tied
    many times over: the argmax must be the lowest index ("vLLM EAGLE in
    practice", 无损性保障: greedy verification equals greedy decoding).  Each
    row's first maximum is planted on (or straddling) a boundary of the
    vocabulary pieces the kernels reduce separately: the row scan's chunks
    (one batch-1 tree of 60 nodes) and the level walk's per-CTA slices (a batch
    of 32), for every chunk or cluster count they can take; later maxima
    follow in the pieces after it."""
    rng = np.random.default_rng(V + 7 * B)
    bounds = sorted({c * _chunk_len(V, n) for n in range(2, 33) for c in range(1, n)})
    bounds = [x for x in bounds if 4 <= x < V - 4]
    logits = rng.integers(-3, 3, size=(B, N, V)).astype(np.float32)   # -3 .. 2
    rows = logits.reshape(B * N, V)
    for r in range(B * N):
        s = bounds[(r * 7919) % len(bounds)]
        kind = r % 3
        if kind == 0:
            rows[r, s] = 3.0                                   # first maximum opens a piece
        elif kind == 1:
            rows[r, s - 1] = rows[r, s] = 3.0                  # tie across the boundary
        else:
            rows[r, s - 4:s + 4] = 3.0                         # a run across it
        later = rng.choice(np.arange(s + 4, V), size=16, replace=False)
        rows[r, later] = 3.0                                   # more ties further on
    par = random_trees(rng, B, N, max_depth=6)
    am = np.argmax(logits, axis=2)                             # first maximum of each row
    tok = rng.integers(0, V, size=(B, N)).astype(np.int32)
    for b in range(B):
        for c in range(1, N):
            if rng.random() < 0.75:
                tok[b, c] = am[b, par[b, c]]
    w = {"parents": par, "draft_tokens": tok, "logits": logits}
    mp = W.max_path_len(par)
    got = run_accept(tv, w, 0, mp)
    ref = orc.accept_greedy(par, tok, logits, mp)
    assert_same(got, ref)
    assert (ref[3] == 0).all() and ref[0].max() > 0


def test_accept_row_scan_timeout_then_recovers(tv, orc, monkeypatch):
    """The row scan's waits for streamed data are bounded.  With the test-only
    limit TV_TEST_DATA_WAIT_NS=1 every chunk's first wait runs out: the kernel
    drains the copies it has in flight (those waits keep the full limit) and
    every sequence reports TV_ERR_TIMEOUT (6) with the defined failure outputs.
    The next call without the setting is exact again (the arrival counters
    were left at zero)."""
    rng = np.random.default_rng(5)
    B, N, V = 3, 9, 65536                                      # batch 1-3: the row scan
    par = random_trees(rng, B, N, max_depth=4)
    logits = rng.standard_normal((B, N, V)).astype(np.float32)
    am = np.argmax(logits, axis=2)
    tok = np.array([[am[b, par[b, c]] if c else 0 for c in range(N)] for b in range(B)], np.int32)
    w = {"parents": par, "draft_tokens": tok, "logits": logits}
    mp = W.max_path_len(par)
    monkeypatch.setenv("TV_TEST_DATA_WAIT_NS", "1")
    acc, path, out, st = run_accept(tv, w, 0, mp)
    assert (st == tv.TV_ERR_TIMEOUT).all(), st
    assert (acc == 0).all() and (path[:, 0] == 0).all() and (path[:, 1:] == -1).all()
    assert (out == -1).all()
    monkeypatch.delenv("TV_TEST_DATA_WAIT_NS")
    got = run_accept(tv, w, 0, mp)
    assert_same(got, orc.accept_greedy(par, tok, logits, mp))


@pytest.mark.parametrize("V", [4096, 8196])
def test_stochastic_chain_weight_edge_values(tv, orc, V):
    """Chain acceptance whose residual and target rows hold every class of
    value the fixed-point weight rule separates (infinities, NaN, values at
    and above 1, negative zero, subnormals, values around 2^-40 where the
    weight becomes 0 or 1, and values on 2^-16 boundaries), on rows that take
    the streaming path (16-byte aligned, length a multiple of 4): the draw
    must equal the oracle's bit for bit."""
    rng = np.random.default_rng(V + 1)
    B, N = 48, 3
    p = rng.dirichlet(np.ones(V) * 0.5, size=(B, N)).astype(np.float32)
    q = rng.dirichlet(np.ones(V) * 0.5, size=(B, N)).astype(np.float32)
    tok = rng.integers(0, V, size=(B, N)).astype(np.int32)
    p[np.arange(B), 0, tok[:, 1]] = 0.0                 # the first draft is rejected
    f = np.float32
    sp = np.array([np.inf, np.nan, 2.0, 1.0, f(1) - f(2.0 ** -24), -0.0, 1e-40, 9.0e-13,
                   f(2.0 ** -40), f(2.0 ** -40) * f(1.5), 3e-12, 0.5, f(2.0 ** -16),
                   f(2.0 ** -16) + f(2.0 ** -39), -1.0, -np.inf], np.float32)
    sq = np.array([-np.inf, np.nan, 0.0, 1e-40, -0.0, 0.25, f(2.0 ** -16)], np.float32)
    for b in range(B):
        free = np.setdiff1d(np.arange(V), [tok[b, 1]])
        cols = rng.choice(free, size=sp.size + sq.size + 1, replace=False)
        p[b, 0, cols[: sp.size]] = sp
        q[b, 1, cols[sp.size: -1]] = sq
        p[b, 0, cols[-1]] = q[b, 1, cols[-1]] = np.inf  # inf - inf: NaN residual
        if b % 4 == 0:                                  # residual without mass: target row draw
            q[b, 1, :] = np.maximum(p[b, 0, :], 0) + 1
            q[b, 1, np.isnan(q[b, 1])] = 1.0
    w = {"parents": np.tile(np.arange(-1, N - 1, dtype=np.int32), (B, 1)), "draft_tokens": tok,
         "p": p, "q_probs": q}
    for seed, offset in ((3, 0), (11, 5)):
        got = run_accept(tv, w, 1, N, seed=seed, offset=offset)
        ref = orc.accept_stochastic(w["parents"], tok, p, q, seed, offset, N)
        assert_same(got, ref)


@pytest.mark.parametrize("V", [1, 5, 8, 64, 4099, 50000])
def test_stochastic_accept_paths_small(tv, orc, V):
    """High-acceptance and degenerate draft/target pairs: all-accepted bonus
    draws, zero-mass residuals (fallback to the target row), NaN entries,
    non-chains and out-of-range tokens."""
    rng = np.random.default_rng(V)
    B, N = 400, 6
    p = rng.dirichlet(np.ones(V) * 0.3, size=(B, N)).astype(np.float32)
    q = np.zeros_like(p)
    q[:, 1:] = p[:, :-1]
    mix = rng.random(B) < 0.5                         # half the sequences: perturbed drafts
    q[mix, 1:] = rng.dirichlet(np.ones(V) * 0.3, size=(int(mix.sum()), N - 1)).astype(np.float32)
    tok = np.zeros((B, N), np.int32)
    for b in range(B):
        for k in range(1, N):
            row = q[b, k].astype(np.float64)
            tok[b, k] = rng.choice(V, p=row / row.sum())
    par = np.tile(np.arange(-1, N - 1, dtype=np.int32), (B, 1))
    par[3, 4] = 1                                      # not a chain
    tok[4, 2] = -1                                     # out of range
    p[8, 0, :] = np.nan                                # accept test fails; residual NaN -> 0 mass
    p[9, 0, :] = 0.0                                   # zero-mass target row
    w = {"parents": par, "draft_tokens": tok, "p": p, "q_probs": q}
    got = run_accept(tv, w, 1, N, seed=99, offset=5)
    ref = orc.accept_stochastic(par, tok, p, q, 99, 5, N)
    assert_same(got, ref)
    assert ref[3][3] == orc.OK and ref[3][4] == orc.OUT_OF_RANGE  # a tree is walked
    assert (ref[0][~mix] == N - 1).sum() > 0


def random_tree(rng, N, branch):
    par = np.full(N, -1, np.int32)
    kids = np.zeros(N, int)
    for i in range(1, N):
        cand = [j for j in range(i) if kids[j] < branch]
        par[i] = rng.choice(cand)
        kids[par[i]] += 1
    return par


@pytest.mark.parametrize("V", [8, 4099, 128256])
def test_stochastic_accept_branching_trees(tv, orc, V):
    """Multi-candidate rejection sampling on random trees: accept lengths, paths
    and tokens bit-exact against the oracle, including drafts equal to the
    target (deep acceptance), drafts disjoint from it (every child rejected),
    a NaN target row and a zero-mass target row."""
    rng = np.random.default_rng(V + 3)
    B = 40 if V > 10000 else 300
    N = 12
    par = np.stack([random_tree(rng, N, 3) for _ in range(B)])
    p = rng.dirichlet(np.ones(V) * 0.3, size=(B, N)).astype(np.float32)
    qpar = rng.dirichlet(np.ones(V) * 0.3, size=(B, N)).astype(np.float32)
    q = np.zeros_like(p)
    for b in range(B):
        for c in range(1, N):
            q[b, c] = qpar[b, par[b, c]]
    same = rng.random(B) < 0.3                          # drafts equal to the target
    for b in np.nonzero(same)[0]:
        for c in range(1, N):
            q[b, c] = p[b, par[b, c]]
    tok = np.zeros((B, N), np.int32)
    for b in range(B):
        for c in range(1, N):
            cdf = np.cumsum(q[b, c].astype(np.float64))
            tok[b, c] = min(int(np.searchsorted(cdf / cdf[-1], rng.random())), V - 1)
    if V >= 8:
        p[1, :, : V // 2] = 0.0                          # disjoint supports: reject every child
        p[1] /= p[1].sum(axis=1, keepdims=True)
        q[1, :, V // 2:] = 0.0
        q[1] /= np.maximum(q[1].sum(axis=1, keepdims=True), 1e-30)
        tok[1, 1:] = rng.integers(0, V // 2, size=N - 1)
    p[2, 0, :] = np.nan
    p[3, 0, :] = 0.0
    w = {"parents": par, "draft_tokens": tok, "p": p, "q_probs": q}
    max_path = N
    got = run_accept(tv, w, 1, max_path, seed=21, offset=9)
    ref = orc.accept_stochastic(par, tok, p, q, 21, 9, max_path)
    assert_same(got, ref)
    assert (ref[0][same & (np.arange(B) >= 4)] >= 1).all()
    assert ref[0][3] == 0 and ref[3][3] == orc.BAD_VALUES


# ------------------------------------------------------------------ K/V append

@pytest.mark.parametrize("bf16,theta", [(True, 500000.0), (True, 0.0), (False, 10000.0)])
def test_kv_append_matches_oracle(tv, orc, bf16, theta):
    """Tree K/V rows into the paged cache at P + i, keys rotated by P + depth(i):
    copies bit-exact; rotated keys equal to the oracle's up to one unit in the
    last place of the cache type (double-precision sin/cos/pow of the device and
    of the host library may differ in their last bit); a bad block, a negative
    prefix and a bad depth leave their sequences untouched with status 3."""
    rng = np.random.default_rng(int(theta) % 97 + bf16)
    B, N, Hkv, d, bs = 6, 26, 8, 128, 16
    P = rng.integers(0, 3000, size=B).astype(np.int32)
    nb = [(int(x) + N + bs - 1) // bs for x in P]
    maxb = max(nb)
    perm = rng.permutation(sum(nb) + 4)
    table = np.full((B, maxb), -1, np.int32)
    k = 0
    for b in range(B):
        table[b, :nb[b]] = perm[k:k + nb[b]]
        k += nb[b]
    num_blocks = sum(nb) + 4
    mk = (lambda a: W.f32_to_bf16_bits(a.astype(np.float32))) if bf16 else (lambda a: a.astype(np.float32))
    kc = mk(rng.standard_normal((num_blocks, Hkv, bs, d)))
    vc = mk(rng.standard_normal((num_blocks, Hkv, bs, d)))
    kn = mk(rng.standard_normal((B, N, Hkv, d)) * 3)
    vn = mk(rng.standard_normal((B, N, Hkv, d)))
    depth = np.stack([orc.tree_mask(random_tree(rng, N, 3)[None])[1][0] for _ in range(B)]).astype(np.int32)
    table[1, int(P[1]) // bs] = num_blocks + 2           # bad block
    P[2] = -5                                            # negative prefix
    if theta > 0:
        depth[3, 7] = N                                  # bad depth (rotation only)
    kr, vr = kc.copy(), vc.copy()
    st_ref = orc.tree_kv_append(kn, vn, depth, kr, vr, table, P, rope_theta=theta)
    to = (lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()) if bf16 else \
        (lambda a: torch.from_numpy(a).cuda())
    kd, vd = to(kc), to(vc)
    st = torch.full((B,), -9, dtype=torch.int32, device="cuda")
    tv.tree_kv_append(to(kn), to(vn), dev(depth), kd, vd, dev(table), dev(P), st, rope_theta=theta)
    torch.cuda.synchronize()
    back = (lambda t: t.view(torch.int16).cpu().numpy().view(np.uint16)) if bf16 else \
        (lambda t: t.cpu().numpy())
    kg, vg = back(kd), back(vd)
    assert list(st.cpu().numpy()) == list(st_ref)
    assert st_ref[1] == orc.OUT_OF_RANGE and st_ref[2] == orc.OUT_OF_RANGE
    assert np.array_equal(vg, vr)
    if theta <= 0:
        assert np.array_equal(kg, kr)
        return
    bits = np.uint16 if bf16 else np.uint32
    diff = np.abs(kg.view(bits).astype(np.int64) - kr.view(bits).astype(np.int64))
    assert diff.max() <= 1, diff.max()
    assert (diff > 0).mean() < 1e-3
    assert not np.array_equal(kg, kc)                    # keys were written


# ------------------------------------------------------------------ compaction

def run_compact(tv, k, v, bt, P, path, acc, bf16, num_layers=1, layer_stride=0):
    kd, vd = dev(k, bf16), dev(v, bf16)
    B, mp = path.shape
    nl = torch.full((B,), -9, dtype=torch.int32, device="cuda")
    src = torch.full((B, mp), -9, dtype=torch.int64, device="cuda")
    dst = torch.full((B, mp), -9, dtype=torch.int64, device="cuda")
    st = torch.full((B,), -9, dtype=torch.int32, device="cuda")
    tv.kv_compact(kd, vd, dev(bt), dev(P), dev(path), dev(acc), nl, st, src_slots=src,
                  dst_slots=dst, num_layers=num_layers, layer_stride=layer_stride)
    torch.cuda.synchronize()
    view = (lambda t: t.view(torch.int16).cpu().numpy().view(np.uint16)) if bf16 else \
        (lambda t: t.cpu().numpy())
    return view(kd), view(vd), nl.cpu().numpy(), src.cpu().numpy(), dst.cpu().numpy(), \
        st.cpu().numpy()


@pytest.mark.parametrize("bf16,num_layers", [(True, 1), (True, 3), (False, 1)])
def test_compaction_bit_exact(tv, orc, bf16, num_layers):
    rng = np.random.default_rng(num_layers)
    B, Hkv, d, bs, N = 6, 4, 128, 16, 30
    P = rng.integers(0, 200, size=B).astype(np.int32)
    nb = [(int(x) + N + bs - 1) // bs for x in P]
    perm = rng.permutation(sum(nb))
    bt = np.full((B, max(nb)), -1, np.int32)
    o = 0
    for b in range(B):
        bt[b, :nb[b]] = perm[o:o + nb[b]]
        o += nb[b]
    dt = np.uint16 if bf16 else np.float32
    shape = (num_layers, sum(nb), Hkv, bs, d)
    k = rng.integers(0, 60000, size=shape).astype(dt) if bf16 else rng.standard_normal(shape).astype(dt)
    v = rng.integers(0, 60000, size=shape).astype(dt) if bf16 else rng.standard_normal(shape).astype(dt)
    max_path = 9
    par = random_trees(rng, B, N, max_depth=max_path - 1)
    # accepted paths: root path of a random node, from the oracle's own walk
    path = np.full((B, max_path), -1, np.int32)
    acc = np.zeros(B, np.int32)
    for b in range(B):
        c = int(rng.integers(N))
        chain = [c]
        while par[b, chain[-1]] >= 0:
            chain.append(int(par[b, chain[-1]]))
        chain = chain[::-1]
        acc[b] = len(chain) - 1
        path[b, :len(chain)] = chain
    acc[2] = max_path          # out of range -> status 3, untouched
    stride = int(np.prod(shape[1:]))
    got = run_compact(tv, k, v, bt, P, path, acc, bf16, num_layers, stride)
    kr, vr = k.copy(), v.copy()
    ref = orc.kv_compact(kr, vr, bt, P, path, acc, num_layers=num_layers, layer_stride=stride)
    assert np.array_equal(got[0], kr) and np.array_equal(got[1], vr)
    assert_same(got[2:], ref)
    assert ref[3][2] == orc.OUT_OF_RANGE


# ------------------------------------------------------------------ whole step

@pytest.mark.parametrize("name", ["llama3_8b_tree60", "llama3_8b_b128_chain5"])
def test_graph_replay_matches_eager_step(tv, name):
    """The step captured as a CUDA graph and replayed gives the same outputs and
    cache contents, bit for bit, as the eager step on the same inputs."""
    from eagle_speculative_decoding_parent_gb300.pipeline import VerifyStep
    spec = W.SPECS[name]
    w = W.make(name)
    B, N = w["parents"].shape
    mp = W.max_path_len(w["parents"])
    mode = 0 if spec.mode == "greedy" else 1

    def fresh():
        return to_device(w)

    def make_step(d):
        return VerifyStep(B=B, N=N, Hq=spec.Hq, Hkv=spec.Hkv, d=spec.d,
                          max_blocks=w["block_table"].shape[1], bs=spec.bs, dtype=d["q"].dtype,
                          max_path=mp, V=spec.V, mode=mode)

    def args(d):
        return dict(parents=d["parents"], q=d["q"], k_cache=d["k_cache"], v_cache=d["v_cache"],
                    block_table=d["block_table"], prefix_lens=d["prefix_lens"],
                    draft_tokens=d["draft_tokens"], target=d["logits"] if mode == 0 else d["p"],
                    draft_probs=None if mode == 0 else d["q_probs"], mode=mode,
                    seed=w.get("seed", 0), offset=w.get("offset", 0))

    def outputs(st, d):
        torch.cuda.synchronize()
        return [t.cpu().clone() for t in (st.out, st.accept_len, st.path, st.out_tokens,
                                          st.new_lens, d["k_cache"], d["v_cache"])]

    d1 = fresh()
    s1 = make_step(d1)
    s1.run(**args(d1))
    ref = outputs(s1, d1)
    d2 = fresh()
    s2 = make_step(d2)
    graph = s2.capture(**args(d2))      # one eager step, then the recording
    orig = fresh()
    d2["k_cache"].copy_(orig["k_cache"])  # undo that step's compaction, same addresses
    d2["v_cache"].copy_(orig["v_cache"])
    graph.replay()
    got = outputs(s2, d2)
    for a, b in zip(ref, got):
        assert torch.equal(a.view(torch.uint8) if a.dtype == torch.bfloat16 else a,
                           b.view(torch.uint8) if b.dtype == torch.bfloat16 else b)


@pytest.mark.parametrize("name", list(W.SPECS))
def test_full_step_matches_oracle(tv, orc, name):
    """mask -> attention -> accept -> compaction on the GPU, each output
    compared with the oracle run on the same inputs."""
    from eagle_speculative_decoding_parent_gb300.pipeline import VerifyStep
    spec = W.SPECS[name]
    w = W.make(name)
    B, N = w["parents"].shape
    mp = W.max_path_len(w["parents"])
    d = to_device(w)
    dtype = d["q"].dtype
    mode = 0 if spec.mode == "greedy" else 1
    step = VerifyStep(B=B, N=N, Hq=spec.Hq, Hkv=spec.Hkv, d=spec.d,
                      max_blocks=w["block_table"].shape[1], bs=spec.bs, dtype=dtype, max_path=mp,
                      V=spec.V, mode=mode)
    step.run(parents=d["parents"], q=d["q"], k_cache=d["k_cache"], v_cache=d["v_cache"],
             block_table=d["block_table"], prefix_lens=d["prefix_lens"],
             draft_tokens=d["draft_tokens"], target=d["logits"] if mode == 0 else d["p"],
             draft_probs=None if mode == 0 else d["q_probs"], mode=mode,
             seed=w.get("seed", 0), offset=w.get("offset", 0))
    torch.cuda.synchronize()
    mask, depth, mst = orc.tree_mask(w["parents"])
    assert np.array_equal(step.mask.cpu().numpy().view(np.uint64), mask)
    assert np.array_equal(step.depth.cpu().numpy(), depth)
    w["_mask"] = mask
    ref_o, _ = oracle_attention(orc, w)                 # every node
    got_o = host_f32(step.out).reshape(ref_o.shape)
    if spec.bf16:
        assert_close_bf16(got_o, ref_o)
    else:
        np.testing.assert_allclose(got_o, ref_o, atol=F32_MAX, rtol=0)
    if mode == 0:
        ref_a = orc.accept_greedy(w["parents"], w["draft_tokens"], w["logits"], mp)
    else:
        ref_a = orc.accept_stochastic(w["parents"], w["draft_tokens"], w["p"], w["q_probs"],
                                      w["seed"], w["offset"], mp)
    got_a = (step.accept_len.cpu().numpy(), step.path.cpu().numpy(),
             step.out_tokens.cpu().numpy(), step.st_accept.cpu().numpy())
    assert_same(got_a, ref_a)
    kr, vr = w["k_cache"].copy(), w["v_cache"].copy()
    ref_c = orc.kv_compact(kr, vr, w["block_table"], w["prefix_lens"], ref_a[1], ref_a[0])
    got_c = (step.new_lens.cpu().numpy(), step.src_slots.cpu().numpy(),
             step.dst_slots.cpu().numpy(), step.st_compact.cpu().numpy())
    assert_same(got_c, ref_c)
    view = (lambda t: t.view(torch.int16).cpu().numpy().view(np.uint16)) if spec.bf16 else \
        (lambda t: t.cpu().numpy())
    assert np.array_equal(view(d["k_cache"]), kr)
    assert np.array_equal(view(d["v_cache"]), vr)
