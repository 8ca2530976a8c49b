"""GPU parity of draft-tree construction: draft_tree_expand (through the C ABI)
against the oracle, layer by layer, on seeded synthetic draft logits.

The top-k of every row is decided by exact comparisons of fp32 logits on both
sides, so it must match bit for bit.  Scores are cumulative log-probabilities
formed in binary32 on both sides; the logsumexp they subtract is reduced in
binary32 in the kernel's order and accumulated in double then rounded once in
the oracle (the two agree within about 1e-6 per row at these vocabulary
sizes), so the scores must agree within SCORE_TOL.  The frontier and the final cut rank those
scores, so a sequence is compared exactly (frontiers, parents, tokens) when
every ranking gap the oracle saw is at least EXACT_MARGIN; a sequence with a
closer call may legitimately break it the other way, and for it the test
checks that the tree is a valid breadth-first draft tree whose sorted scores
match the oracle's.  Rows are indexed by frontier position, so such a swap
changes parent scores by less than the gap and leaves the score multiset
within tolerance.

"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

SCORE_TOL = 1e-4
EXACT_MARGIN = 3e-4


@pytest.fixture(scope="module")
def tv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import eagle_speculative_decoding_parent_gb300 as m
    return m


def draft_rows(seed, B, V, k, L, sigma=3.0):
    rng = np.random.default_rng(seed)
    return [(sigma * rng.standard_normal((B, 1 if l == 0 else k, V))).astype(np.float32)
            for l in range(L)]


def run_gpu(tv, rows, roots, k, N, ws=None):
    B, L = len(roots), len(rows)
    dev = torch.device("cuda")
    if ws is None:
        ws = torch.zeros(tv.draft_tree_workspace(B, k, L), dtype=torch.uint8, device=dev)
    status = torch.full((B,), -7, dtype=torch.int32, device=dev)
    root_t = torch.from_numpy(np.asarray(roots, np.int32)).to(dev)
    parents = torch.full((B, N), -7, dtype=torch.int32, device=dev)
    tokens = torch.full((B, N), -7, dtype=torch.int32, device=dev)
    scores = torch.full((B, N), 7.0, dtype=torch.float32, device=dev)
    fronts = []
    for layer, r in enumerate(rows):
        ft = torch.full((B, k), -7, dtype=torch.int32, device=dev)
        fs = torch.full((B, k), -7, dtype=torch.int32, device=dev)
        last = layer == L - 1
        tv.draft_tree_expand(torch.from_numpy(r).to(dev), layer, L, status, ws, topk=k,
                             root_tokens=root_t, N=N, front_tokens=ft, front_src=fs,
                             parents=parents if last else None, tokens=tokens if last else None,
                             scores=scores if last else None)
        fronts.append((ft, fs))
    torch.cuda.synchronize()
    fronts = [(a.cpu().numpy(), s.cpu().numpy()) for a, s in fronts]
    return (parents.cpu().numpy(), tokens.cpu().numpy(), scores.cpu().numpy(), fronts,
            status.cpu().numpy())


def check_valid_tree(par, tok, sc, V, k, L, root):
    N = len(par)
    assert par[0] == -1 and tok[0] == root and sc[0] == 0.0
    dep = [0] * N
    for i in range(1, N):
        assert 0 <= par[i] < i and 0 <= tok[i] < V
        dep[i] = dep[par[i]] + 1
        assert dep[i] <= L and sc[i] <= sc[par[i]]
    assert all(par[i] <= par[i + 1] for i in range(1, N - 1))      # breadth-first
    for i in range(1, N - 1):
        if par[i] == par[i + 1]:
            assert sc[i] >= sc[i + 1]
    for u in range(N):
        assert sum(1 for i in range(1, N) if par[i] == u) <= k


def compare(tv, orc, rows, roots, k, N, min_exact=1):
    B, L, V = len(roots), len(rows), rows[0].shape[-1]
    gp, gt, gs, gf, gst = run_gpu(tv, rows, roots, k, N)
    op, ot, osc, of, ost, margin = orc.draft_tree(rows, roots, k, N)
    assert (gst == ost).all(), (gst, ost)
    exact = 0
    for b in range(B):
        if ost[b] != 0:
            assert (gp[b] == -1).all() and (gt[b] == -1).all() and (gs[b] == -np.inf).all()
            continue
        if margin[b] >= EXACT_MARGIN:
            exact += 1
            for layer in range(L):
                assert (gf[layer][0][b] == of[layer][0][b]).all(), (b, layer)
                assert (gf[layer][1][b] == of[layer][1][b]).all(), (b, layer)
            assert (gp[b] == op[b]).all() and (gt[b] == ot[b]).all(), b
            assert np.abs(gs[b].astype(np.float64) - osc[b]).max() <= SCORE_TOL, b
        else:
            check_valid_tree(gp[b], gt[b], gs[b], V, k, L, roots[b])
            assert np.abs(np.sort(gs[b].astype(np.float64)) - np.sort(osc[b])).max() <= 1e-3
    assert exact >= min_exact
    return exact


SMALL = [  # B, V, topk, layers, N, seed (chunks hold at least 16384 logits)
    (3, 1000, 4, 4, 20, 1),     # 16-byte loads, one chunk per row
    (2, 1001, 3, 3, 13, 2),     # odd vocabulary: scalar loads
    (4, 50000, 8, 3, 64, 3),    # 8-entry lists, several chunks
    (2, 3000, 10, 2, 64, 4),    # 16-entry lists for k = 10
    (2, 40000, 16, 2, 64, 5),   # k = 16, three chunks, ragged tail
    (2, 40001, 4, 2, 16, 10),   # scalar loads over three chunks
    (2, 777, 1, 6, 7, 6),       # k = 1: the greedy chain
    (2, 500, 5, 1, 6, 7),       # one layer: expand and finish in one call
    (3, 64, 4, 3, 1, 8),        # N = 1: the root alone
    (2, 4096, 2, 5, 19, 9),     # N = every created node
]


@pytest.mark.parametrize("B,V,k,L,N,seed", SMALL)
def test_draft_tree_matches_oracle(tv, orc, B, V, k, L, N, seed):
    rows = draft_rows(seed, B, V, k, L)
    roots = (np.arange(B) * 7 + 3) % V
    compare(tv, orc, rows, roots, k, N)


FULL = [  # B, V, topk, layers, N, seed: Llama-3 / Qwen2 vocabularies
    (1, 128256, 4, 6, 60, 21),  # batch 1, the 60-node EAGLE-2 shape
    (32, 128256, 4, 6, 26, 22),
    (8, 152064, 8, 6, 63, 23),
]


@pytest.mark.parametrize("B,V,k,L,N,seed", FULL)
def test_draft_tree_full_vocabulary(tv, orc, B, V, k, L, N, seed):
    rows = draft_rows(seed, B, V, k, L)
    roots = (np.arange(B) * 7919 + 11) % V
    compare(tv, orc, rows, roots, k, N, min_exact=1)


def test_draft_tree_ties_and_minus_infinity(tv, orc):
    """Integer logits (many exact ties, decided by token id and creation order)
    and rows that are mostly -inf."""
    B, V, k, L, N = 4, 300, 4, 3, 15
    rng = np.random.default_rng(31)
    rows = [rng.integers(-3, 4, size=(B, 1 if l == 0 else k, V)).astype(np.float32)
            for l in range(L)]
    for r in rows:
        r[1][:, 10:] = -np.inf
    roots = np.array([0, 1, 2, 3])
    gp, gt, gs, gf, gst = run_gpu(tv, rows, roots, k, N)
    op, ot, osc, of, ost, margin = orc.draft_tree(rows, roots, k, N)
    assert (gst == ost).all() and (ost == 0).all()
    for b in range(B):
        # the first layer's candidates tie only by token id: exact on both sides
        assert (gf[0][0][b] == of[0][0][b]).all()
        check_valid_tree(gp[b], gt[b], gs[b], V, k, L, roots[b])
        assert np.abs(np.sort(gs[b].astype(np.float64)) - np.sort(osc[b])).max() <= 1e-3
        if margin[b] >= EXACT_MARGIN:
            assert (gp[b] == op[b]).all() and (gt[b] == ot[b]).all()


def test_draft_tree_errors_are_per_sequence(tv, orc):
    B, V, k, L, N = 4, 2000, 4, 3, 12
    rows = draft_rows(41, B, V, k, L)
    rows[1][1, 2, 77] = np.nan        # sequence 1: NaN at layer 1
    rows[2][2, 0, 5] = np.inf         # sequence 2: +inf at layer 2
    roots = np.array([5, 6, 7, V])    # sequence 3: root token out of range
    gp, gt, gs, gf, gst = run_gpu(tv, rows, roots, k, N)
    assert list(gst) == [0, 7, 7, 3]
    op, ot, osc, of, ost, margin = orc.draft_tree(rows[:], np.minimum(roots, V - 1), k, N)
    if margin[0] >= EXACT_MARGIN:
        assert (gp[0] == op[0]).all() and (gt[0] == ot[0]).all()
    for b in (1, 2, 3):
        assert (gp[b] == -1).all() and (gt[b] == -1).all() and (gs[b] == -np.inf).all()
    assert (gf[1][0][1] == -1).all() and (gf[2][0][2] == -1).all() and (gf[0][0][3] == -1).all()


def test_draft_tree_workspace_reuse_and_order_check(tv, orc):
    """The arrival counters return to zero, so one workspace serves tree after
    tree; a layer issued without the previous one is reported, not guessed."""
    B, V, k, L, N = 2, 3000, 3, 3, 10
    ws = torch.zeros(tv.draft_tree_workspace(B, k, L), dtype=torch.uint8, device="cuda")
    for seed in (51, 52):
        rows = draft_rows(seed, B, V, k, L)
        roots = np.array([1, 2])
        gp, gt, gs, gf, gst = run_gpu(tv, rows, roots, k, N, ws=ws)
        op, ot, osc, of, ost, margin = orc.draft_tree(rows, roots, k, N)
        assert (gst == 0).all()
        for b in range(B):
            if margin[b] >= EXACT_MARGIN:
                assert (gp[b] == op[b]).all() and (gt[b] == ot[b]).all()
    assert (ws[:256].cpu().numpy() == 0).all()          # counters back at zero
    fresh = torch.zeros_like(ws)
    status = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    rows = torch.from_numpy(draft_rows(53, B, V, k, L)[1]).cuda()
    tv.draft_tree_expand(rows, 1, L, status, fresh, topk=k)
    torch.cuda.synchronize()
    assert (status.cpu().numpy() == 8).all()             # no layer-0 state: TV_ERR_WORKSPACE


def test_draft_tree_feeds_the_verification_step(tv, orc):
    """The tree this call writes is what tree_mask_build takes: topological,
    root first.  Its mask and depths equal the oracle's for the same parents."""
    B, V, k, L, N = 4, 2048, 4, 5, 48
    rows = draft_rows(61, B, V, k, L)
    roots = np.array([1, 2, 3, 4])
    gp, gt, gs, gf, gst = run_gpu(tv, rows, roots, k, N)
    assert (gst == 0).all()
    par = torch.from_numpy(gp).cuda()
    mask = torch.zeros((B, N), dtype=torch.int64, device="cuda")
    depth = torch.zeros((B, N), dtype=torch.int32, device="cuda")
    status = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    tv.tree_mask_build(par, mask, depth, status)
    torch.cuda.synchronize()
    om, od, ost = orc.tree_mask(gp)
    assert (status.cpu().numpy() == 0).all() and (ost == 0).all()
    assert (mask.cpu().numpy().view(np.uint64) == om).all()
    assert (depth.cpu().numpy() == od).all()
    assert od.max() <= L
