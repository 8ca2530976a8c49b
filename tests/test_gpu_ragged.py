"""Trees with fewer nodes than the batch's N (per-sequence node counts) on the
GPU, against the oracle ("P-EAGLE in vLLM", practice 5: shapes stay fixed so
that a captured CUDA graph serves every step).

Each sequence's tree is its first counts[b] node slots.  The K/V rows of the
absent slots are NaN and the blocks past each sequence's last present key
are removed from its table, so a kernel that read an absent key or checked an
absent block would change an output or a status.  Absent output rows are
filled with a marker first and must keep it.  Mask, depth, acceptance,
compaction and append are bit-exact; attention is within the bf16 / fp32
tolerances used everywhere else.
"""
import numpy as np
import pytest
import torch

import workloads as W
from gpu_util import dev, host_f32

pytestmark = pytest.mark.gpu

BF16_MAX, BF16_MEAN, F32_MAX = 2e-2, 2e-3, 1e-5
MARK_BF16 = 0x7F7F  # a finite bf16 pattern no attention output here takes


@pytest.fixture(scope="module")
def tv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import eagle_speculative_decoding_parent_gb300 as m
    return m


def counts_for(B, N, seed):
    rng = np.random.default_rng(seed)
    c = rng.integers(1, N + 1, size=B).astype(np.int32)
    c[0] = N                      # a full tree
    if B > 1:
        c[1] = 1                  # the root alone
    return c


def raggedise(w, counts):
    """Absent K/V rows -> NaN, blocks past the last present key -> -1."""
    spec = w["spec"]
    B, N = w["parents"].shape
    nan = np.uint16(0x7FC0) if spec.bf16 else np.float32(np.nan)
    bt = w["block_table"].copy()
    for b in range(B):
        P = int(w["prefix_lens"][b])
        for t in range(P + counts[b], P + N):
            blk = bt[b, t // spec.bs]
            w["k_cache"][blk, :, t % spec.bs] = nan
            w["v_cache"][blk, :, t % spec.bs] = nan
        last = (P + counts[b] + spec.bs - 1) // spec.bs
        bt[b, last:] = -1
    w["block_table"] = bt


CASES = [
    # name, overrides: every attention kernel family and both acceptance modes
    ("tiny_fp32", dict(B=3, N=7)),                                     # fp32 kernel, greedy
    ("llama3_8b_tree60", dict(B=3, P_lo=300, P_hi=900, V=4096)),       # tcgen05, two row tiles
    ("llama3_8b_b32_tree26", dict(B=10, P_hi=1500, V=128256)),        # tcgen05, walk acceptance
    ("llama3_8b_b128_chain5", dict(B=8, P_hi=1500, V=4096)),          # chain, stochastic
    ("qwen2_7b_32k_tree63", dict(B=4, P_lo=700, P_hi=1200, V=4096)),  # four row tiles
    ("llama3_8b_b32_tree26", dict(B=5, d=64, Hq=16, Hkv=4, P_hi=700, V=4096)),  # warp-MMA, d = 64
    ("llama3_8b_b32_tree26", dict(B=4, P_hi=900, V=2048, mode="stochastic",
                                  temperature=0.8)),                  # stochastic, branching trees
]


@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("split", [None, "1"])
def test_ragged_step_matches_oracle(tv, orc, case, split, monkeypatch):
    name, over = CASES[case]
    if split is not None:
        if over.get("d", 128) != 128 or name == "tiny_fp32":
            pytest.skip("the balanced split is a tensor-core schedule")
        monkeypatch.setenv("TV_SPLIT", split)
    w = W.make(name, **over)
    spec = w["spec"]
    B, N = w["parents"].shape
    counts = counts_for(B, N, 17 + case)
    raggedise(w, counts)
    mp = W.max_path_len(w["parents"])
    d = {k: dev(w[k]) for k in ("parents", "prefix_lens", "block_table", "draft_tokens")}
    for k in ("q", "k_cache", "v_cache"):
        d[k] = dev(w[k], spec.bf16)
    greedy = spec.mode == "greedy"
    target = dev(w["logits"] if greedy else w["p"])
    draft = None if greedy else dev(w["q_probs"])
    cnt = dev(counts)
    mode = tv.GREEDY if greedy else tv.STOCHASTIC
    i32 = dict(dtype=torch.int32, device="cuda")

    mask = torch.zeros((B, N), dtype=torch.int64, device="cuda")
    depth = torch.zeros((B, N), **i32)
    st = torch.full((B,), -9, **i32)
    tv.tree_mask_build(d["parents"], mask, depth, st, node_counts=cnt)
    rm, rd, rs = orc.tree_mask(w["parents"], counts)
    torch.cuda.synchronize()
    assert np.array_equal(mask.cpu().numpy().view(np.uint64), rm)
    assert np.array_equal(depth.cpu().numpy(), rd) and np.array_equal(st.cpu().numpy(), rs)

    out = torch.empty_like(d["q"])
    if spec.bf16:
        out.view(torch.int16).fill_(MARK_BF16)
    else:
        out.fill_(12345.0)
    ws = torch.zeros(max(256, tv.tree_verify_attention_workspace(
        B, N, spec.Hq, spec.Hkv, spec.d, w["block_table"].shape[1], spec.bs, d["q"].dtype)),
        dtype=torch.uint8, device="cuda")
    sta = torch.full((B,), -9, **i32)
    tv.tree_verify_attention(d["q"], d["k_cache"], d["v_cache"], d["block_table"],
                             d["prefix_lens"], mask, out, sta, ws, node_counts=cnt)
    torch.cuda.synchronize()
    assert (sta.cpu().numpy() == 0).all()
    ref, rst = orc.attention(w["q"], w["k_cache"], w["v_cache"], w["block_table"],
                             w["prefix_lens"], rm, bf16=spec.bf16, nthreads=8, counts=counts)
    assert (rst == 0).all()
    got = host_f32(out).reshape(B, N, spec.Hq, spec.d)
    ref = ref.reshape(B, N, spec.Hq, spec.d)
    present = np.arange(N)[None, :] < counts[:, None]
    err = np.abs(got[present].astype(np.float64) - ref[present])
    if spec.bf16:
        assert err.max() <= BF16_MAX and err.mean() <= BF16_MEAN, (err.max(), err.mean())
        raw = out.view(torch.int16).cpu().numpy().view(np.uint16).reshape(B, N, -1)
        assert (raw[~present] == MARK_BF16).all()          # absent rows not written
    else:
        assert err.max() <= F32_MAX
        assert (got[~present] == 12345.0).all()

    acc = torch.full((B,), -9, **i32)
    path = torch.full((B, mp), -9, **i32)
    toks = torch.full((B, mp), -9, **i32)
    stc = torch.full((B,), -9, **i32)
    aws = torch.zeros(max(256, tv.tree_accept_workspace(mode, B, N, spec.V)), dtype=torch.uint8,
                      device="cuda")
    tv.tree_accept(mode, d["parents"], d["draft_tokens"], target, draft, acc, path, toks, stc,
                   seed=w.get("seed", 0), workspace=aws, node_counts=cnt)
    torch.cuda.synchronize()
    if greedy:
        ra = orc.accept_greedy(w["parents"], w["draft_tokens"], w["logits"], mp, counts=counts)
    else:
        ra = orc.accept_stochastic(w["parents"], w["draft_tokens"], w["p"], w["q_probs"],
                                   w["seed"], 0, mp, counts=counts)
    for g, r in zip((acc, path, toks, stc), ra):
        assert np.array_equal(g.cpu().numpy(), r)
    assert (ra[0] < counts).all()                          # no absent node accepted


def test_ragged_append_and_bad_counts(tv, orc):
    """tree_kv_append writes only present nodes; a count outside [1, N] gives
    the sequence OUT_OF_RANGE in every step that takes counts."""
    rng = np.random.default_rng(3)
    B, N, Hkv, d, bs = 5, 9, 2, 128, 16
    counts = np.array([9, 1, 4, 0, 10], np.int32)        # 0 and 10: outside [1, N]
    P = rng.integers(0, 50, size=B).astype(np.int32)
    nb = [(int(x) + N + bs - 1) // bs for x in P]
    bt = np.full((B, max(nb)), -1, np.int32)
    perm = rng.permutation(sum(nb))
    o = 0
    for b in range(B):
        bt[b, :nb[b]] = perm[o:o + nb[b]]
        o += nb[b]
    par = np.array([[-1] + [int(rng.integers(0, i)) for i in range(1, N)] for _ in range(B)], np.int32)
    kn = W.f32_to_bf16_bits(rng.standard_normal((B, N, Hkv, d)).astype(np.float32))
    vn = W.f32_to_bf16_bits(rng.standard_normal((B, N, Hkv, d)).astype(np.float32))
    kc = W.f32_to_bf16_bits(rng.standard_normal((sum(nb), Hkv, bs, d)).astype(np.float32))
    vc = W.f32_to_bf16_bits(rng.standard_normal((sum(nb), Hkv, bs, d)).astype(np.float32))
    _, depth, ms = orc.tree_mask(par, counts)
    assert list(ms) == [0, 0, 0, orc.OUT_OF_RANGE, orc.OUT_OF_RANGE]
    kd, vd = dev(kc, True), dev(vc, True)
    st = torch.full((B,), -9, dtype=torch.int32, device="cuda")
    tv.tree_kv_append(dev(kn, True), dev(vn, True), dev(depth), kd, vd, dev(bt), dev(P), st,
                      rope_theta=10000.0, node_counts=dev(counts))
    torch.cuda.synchronize()
    kr, vr = kc.copy(), vc.copy()
    rs = orc.tree_kv_append(kn, vn, depth, kr, vr, bt, P, rope_theta=10000.0, counts=counts)
    assert np.array_equal(st.cpu().numpy(), rs) and list(rs[3:]) == [orc.OUT_OF_RANGE] * 2
    gk = kd.view(torch.int16).cpu().numpy().view(np.uint16)
    gv = vd.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(gv, vr)
    # rotated keys: within one unit in the last place of bf16 (host and device sin/cos)
    diff = np.abs(gk.astype(np.int32) - kr.astype(np.int32))
    assert diff.max() <= 1
    mask = torch.zeros((B, N), dtype=torch.int64, device="cuda")
    sm = torch.full((B,), -9, dtype=torch.int32, device="cuda")
    tv.tree_mask_build(dev(par), mask, None, sm, node_counts=dev(counts))
    torch.cuda.synchronize()
    assert np.array_equal(sm.cpu().numpy(), ms)


def test_graph_replay_across_count_vectors(tv, orc):
    """One captured verification step (mask, attention, acceptance,
    compaction) replayed with two different count vectors written into the
    same tensor: each replay equals the oracle for its counts, and replaying
    the first vector again is bit-identical to its first replay."""
    from eagle_speculative_decoding_parent_gb300.pipeline import VerifyStep
    w = W.make("llama3_8b_b32_tree26", B=6, P_hi=1500, V=4096)
    spec = w["spec"]
    B, N = w["parents"].shape
    ca = counts_for(B, N, 5)
    cb = counts_for(B, N, 6)
    cb[0], cb[1] = 1, N
    raggedise(w, np.maximum(ca, cb))          # rows absent under both vectors
    mp = W.max_path_len(w["parents"])
    d = {k: dev(w[k]) for k in ("parents", "prefix_lens", "block_table", "draft_tokens", "logits")}
    for k in ("q", "k_cache", "v_cache"):
        d[k] = dev(w[k], True)
    k0, v0 = d["k_cache"].clone(), d["v_cache"].clone()
    cnt = dev(ca)
    step = VerifyStep(B=B, N=N, Hq=spec.Hq, Hkv=spec.Hkv, d=spec.d,
                      max_blocks=w["block_table"].shape[1], bs=spec.bs, dtype=torch.bfloat16,
                      max_path=mp, V=spec.V, mode=tv.GREEDY)
    args = dict(parents=d["parents"], q=d["q"], k_cache=d["k_cache"], v_cache=d["v_cache"],
                block_table=d["block_table"], prefix_lens=d["prefix_lens"],
                draft_tokens=d["draft_tokens"], target=d["logits"], mode=tv.GREEDY,
                node_counts=cnt)
    graph = step.capture(**args)

    def replay(counts):
        cnt.copy_(torch.from_numpy(counts))
        d["k_cache"].copy_(k0)
        d["v_cache"].copy_(v0)
        step.out.view(torch.int16).fill_(MARK_BF16)
        graph.replay()
        torch.cuda.synchronize()
        return {k: getattr(step, k).clone() for k in ("mask", "out", "accept_len", "path",
                                                       "out_tokens", "new_lens")}

    def check(res, counts):
        rm, _, _ = orc.tree_mask(w["parents"], counts)
        assert np.array_equal(res["mask"].cpu().numpy().view(np.uint64), rm)
        ref, _ = orc.attention(w["q"], w["k_cache"], w["v_cache"], w["block_table"],
                               w["prefix_lens"], rm, bf16=True, nthreads=8, counts=counts)
        got = host_f32(res["out"]).reshape(B, N, spec.Hq, spec.d)
        ref = ref.reshape(B, N, spec.Hq, spec.d)
        present = np.arange(N)[None, :] < counts[:, None]
        err = np.abs(got[present].astype(np.float64) - ref[present])
        assert err.max() <= BF16_MAX and err.mean() <= BF16_MEAN
        raw = res["out"].view(torch.int16).cpu().numpy().view(np.uint16).reshape(B, N, -1)
        assert (raw[~present] == MARK_BF16).all()
        ra = orc.accept_greedy(w["parents"], w["draft_tokens"], w["logits"], mp, counts=counts)
        for k, r in zip(("accept_len", "path", "out_tokens"), ra[:3]):
            assert np.array_equal(res[k].cpu().numpy(), r)
        assert np.array_equal(res["new_lens"].cpu().numpy(), w["prefix_lens"] + ra[0] + 1)

    ra1 = replay(ca)
    check(ra1, ca)
    rb = replay(cb)
    check(rb, cb)
    ra2 = replay(ca)
    for k in ra1:
        assert torch.equal(ra1[k], ra2[k]), k
