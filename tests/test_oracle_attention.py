"""Pins for the oracle's tree-masked paged GQA attention (CPU only).

What the pages fix ("vLLM-TreeEagle", 核心组件 / TreeAttentionLayer;
"P-EAGLE in vLLM", 技术原理和实现方式 step 3): every draft node is scored in
one target pass, attending to the sequence's cached prefix and, through the
tree mask, to its own root path.  The pins below do not reuse the oracle's
arithmetic:

* torch's scaled_dot_product_attention in float64 on a dense layout with an
  explicit boolean mask (ancestor relation from a transitive closure);
* a chain tree equals N sequential causal decode steps (one-node trees);
* closed forms: uniform weights, constant values, GQA head grouping, a lone
  root with an empty prefix, the two-key logistic form that fixes the scale;
* relocating physical blocks (a new block table) changes nothing.
The dense -> paged layout is produced here with reshapes and fancy indexing,
not with the oracle's slot arithmetic.
"""
import numpy as np
import pytest
import torch

from workloads import f32_to_bf16_bits, bf16_bits_to_f32


def closure(par):
    N = len(par)
    R = np.eye(N, dtype=bool)
    for i in range(1, N):
        R[i, par[i]] = True
    for k in range(N):
        R = R | (R[:, [k]] & R[[k], :])
    return R  # R[i, j]: j is i or an ancestor of i


def random_tree(rng, N):
    return [-1] + [int(rng.integers(i)) for i in range(1, N)]


def paged_from_dense(dense_list, Hkv, d, bs, rng, dtype):
    """dense_list[b]: [L_b, Hkv, d] -> (cache [nb, Hkv, bs, d], block_table)."""
    pages, owners = [], []
    for b, x in enumerate(dense_list):
        L = x.shape[0]
        nb = -(-L // bs)
        pad = np.zeros((nb * bs - L, Hkv, d), dtype)
        x = np.concatenate([x, pad]).reshape(nb, bs, Hkv, d).transpose(0, 2, 1, 3)
        pages.extend(list(x))
        owners.append(nb)
    perm = rng.permutation(len(pages))            # logical page k lives in block perm[k]
    cache = np.zeros((len(pages), Hkv, bs, d), dtype)
    cache[perm] = np.stack(pages)
    table = np.full((len(dense_list), max(owners)), -1, np.int32)
    k = 0
    for b, nb in enumerate(owners):
        table[b, :nb] = perm[k:k + nb]
        k += nb
    return cache, table


def make_case(rng, B, N, Hq, Hkv, d, bs, Ps, trees=None):
    q = rng.standard_normal((B, N, Hq, d)).astype(np.float32)
    kd = [rng.standard_normal((P + N, Hkv, d)).astype(np.float32) for P in Ps]
    vd = [rng.standard_normal((P + N, Hkv, d)).astype(np.float32) for P in Ps]
    trees = trees or [random_tree(rng, N) for _ in range(B)]
    return q, kd, vd, trees


def run_oracle(orc, q, kd, vd, trees, Ps, Hkv, d, bs, rng, **kw):
    B, N = q.shape[:2]
    kc, table = paged_from_dense(kd, Hkv, d, bs, np.random.default_rng(1), np.float32)
    vc, table2 = paged_from_dense(vd, Hkv, d, bs, np.random.default_rng(1), np.float32)
    assert (table == table2).all()
    mask, _, st = orc.tree_mask(np.array(trees, np.int32))
    assert (st == 0).all()
    out, status = orc.attention(q, kc, vc, table, np.array(Ps, np.int32), mask, bf16=False, **kw)
    assert (status == 0).all()
    return out.reshape(B, N, q.shape[2], d)


def sdpa_reference(q, kd, vd, trees, Ps, Hq, Hkv):
    outs = []
    G = Hq // Hkv
    for b, P in enumerate(Ps):
        N = q.shape[1]
        R = closure(trees[b])
        L = P + N
        vis = np.zeros((N, L), bool)
        vis[:, :P] = True
        vis[:, P:] = R
        qq = torch.from_numpy(q[b].astype(np.float64)).permute(1, 0, 2)[None]          # [1,Hq,N,d]
        kk = torch.from_numpy(kd[b].astype(np.float64)).permute(1, 0, 2)
        vv = torch.from_numpy(vd[b].astype(np.float64)).permute(1, 0, 2)
        kk = kk.repeat_interleave(G, dim=0)[None]
        vv = vv.repeat_interleave(G, dim=0)[None]
        o = torch.nn.functional.scaled_dot_product_attention(
            qq, kk, vv, attn_mask=torch.from_numpy(vis)[None, None])
        outs.append(o[0].permute(1, 0, 2).numpy())
    return np.stack(outs)


@pytest.mark.parametrize("Hq,Hkv,bs", [(4, 2, 16), (6, 2, 8), (2, 1, 16), (8, 8, 32)])
def test_attention_matches_sdpa(orc, Hq, Hkv, bs):
    rng = np.random.default_rng(Hq * 10 + Hkv)
    B, N, d = 3, 9, 16
    Ps = [0, 37, 70]
    q, kd, vd, trees = make_case(rng, B, N, Hq, Hkv, d, bs, Ps)
    got = run_oracle(orc, q, kd, vd, trees, Ps, Hkv, d, bs, rng)
    ref = sdpa_reference(q, kd, vd, trees, Ps, Hq, Hkv)
    np.testing.assert_allclose(got, ref, rtol=1e-11, atol=1e-12)


def test_chain_equals_sequential_decode(orc):
    """A chain of N nodes verified at once == N one-token decode steps."""
    rng = np.random.default_rng(3)
    N, Hq, Hkv, d, bs, P = 8, 4, 2, 32, 16, 45
    q, kd, vd, _ = make_case(rng, 1, N, Hq, Hkv, d, bs, [P])
    chain = [list(range(-1, N - 1))]
    tree_out = run_oracle(orc, q, kd, vd, chain, [P], Hkv, d, bs, rng)
    for i in range(N):
        # step i: prefix = first P+i positions, a one-node tree holding node i
        step = run_oracle(orc, q[:, i:i + 1], [kd[0][:P + i + 1]], [vd[0][:P + i + 1]],
                          [[-1]], [P + i], Hkv, d, bs, rng)
        assert np.array_equal(step[0, 0], tree_out[0, i])


def test_uniform_scores_give_mean_of_visible_values(orc):
    rng = np.random.default_rng(4)
    N, Hq, Hkv, d, bs, P = 7, 2, 1, 8, 16, 20
    q, kd, vd, _ = make_case(rng, 1, N, Hq, Hkv, d, bs, [P])
    kd[0][:] = kd[0][0]                      # every key identical -> equal scores
    trees = [[-1, 0, 0, 1, 1, 2, 2]]
    out = run_oracle(orc, q, kd, vd, trees, [P], Hkv, d, bs, rng)
    R = closure(trees[0])
    for i in range(N):
        rows = list(range(P)) + [P + j for j in range(N) if R[i, j]]
        exp = vd[0][rows, 0].astype(np.float64).mean(axis=0)
        np.testing.assert_allclose(out[0, i, 0], exp, rtol=1e-12, atol=1e-13)


def test_constant_values_and_gqa_grouping(orc):
    rng = np.random.default_rng(5)
    N, Hq, Hkv, d, bs, P = 5, 12, 3, 8, 8, 19
    q, kd, vd, _ = make_case(rng, 2, N, Hq, Hkv, d, bs, [P, 3])
    for b in range(2):
        for g in range(Hkv):
            vd[b][:, g, :] = g + 1.0           # kv head g holds the constant g+1
    out = run_oracle(orc, q, kd, vd, [random_tree(rng, N) for _ in range(2)], [P, 3],
                     Hkv, d, bs, rng)
    for h in range(Hq):
        np.testing.assert_allclose(out[:, :, h], h // (Hq // Hkv) + 1.0, rtol=1e-13)


def test_lone_root_with_empty_prefix_returns_its_value(orc):
    rng = np.random.default_rng(6)
    N, Hq, Hkv, d, bs = 4, 2, 1, 16, 16
    q, kd, vd, _ = make_case(rng, 1, N, Hq, Hkv, d, bs, [0])
    out = run_oracle(orc, q, kd, vd, [[-1, 0, 1, 2]], [0], Hkv, d, bs, rng)
    np.testing.assert_array_equal(out[0, 0, 0], vd[0][0, 0].astype(np.float64))
    np.testing.assert_array_equal(out[0, 0, 1], vd[0][0, 0].astype(np.float64))


def test_two_keys_logistic_form_fixes_scale(orc):
    """Prefix of one key plus the root: O = v0 + (v1 - v0) * sigmoid((s1 - s0)/sqrt(d))."""
    rng = np.random.default_rng(7)
    d = 64
    q, kd, vd, _ = make_case(rng, 1, 1, 1, 1, d, 16, [1])
    out = run_oracle(orc, q, kd, vd, [[-1]], [1], 1, d, 16, rng)
    qv = q[0, 0, 0].astype(np.float64)
    k0, k1 = kd[0][0, 0].astype(np.float64), kd[0][1, 0].astype(np.float64)
    v0, v1 = vd[0][0, 0].astype(np.float64), vd[0][1, 0].astype(np.float64)
    z = (qv @ k1 - qv @ k0) / np.sqrt(d)
    exp = v0 + (v1 - v0) / (1.0 + np.exp(-z))
    np.testing.assert_allclose(out[0, 0, 0], exp, rtol=1e-12, atol=1e-14)
    # an explicit scale overrides 1/sqrt(d)
    out2 = run_oracle(orc, q, kd, vd, [[-1]], [1], 1, d, 16, rng, scale=0.5)
    exp2 = v0 + (v1 - v0) / (1.0 + np.exp(-(qv @ k1 - qv @ k0) * 0.5))
    np.testing.assert_allclose(out2[0, 0, 0], exp2, rtol=1e-12, atol=1e-14)


def test_block_relocation_invariance_and_bf16_widening(orc):
    rng = np.random.default_rng(8)
    B, N, Hq, Hkv, d, bs = 2, 6, 4, 2, 16, 16
    Ps = [33, 50]
    q, kd, vd, trees = make_case(rng, B, N, Hq, Hkv, d, bs, Ps)
    kc, table = paged_from_dense(kd, Hkv, d, bs, np.random.default_rng(10), np.float32)
    vc, _ = paged_from_dense(vd, Hkv, d, bs, np.random.default_rng(10), np.float32)
    mask, _, _ = orc.tree_mask(np.array(trees, np.int32))
    P = np.array(Ps, np.int32)
    o1, _ = orc.attention(q, kc, vc, table, P, mask, bf16=False)
    # move every block to a new physical index
    perm = np.random.default_rng(11).permutation(kc.shape[0])
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    table2 = np.where(table >= 0, perm[np.maximum(table, 0)], -1).astype(np.int32)
    o2, _ = orc.attention(q, kc2, vc2, table2, P, mask, bf16=False)
    assert np.array_equal(o1, o2)
    # bf16 inputs are widened exactly: bf16 path == f32 path on bf16-representable data
    qb, kb, vb = (f32_to_bf16_bits(x) for x in (q, kc, vc))
    o3, _ = orc.attention(qb, kb, vb, table, P, mask, bf16=True)
    o4, _ = orc.attention(bf16_bits_to_f32(qb), bf16_bits_to_f32(kb), bf16_bits_to_f32(vb),
                          table, P, mask, bf16=False)
    assert np.array_equal(o3, o4)


def test_selection_and_threads_do_not_change_values(orc):
    rng = np.random.default_rng(9)
    B, N, Hq, Hkv, d, bs = 3, 5, 4, 1, 8, 16
    Ps = [10, 0, 31]
    q, kd, vd, trees = make_case(rng, B, N, Hq, Hkv, d, bs, Ps)
    kc, table = paged_from_dense(kd, Hkv, d, bs, np.random.default_rng(2), np.float32)
    vc, _ = paged_from_dense(vd, Hkv, d, bs, np.random.default_rng(2), np.float32)
    mask, _, _ = orc.tree_mask(np.array(trees, np.int32))
    P = np.array(Ps, np.int32)
    full, _ = orc.attention(q, kc, vc, table, P, mask, bf16=False, nthreads=3)
    sel = [14, 0, 7]
    part, _ = orc.attention(q, kc, vc, table, P, mask, bf16=False, sel=sel)
    assert np.array_equal(part, full[sel])


def test_out_of_range_blocks_set_status_and_zero_output(orc):
    rng = np.random.default_rng(12)
    B, N, Hq, Hkv, d, bs = 2, 3, 2, 1, 8, 16
    Ps = [20, 20]
    q, kd, vd, trees = make_case(rng, B, N, Hq, Hkv, d, bs, Ps)
    kc, table = paged_from_dense(kd, Hkv, d, bs, np.random.default_rng(2), np.float32)
    vc, _ = paged_from_dense(vd, Hkv, d, bs, np.random.default_rng(2), np.float32)
    mask, _, _ = orc.tree_mask(np.array(trees, np.int32))
    table = table.copy()
    table[1, 1] = kc.shape[0]          # one block id beyond the cache
    out, st = orc.attention(q, kc, vc, table, np.array(Ps, np.int32), mask, bf16=False)
    assert st[0] == 0 and st[1] == orc.OUT_OF_RANGE
    assert (out[N:] == 0).all() and np.abs(out[:N]).sum() > 0
