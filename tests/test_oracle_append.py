"""Oracle pins for the tree K/V append ("EAGLE code principles", KV缓存优化:
KVCache.cat puts the new tokens' rows after the prefix; the tree's node i sits
at logical position P + i, and its rotary position is P + depth(i)).

Pinned against: the block-table slot mapping written out by hand, a plain copy
when the rotation is off, the identity at position 0, the closed form of a
single rotating pair (head size 2, numpy's cos/sin), pair norms, the
relative-position property of rotary embeddings, equal rotations of siblings,
and the all-or-nothing error rule."""
import numpy as np
import pytest

import oracle
import workloads as W


def setup(rng, B=3, N=7, Hkv=2, d=8, bs=4, f32=True):
    P = rng.integers(0, 9, size=B).astype(np.int32)
    nb = [(int(p) + N + bs - 1) // bs for p in P]
    maxb = max(nb)
    perm = rng.permutation(sum(nb) + 3)                 # three spare blocks
    table = np.full((B, maxb), -1, np.int32)
    k = 0
    for b in range(B):
        table[b, :nb[b]] = perm[k:k + nb[b]]
        k += nb[b]
    num_blocks = sum(nb) + 3
    mk = (lambda a: a.astype(np.float32)) if f32 else (lambda a: W.f32_to_bf16_bits(a.astype(np.float32)))
    kc = mk(rng.standard_normal((num_blocks, Hkv, bs, d)))
    vc = mk(rng.standard_normal((num_blocks, Hkv, bs, d)))
    kn = mk(rng.standard_normal((B, N, Hkv, d)))
    vn = mk(rng.standard_normal((B, N, Hkv, d)))
    return P, table, kc, vc, kn, vn


def slot(table, b, t, bs):
    return table[b, t // bs], t % bs


@pytest.mark.parametrize("f32", [True, False])
def test_plain_copy_lands_on_the_mapped_slots_only(f32):
    rng = np.random.default_rng(1)
    P, table, kc, vc, kn, vn = setup(rng, f32=f32)
    k0, v0 = kc.copy(), vc.copy()
    st = oracle.tree_kv_append(kn, vn, None, kc, vc, table, P, rope_theta=0.0)
    assert (st == 0).all()
    B, N, Hkv, d = kn.shape
    bs = kc.shape[2]
    touched = np.zeros(kc.shape[:3], bool)
    for b in range(B):
        for i in range(N):
            blk, row = slot(table, b, int(P[b]) + i, bs)
            touched[blk, :, row] = True
            assert np.array_equal(kc[blk, :, row], kn[b, i]) and np.array_equal(vc[blk, :, row], vn[b, i])
    assert np.array_equal(kc[~touched], k0[~touched]) and np.array_equal(vc[~touched], v0[~touched])


def test_position_zero_is_the_identity():
    rng = np.random.default_rng(2)
    P, table, kc, vc, kn, vn = setup(rng, B=1)
    P[:] = 0
    depth = np.zeros((1, kn.shape[1]), np.int32)        # every node at depth 0
    st = oracle.tree_kv_append(kn, vn, depth, kc, vc, table, P, rope_theta=10000.0)
    assert (st == 0).all()
    for i in range(kn.shape[1]):
        blk, row = slot(table, 0, i, kc.shape[2])
        assert np.array_equal(kc[blk, :, row], kn[0, i])


def test_single_pair_matches_the_closed_form_rotation():
    """Head size 2: one pair (x, y) rotated by angle = position (theta^0 = 1)."""
    rng = np.random.default_rng(3)
    P, table, kc, vc, kn, vn = setup(rng, B=2, N=5, Hkv=3, d=2, bs=2)
    depth = np.tile(np.array([0, 1, 1, 2, 3], np.int32), (2, 1))
    st = oracle.tree_kv_append(kn, vn, depth, kc, vc, table, P, rope_theta=500000.0)
    assert (st == 0).all()
    for b in range(2):
        for i in range(5):
            blk, row = slot(table, b, int(P[b]) + i, 2)
            a = float(P[b] + depth[b, i])
            x, y = kn[b, i, :, 0].astype(np.float64), kn[b, i, :, 1].astype(np.float64)
            ref = np.stack([x * np.cos(a) - y * np.sin(a), y * np.cos(a) + x * np.sin(a)], -1)
            np.testing.assert_allclose(kc[blk, :, row], ref.astype(np.float32), rtol=1e-6, atol=1e-6)


def test_rotation_keeps_pair_norms_and_relative_positions():
    """|(k_j, k_{j+d/2})| is unchanged, and <rot(a, m), rot(c, n)> depends only on
    m - n (float32 caches, so only binary32 rounding separates the two sides)."""
    rng = np.random.default_rng(4)
    d, N, bs = 16, 6, 8
    P = np.array([3, 40], np.int32)                      # the same keys 37 positions apart
    table = np.full((2, 6), -1, np.int32)
    table[0, :2] = [0, 1]
    table[1, :6] = np.arange(2, 8)
    kc = np.zeros((8, 1, bs, d), np.float32)
    vc = np.zeros_like(kc)
    kn = rng.standard_normal((2, N, 1, d)).astype(np.float32)
    kn[1] = kn[0]
    vn = np.zeros_like(kn)
    depth = np.tile(np.arange(N, dtype=np.int32), (2, 1))
    st = oracle.tree_kv_append(kn, vn, depth, kc, vc, table, P, rope_theta=10000.0)
    assert (st == 0).all()
    def rows(b):
        out = []
        for i in range(N):
            blk, row = slot(table, b, int(P[b]) + i, bs)
            out.append(kc[blk, 0, row])
        return np.stack(out).astype(np.float64)
    r0, r1 = rows(0), rows(1)
    h = d // 2
    n_in = kn[0, :, 0].astype(np.float64)
    np.testing.assert_allclose(np.hypot(r0[:, :h], r0[:, h:]), np.hypot(n_in[:, :h], n_in[:, h:]), rtol=2e-6)
    g0, g1 = r0 @ r0.T, r1 @ r1.T                        # all pairs (m, n): depends on m - n only
    np.testing.assert_allclose(g0, g1, rtol=1e-4, atol=1e-4)
    assert not np.allclose(r0, r1, atol=1e-3)            # the rows themselves differ


def test_siblings_at_equal_depth_get_equal_rotations():
    rng = np.random.default_rng(5)
    P, table, kc, vc, kn, vn = setup(rng, B=1, N=4, Hkv=2, d=8)
    kn[0, 2] = kn[0, 1]
    depth = np.array([[0, 1, 1, 2]], np.int32)           # nodes 1 and 2 are siblings
    assert (oracle.tree_kv_append(kn, vn, depth, kc, vc, table, P, rope_theta=10000.0) == 0).all()
    b1, r1 = slot(table, 0, int(P[0]) + 1, kc.shape[2])
    b2, r2 = slot(table, 0, int(P[0]) + 2, kc.shape[2])
    assert np.array_equal(kc[b1, :, r1], kc[b2, :, r2])
    assert not np.array_equal(kc[b1, :, r1], kn[0, 1])  # rotated (position P + 1 > 0)


def test_bad_block_negative_prefix_or_depth_leave_the_sequence_untouched():
    rng = np.random.default_rng(6)
    P, table, kc, vc, kn, vn = setup(rng, B=3)
    table = table.copy()
    table[0, int(P[0]) // kc.shape[2]] = kc.shape[0] + 5  # block of position P_0: outside the cache
    P[1] = -1
    depth = np.zeros((3, kn.shape[1]), np.int32)
    depth[2, 3] = kn.shape[1]                            # depth outside [0, N)
    k0, v0 = kc.copy(), vc.copy()
    st = oracle.tree_kv_append(kn, vn, depth, kc, vc, table, P, rope_theta=10000.0)
    assert list(st) == [oracle.OUT_OF_RANGE] * 3
    assert np.array_equal(kc, k0) and np.array_equal(vc, v0)
