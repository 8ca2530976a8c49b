"""Pins for the oracle's KV compaction (CPU only).

"EAGLE code principles" (KV缓存优化): KVCache.copy(indices, prev_length)
selects the kept entries with index_select, locates the destination with
narrow(dim, prev_length, n) and copies them there.  With one contiguous block
per sequence the paged layout reduces to exactly that view, so torch's own
index_select / narrow / copy_ is the reference.  For paged caches the rows are
tagged with their original logical position and the result is decoded.
"""
import numpy as np
import pytest
import torch


def test_contiguous_cache_equals_index_select_narrow_copy(orc):
    rng = np.random.default_rng(0)
    Hkv, d, bs = 3, 8, 64
    P, N = 20, 12
    k = rng.standard_normal((1, Hkv, bs, d)).astype(np.float32)
    v = rng.standard_normal((1, Hkv, bs, d)).astype(np.float32)
    path = np.array([[0, 2, 3, 7, 11, -1, -1]], np.int32)   # increasing, path[j] >= j
    A = 4
    table = np.array([[0]], np.int32)
    kt, vt = torch.from_numpy(k.copy()), torch.from_numpy(v.copy())
    new_lens, src, dst, st = orc.kv_compact(k, v, table, np.array([P], np.int32), path,
                                            np.array([A], np.int32))
    idx = torch.from_numpy((P + path[0, :A + 1]).astype(np.int64))
    for t in (kt, vt):
        data = t[0]                                   # [Hkv, bs, d], token dim = 1
        tgt = data.index_select(1, idx)
        data.narrow(1, P, A + 1).copy_(tgt)
    assert st[0] == 0 and new_lens[0] == P + A + 1
    assert np.array_equal(k, kt.numpy()) and np.array_equal(v, vt.numpy())
    assert list(src[0, :A + 1]) == list(P + path[0, :A + 1]) and (src[0, A + 1:] == -1).all()
    assert list(dst[0, :A + 1]) == list(range(P, P + A + 1))


def tagged_cache(num_blocks, Hkv, bs, d, table, salt):
    """Row (block, g, r) of a cache whose logical owner is (b, t) holds the tag
    [b, t, g, salt, ...]; unowned rows hold -1."""
    c = np.full((num_blocks, Hkv, bs, d), -1, np.int32)
    for b in range(table.shape[0]):
        for j, blk in enumerate(table[b]):
            if blk < 0:
                continue
            for r in range(bs):
                for g in range(Hkv):
                    c[blk, g, r, :4] = [b, j * bs + r, g, salt]
    return c


@pytest.mark.parametrize("num_layers", [1, 2])
def test_paged_compaction_moves_tagged_rows(orc, num_layers):
    rng = np.random.default_rng(1)
    B, Hkv, d, bs, N = 4, 2, 8, 16, 20
    P = np.array([5, 16, 31, 0], np.int32)
    nb = [(p + N + bs - 1) // bs for p in P]
    perm = rng.permutation(sum(nb))
    table = np.full((B, max(nb)), -1, np.int32)
    o = 0
    for b in range(B):
        table[b, :nb[b]] = perm[o:o + nb[b]]
        o += nb[b]
    layers_k = [tagged_cache(sum(nb), Hkv, bs, d, table, 10 + l) for l in range(num_layers)]
    layers_v = [tagged_cache(sum(nb), Hkv, bs, d, table, 20 + l) for l in range(num_layers)]
    k = np.stack(layers_k)
    v = np.stack(layers_v)
    before_k, before_v = k.copy(), v.copy()
    max_path = 8
    path = np.full((B, max_path), -1, np.int32)
    acc = np.array([3, 0, 7, 5], np.int32)
    path[0, :4] = [0, 4, 9, 19]
    path[1, :1] = [0]
    path[2, :8] = [0, 1, 2, 3, 4, 5, 6, 7]              # identity: nothing moves
    path[3, :6] = [0, 2, 3, 5, 6, 8]                    # dst j can be the src of an earlier row
    stride = k[0].size
    new_lens, src, dst, st = orc.kv_compact(k, v, table, P, path, acc, num_layers=num_layers,
                                            layer_stride=stride)
    assert (st == 0).all()
    assert list(new_lens) == list(P + acc + 1)
    for l in range(num_layers):
        for cache, before, salt in ((k[l], before_k[l], 10 + l), (v[l], before_v[l], 20 + l)):
            expect = before.copy()
            for b in range(B):
                for j in range(acc[b] + 1):
                    t_dst = P[b] + j
                    blk, r = table[b, t_dst // bs], t_dst % bs
                    for g in range(Hkv):
                        expect[blk, g, r, :4] = [b, P[b] + path[b, j], g, salt]
            assert np.array_equal(cache, expect)


def test_compaction_errors_leave_cache_untouched(orc):
    Hkv, d, bs = 1, 4, 16
    table = np.array([[0, 1], [2, -1], [3, 4]], np.int32)
    k = np.arange(5 * Hkv * bs * d, dtype=np.float32).reshape(5, Hkv, bs, d)
    v = -k
    k0, v0 = k.copy(), v.copy()
    P = np.array([10, 15, -1], np.int32)
    path = np.array([[0, 30, -1], [0, 1, 2], [0, 1, -1]], np.int32)
    acc = np.array([1, 2, 1], np.int32)
    new_lens, src, dst, st = orc.kv_compact(k, v, table, P, path, acc)
    # seq 0: source position 40 beyond its two blocks; seq 1: block -1 reached;
    # seq 2: negative prefix
    assert list(st) == [orc.OUT_OF_RANGE] * 3
    assert list(new_lens) == [10, 15, -1]
    assert (src == -1).all() and (dst == -1).all()
    assert np.array_equal(k, k0) and np.array_equal(v, v0)
    # accept_len beyond max_path
    new_lens, src, dst, st = orc.kv_compact(k, v, table[:1], P[:1], path[:1],
                                            np.array([3], np.int32))
    assert st[0] == orc.OUT_OF_RANGE
