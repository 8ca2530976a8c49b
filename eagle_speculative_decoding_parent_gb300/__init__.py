"""Python binding of libtreeverify (EAGLE draft-tree verification on GB300).

Argument marshalling only: every step runs in the library's CUDA kernels.
The functions carry the C entry points' names and take torch CUDA tensors
(PyTorch is used for device memory and streams).  Each call is asynchronous
on the current torch stream (or ``stream``) and raises ``TreeVerifyError``
when the library returns a host-side error; per-sequence data errors are
reported in the ``status`` tensors, as the C header describes.

There is no CPU fallback: importing this package fails if the compiled
library is missing (run ``__graft_entry__.build()`` or ``python -m
eagle_speculative_decoding_parent_gb300._build``).
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

__all__ = ["TV_OK", "TV_ERR_BAD_TREE", "TV_ERR_OUT_OF_RANGE", "TV_ERR_UNSUPPORTED",
           "TV_ERR_TIMEOUT", "TV_ERR_BAD_VALUES", "TV_F32", "TV_BF16", "GREEDY", "STOCHASTIC",
           "TreeVerifyError", "library_path", "status_string", "tree_mask_build",
           "tree_verify_attention_workspace", "tree_verify_attention_kernels", "tree_kv_append",
           "tree_verify_attention",
           "tree_verify_attention_noalloc", "tree_verify_attention_noalloc_capacity",
           "tree_accept_workspace",
           "tree_accept", "kv_compact", "draft_tree_workspace", "draft_tree_expand"]

(TV_OK, TV_ERR_INVALID_ARG, TV_ERR_BAD_TREE, TV_ERR_OUT_OF_RANGE, TV_ERR_UNSUPPORTED,
 TV_ERR_CUDA, TV_ERR_TIMEOUT, TV_ERR_BAD_VALUES, TV_ERR_WORKSPACE) = range(9)
TV_F32, TV_BF16 = 0, 1
GREEDY, STOCHASTIC = 0, 1


class TreeVerifyError(RuntimeError):
    pass


def library_path() -> str:
    return _build.LIB


if not os.path.exists(_build.LIB):
    raise ImportError(f"libtreeverify is not built ({_build.LIB} missing); "
                      "run python -m eagle_speculative_decoding_parent_gb300._build")

_lib = ctypes.CDLL(_build.LIB)

_i, _u64, _i64, _f, _p, _sz = (ctypes.c_int, ctypes.c_uint64, ctypes.c_int64, ctypes.c_float,
                               ctypes.c_void_p, ctypes.c_size_t)


def _sig(name, res, args):
    fn = getattr(_lib, name)
    fn.restype = res
    fn.argtypes = args
    return fn


_status_string = _sig("tv_status_string", ctypes.c_char_p, [_i])
_abi = _sig("tv_abi_version", _i, [])
_mask = _sig("tree_mask_build", _i, [_p, _i, _i, _p, _p, _p, _p, _p])
_attn_ws = _sig("tree_verify_attention_workspace", _sz, [_i, _i, _i, _i, _i, _i, _i, _i])
_attn_nk = _sig("tree_verify_attention_kernels", _i, [_i, _i, _i, _i, _i, _i, _i, _i, _sz])
_append = _sig("tree_kv_append", _i, [_p, _p, _p, _i, _i, _p, _i, _i, _f, _p, _p, _p, _i, _p, _i,
                                      _i, _i, _p, _p])
_attn = _sig("tree_verify_attention", _i,
             [_p, _p, _p, _p, _i, _p, _p, _i, _i, _p, _i, _i, _i, _i, _i, _i, _f, _p, _p, _p, _sz,
              _p])
_attn_na = _sig("tree_verify_attention_noalloc", _i,
                [_p, _p, _p, _p, _i, _p, _p, _i, _i, _p, _i, _i, _i, _i, _i, _i, _f, _p, _p, _p])
_attn_na_cap = _sig("tree_verify_attention_noalloc_capacity", _sz, [])
_acc_ws = _sig("tree_accept_workspace", _sz, [_i, _i, _i, _i])
_acc = _sig("tree_accept", _i,
            [_i, _p, _p, _p, _p, _i, _i, _p, _i, _u64, _u64, _p, _p, _p, _i, _p, _p, _sz, _p])
_compact = _sig("kv_compact", _i,
                [_p, _p, _i, _i64, _p, _i, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _p, _p, _p,
                 _p, _p])

_draft_ws = _sig("draft_tree_workspace", _sz, [_i, _i, _i])
_draft_expand = _sig("draft_tree_expand", _i, [_p, _p, _i, _i, _i, _i, _i, _i, _p, _p, _p, _p,
                                               _p, _p, _p, _sz, _p])

assert _abi() == 2, "header / library ABI mismatch"


def status_string(code: int) -> str:
    return _status_string(int(code)).decode()


def _check(rc: int, what: str) -> None:
    if rc != TV_OK:
        raise TreeVerifyError(f"{what}: {status_string(rc)} ({rc})")


def _ptr(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch tensor")
    if not t.is_cuda:
        raise ValueError("tensors passed to libtreeverify must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensors passed to libtreeverify must be contiguous")
    return t.data_ptr()


def _want(t, dtype, name, shape=None):
    """Checks a tensor's dtype (and shape) before its pointer reaches the
    library: the kernels index every buffer by the sizes passed beside it."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")


def _counts(node_counts, B):
    """Optional per-sequence node counts: int32 [B] on the device (the tree of
    sequence b is its first node_counts[b] node slots); None for full trees."""
    if node_counts is None:
        return None
    _want(node_counts, torch.int32, "node_counts", (B,))
    return _ptr(node_counts)


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _dtype_code(t):
    if t.dtype == torch.bfloat16:
        return TV_BF16
    if t.dtype == torch.float32:
        return TV_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def tree_mask_build(parents, mask, depth, status, stream=None, *, node_counts=None) -> None:
    """parents int32 [B,N] -> mask int64 (uint64 bits) [B,N], depth int32 [B,N] or None,
    status [B]; node_counts int32 [B] or None (trees of N nodes)."""
    _want(parents, torch.int32, "parents")
    if parents.dim() != 2:
        raise ValueError("parents is int32 [B, N]")
    B, N = parents.shape
    _want(mask, torch.int64, "mask", (B, N))
    if depth is not None:
        _want(depth, torch.int32, "depth", (B, N))
    _want(status, torch.int32, "status", (B,))
    _check(_mask(_ptr(parents), B, N, _counts(node_counts, B), _ptr(mask), _ptr(depth),
                 _ptr(status), _stream(stream)), "tree_mask_build")


def tree_verify_attention_workspace(B, N, Hq, Hkv, d, max_blocks_per_seq, block_size,
                                    dtype=torch.bfloat16) -> int:
    dt = TV_BF16 if dtype == torch.bfloat16 else TV_F32
    return int(_attn_ws(B, N, Hq, Hkv, d, max_blocks_per_seq, block_size, dt))


def tree_verify_attention_kernels(B, N, Hq, Hkv, d, max_blocks_per_seq, block_size,
                                  dtype=torch.bfloat16, workspace_bytes: int = 0) -> int:
    """Kernels one tree_verify_attention call launches (launch accounting)."""
    dt = TV_BF16 if dtype == torch.bfloat16 else TV_F32
    return int(_attn_nk(B, N, Hq, Hkv, d, max_blocks_per_seq, block_size, dt, workspace_bytes))


def _attention_args(q, k_cache, v_cache, block_table, prefix_lens, mask, out, status):
    """Shape and dtype checks shared by both attention entry points."""
    if q.dim() != 4 or k_cache.dim() != 4:
        raise ValueError("q is [B,N,Hq,d] and the caches [num_blocks,Hkv,block_size,d]")
    B, N, Hq, d = q.shape
    num_blocks, Hkv, bs, d2 = k_cache.shape
    if d2 != d:
        raise ValueError("q and the caches disagree on the head size")
    dt = _dtype_code(q)
    _want(k_cache, q.dtype, "k_cache")
    _want(v_cache, q.dtype, "v_cache", k_cache.shape)
    _want(out, q.dtype, "out", q.shape)
    if block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("block_table is int32 [B, max_blocks_per_seq]")
    _want(block_table, torch.int32, "block_table")
    _want(prefix_lens, torch.int32, "prefix_lens", (B,))
    _want(mask, torch.int64, "mask", (B, N))
    _want(status, torch.int32, "status", (B,))
    return B, N, Hq, Hkv, d, bs, num_blocks, dt


def tree_verify_attention(q, k_cache, v_cache, block_table, prefix_lens, mask, out, status,
                          workspace=None, *, scale: float = 0.0, stream=None,
                          node_counts=None) -> None:
    """q [B,N,Hq,d]; caches [num_blocks,Hkv,bs,d]; block_table int32 [B,max_blocks];
    prefix_lens int32 [B]; mask int64 [B,N]; out like q; status int32 [B];
    workspace uint8 tensor (zero-filled before first use); node_counts int32 [B]
    or None (rows of absent nodes are not written)."""
    B, N, Hq, Hkv, d, bs, num_blocks, dt = _attention_args(q, k_cache, v_cache, block_table,
                                                           prefix_lens, mask, out, status)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_attn(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), block_table.shape[1],
                 _ptr(prefix_lens), _ptr(mask), B, N, _counts(node_counts, B), Hq, Hkv, d, bs,
                 num_blocks, dt, scale, _ptr(out), _ptr(status), _ptr(workspace), ws_bytes,
                 _stream(stream)), "tree_verify_attention")


def tree_verify_attention_noalloc_capacity() -> int:
    return int(_attn_na_cap())


def tree_verify_attention_noalloc(q, k_cache, v_cache, block_table, prefix_lens, mask, out,
                                  status, *, scale: float = 0.0, stream=None,
                                  node_counts=None) -> None:
    """tree_verify_attention for callers that cannot hand the library a
    workspace: the scratch is a fixed array inside the library, shared by
    every call on a device (overlapping calls race on it; the C header gives
    the size limit)."""
    B, N, Hq, Hkv, d, bs, num_blocks, dt = _attention_args(q, k_cache, v_cache, block_table,
                                                           prefix_lens, mask, out, status)
    _check(_attn_na(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
                    block_table.shape[1], _ptr(prefix_lens), _ptr(mask), B, N,
                    _counts(node_counts, B), Hq, Hkv, d, bs, num_blocks, dt, scale, _ptr(out),
                    _ptr(status), _stream(stream)), "tree_verify_attention_noalloc")


def tree_accept_workspace(mode, B, N, V) -> int:
    return int(_acc_ws(mode, B, N, V))


def tree_accept(mode, parents, draft_tokens, target, draft_probs, accept_len, path, out_tokens,
                status, *, seed: int = 0, offset: int = 0, workspace=None, stream=None,
                node_counts=None) -> None:
    """Greedy (target = logits) or stochastic (target = p, draft_probs = q) acceptance;
    node_counts int32 [B] or None."""
    if target.dim() != 3:
        raise ValueError("target is float32 [B, N, V]")
    B, N, V = target.shape
    _want(target, torch.float32, "target")
    if draft_probs is not None:
        _want(draft_probs, torch.float32, "draft_probs", target.shape)
    _want(parents, torch.int32, "parents", (B, N))
    _want(draft_tokens, torch.int32, "draft_tokens", (B, N))
    if path.dim() != 2 or path.shape[0] != B:
        raise ValueError("path is int32 [B, max_path]")
    _want(path, torch.int32, "path")
    _want(out_tokens, torch.int32, "out_tokens", path.shape)
    _want(accept_len, torch.int32, "accept_len", (B,))
    _want(status, torch.int32, "status", (B,))
    if workspace is not None:
        _want(workspace, torch.uint8, "workspace")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_acc(mode, _ptr(parents), _ptr(draft_tokens), _ptr(target), _ptr(draft_probs), B, N,
                _counts(node_counts, B), V, seed, offset, _ptr(accept_len), _ptr(path),
                _ptr(out_tokens), path.shape[1], _ptr(status), _ptr(workspace), ws_bytes,
                _stream(stream)), "tree_accept")


def tree_kv_append(k_new, v_new, depth, k_cache, v_cache, block_table, prefix_lens, status, *,
                   rope_theta: float = 0.0, stream=None, node_counts=None) -> None:
    """k_new / v_new [B,N,Hkv,d]; caches [num_blocks,Hkv,bs,d]; depth int32 [B,N]
    (needed when rope_theta > 0); status int32 [B]; node_counts int32 [B] or None."""
    if k_new.dim() != 4 or k_cache.dim() != 4:
        raise ValueError("k_new is [B,N,Hkv,d] and the caches [num_blocks,Hkv,block_size,d]")
    B, N, Hkv, d = k_new.shape
    num_blocks, Hkv2, bs, d2 = k_cache.shape
    if (Hkv2, d2) != (Hkv, d):
        raise ValueError("k_new and the caches disagree on Hkv or the head size")
    _dtype_code(k_cache)
    _want(k_new, k_cache.dtype, "k_new")
    _want(v_new, k_cache.dtype, "v_new", k_new.shape)
    _want(v_cache, k_cache.dtype, "v_cache", k_cache.shape)
    if depth is not None:
        _want(depth, torch.int32, "depth", (B, N))
    if block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("block_table is int32 [B, max_blocks_per_seq]")
    _want(block_table, torch.int32, "block_table")
    _want(prefix_lens, torch.int32, "prefix_lens", (B,))
    _want(status, torch.int32, "status", (B,))
    _check(_append(_ptr(k_new), _ptr(v_new), _ptr(depth), B, N, _counts(node_counts, B), Hkv, d,
                   float(rope_theta),
                   _ptr(k_cache), _ptr(v_cache), _ptr(block_table), block_table.shape[1],
                   _ptr(prefix_lens), bs, num_blocks, _dtype_code(k_cache), _ptr(status), _stream(stream)),
           "tree_kv_append")


def kv_compact(k_cache, v_cache, block_table, prefix_lens, path, accept_len, new_lens, status,
               *, src_slots=None, dst_slots=None, num_layers: int = 1, layer_stride: int = 0,
               stream=None) -> None:
    """Caches [num_layers*][num_blocks,Hkv,bs,d] (layers back to back, ``layer_stride``
    elements apart); path int32 [B,max_path]; accept_len int32 [B]."""
    num_blocks, Hkv, bs, d = k_cache.shape[-4:]
    if path.dim() != 2:
        raise ValueError("path is int32 [B, max_path]")
    B, max_path = path.shape
    _dtype_code(k_cache)
    _want(v_cache, k_cache.dtype, "v_cache", k_cache.shape)
    _want(path, torch.int32, "path")
    if block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("block_table is int32 [B, max_blocks_per_seq]")
    _want(block_table, torch.int32, "block_table")
    for t, n in ((prefix_lens, "prefix_lens"), (accept_len, "accept_len"),
                 (new_lens, "new_lens"), (status, "status")):
        _want(t, torch.int32, n, (B,))
    for t, n in ((src_slots, "src_slots"), (dst_slots, "dst_slots")):
        if t is not None:
            _want(t, torch.int64, n, (B, max_path))
    if num_layers < 1 or (num_layers > 1 and
                          k_cache.numel() < (num_layers - 1) * layer_stride + num_blocks * Hkv * bs * d):
        raise ValueError("the caches hold fewer than num_layers layers at layer_stride")
    _check(_compact(_ptr(k_cache), _ptr(v_cache), num_layers, layer_stride, _ptr(block_table),
                    block_table.shape[1], _ptr(prefix_lens), _ptr(path), _ptr(accept_len),
                    max_path, B, Hkv, d, bs, num_blocks, _dtype_code(k_cache), _ptr(new_lens),
                    _ptr(src_slots), _ptr(dst_slots), _ptr(status), _stream(stream)),
           "kv_compact")


def draft_tree_workspace(B, topk, layers) -> int:
    return int(_draft_ws(B, topk, layers))


def draft_tree_expand(logits, layer, layers, status, workspace, *, topk, root_tokens=None,
                      N=1, front_tokens=None, front_src=None, parents=None, tokens=None,
                      scores=None, stream=None) -> None:
    """One draft-tree layer: logits float32 [B, F, V] (F = 1 at layer 0, else
    topk); root_tokens int32 [B] (layer 0); front_tokens / front_src int32
    [B, topk]; on the last layer parents / tokens int32 [B, N] and scores
    float32 [B, N]; workspace uint8 (zero-filled before the first call)."""
    _want(logits, torch.float32, "logits")
    if logits.dim() != 3:
        raise ValueError("logits is float32 [B, F, V]")
    B, F, V = logits.shape
    _want(status, torch.int32, "status", (B,))
    for t, n, shp in ((root_tokens, "root_tokens", (B,)), (front_tokens, "front_tokens", (B, topk)),
                      (front_src, "front_src", (B, topk)), (parents, "parents", (B, N)),
                      (tokens, "tokens", (B, N))):
        if t is not None:
            _want(t, torch.int32, n, shp)
    if scores is not None:
        _want(scores, torch.float32, "scores", (B, N))
    _want(workspace, torch.uint8, "workspace")
    if F != (1 if layer == 0 else topk):
        raise ValueError(f"layer {layer} takes {1 if layer == 0 else topk} rows per sequence")
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(_draft_expand(_ptr(logits), _ptr(root_tokens), B, V, topk, layer, layers, N, _ptr(front_tokens),
               _ptr(front_src), _ptr(parents), _ptr(tokens), _ptr(scores), _ptr(status),
               _ptr(workspace), ws_bytes, _stream(stream)), "draft_tree_expand")
