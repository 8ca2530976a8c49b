"""One verification step through the four entry points, with its buffers.

A convenience for callers that hold torch tensors: it owns the outputs and
the attention workspace and issues, in stream order,
tree_mask_build -> tree_verify_attention -> tree_accept -> kv_compact,
eagerly (``run``) or as a captured CUDA graph (``capture``, then replay).
Marshalling only; the arithmetic is in the CUDA library.
"""
from __future__ import annotations

import torch

from . import (GREEDY, STOCHASTIC, kv_compact, tree_accept, tree_accept_workspace,
               tree_mask_build, tree_verify_attention, tree_verify_attention_workspace)


class VerifyStep:
    def __init__(self, *, B, N, Hq, Hkv, d, max_blocks, bs, dtype, max_path, V=1,
                 mode=GREEDY, device="cuda"):
        self.B, self.N, self.Hq, self.Hkv, self.d = B, N, Hq, Hkv, d
        self.max_path = max_path
        dev = torch.device(device)
        i32 = dict(dtype=torch.int32, device=dev)
        self.mask = torch.zeros((B, N), dtype=torch.int64, device=dev)
        self.depth = torch.zeros((B, N), **i32)
        self.st_mask = torch.zeros(B, **i32)
        self.out = torch.zeros((B, N, Hq, d), dtype=dtype, device=dev)
        self.st_attn = torch.zeros(B, **i32)
        self.accept_len = torch.zeros(B, **i32)
        self.path = torch.zeros((B, max_path), **i32)
        self.out_tokens = torch.zeros((B, max_path), **i32)
        self.st_accept = torch.zeros(B, **i32)
        self.new_lens = torch.zeros(B, **i32)
        self.src_slots = torch.zeros((B, max_path), dtype=torch.int64, device=dev)
        self.dst_slots = torch.zeros((B, max_path), dtype=torch.int64, device=dev)
        self.st_compact = torch.zeros(B, **i32)
        ws = tree_verify_attention_workspace(B, N, Hq, Hkv, d, max_blocks, bs, dtype)
        self.workspace = torch.zeros(max(ws, 256), dtype=torch.uint8, device=dev)
        aws = tree_accept_workspace(mode, B, N, V)
        self.accept_workspace = torch.zeros(max(aws, 256), dtype=torch.uint8, device=dev)

    def mask_build(self, parents, stream=None, node_counts=None):
        tree_mask_build(parents, self.mask, self.depth, self.st_mask, stream=stream,
                        node_counts=node_counts)

    def attention(self, q, k_cache, v_cache, block_table, prefix_lens, stream=None,
                  node_counts=None):
        tree_verify_attention(q, k_cache, v_cache, block_table, prefix_lens, self.mask, self.out,
                              self.st_attn, self.workspace, stream=stream,
                              node_counts=node_counts)

    def accept(self, mode, parents, draft_tokens, target, draft_probs=None, seed=0, offset=0,
               stream=None, node_counts=None):
        tree_accept(mode, parents, draft_tokens, target, draft_probs, self.accept_len, self.path,
                    self.out_tokens, self.st_accept, seed=seed, offset=offset,
                    workspace=self.accept_workspace, stream=stream, node_counts=node_counts)

    def compact(self, k_cache, v_cache, block_table, prefix_lens, stream=None):
        kv_compact(k_cache, v_cache, block_table, prefix_lens, self.path, self.accept_len,
                   self.new_lens, self.st_compact, src_slots=self.src_slots,
                   dst_slots=self.dst_slots, stream=stream)

    def run(self, *, parents, q, k_cache, v_cache, block_table, prefix_lens, draft_tokens, target,
            draft_probs=None, mode=GREEDY, seed=0, offset=0, stream=None, node_counts=None):
        """node_counts (int32 [B] on the device, or None): each sequence's tree is its
        first node_counts[b] node slots; read on the device, so a captured step serves
        any count vector written into the same tensor."""
        self.mask_build(parents, stream, node_counts)
        self.attention(q, k_cache, v_cache, block_table, prefix_lens, stream, node_counts)
        self.accept(mode, parents, draft_tokens, target, draft_probs, seed, offset, stream,
                    node_counts)
        self.compact(k_cache, v_cache, block_table, prefix_lens, stream)

    def capture(self, **step_args) -> "torch.cuda.CUDAGraph":
        """Records one step (the four launches of ``run`` with these tensors) into
        a CUDA graph; ``graph.replay()`` then re-issues it with one launch.  The
        graph keeps the tensors' addresses and the host-side choices of this call
        (schedule, tensor descriptors): refill the same input tensors in place
        between replays and keep the shapes.  One eager step first takes the
        library's one-time host set-up (function attributes, occupancy queries),
        so none of it is recorded; the caches are mutated by that step like by
        any other (compaction)."""
        stream = torch.cuda.Stream()
        stream.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(stream):
            self.run(**step_args, stream=stream)
        torch.cuda.current_stream().wait_stream(stream)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            self.run(**step_args, stream=torch.cuda.current_stream())
        return graph


__all__ = ["VerifyStep", "GREEDY", "STOCHASTIC"]
