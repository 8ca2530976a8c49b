"""tree_verify_attention_noalloc against tree_verify_attention (GPU).

The no-allocation entry point serves callers that cannot give the library a
scratch buffer (an engine that owns all device memory and does not allocate
while decoding, or a plugin host without an allocator): it takes its scratch
from a fixed array inside the library instead.  Its results must match the
workspace-taking entry point within the attention tolerance used everywhere
else (bf16: max-abs 2e-2, mean-abs 2e-3), on two calls in a row, since every
call reuses the same array and must clear what has to start at zero.

This file is collected after the parity tests so that a run stopping at its
first failure has already run them; it also passes on its own in a fresh
process.
"""
import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


def _dev(a, bf16=False):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if bf16:
        t = t.view(torch.int16).view(torch.bfloat16)
    return t.cuda()


@pytest.mark.parametrize("name,overrides", [
    ("llama3_8b_tree60", {}),                              # split-KV merge path
    ("llama3_8b_b32_tree26", {"B": 2, "P_hi": 3000}),      # ragged prefixes
])
def test_noalloc_matches_workspace_entry_point(name, overrides):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import oracle
    import eagle_speculative_decoding_parent_gb300 as tv

    w = W.make(name, parts=("attn",), **overrides)
    spec = w["spec"]
    B, N = w["parents"].shape
    mask_np, _, _ = oracle.tree_mask(w["parents"])
    q = _dev(w["q"], spec.bf16)
    k = _dev(w["k_cache"], spec.bf16)
    v = _dev(w["v_cache"], spec.bf16)
    bt = _dev(w["block_table"])
    P = _dev(w["prefix_lens"])
    mask = torch.from_numpy(mask_np.view(np.int64)).cuda()
    need = tv.tree_verify_attention_workspace(B, N, spec.Hq, spec.Hkv, spec.d, bt.shape[1],
                                              spec.bs, q.dtype)
    assert need <= tv.tree_verify_attention_noalloc_capacity()

    ws = torch.zeros(max(need, 256), dtype=torch.uint8, device="cuda")
    ref = torch.empty_like(q)
    st_ref = torch.full((B,), -9, dtype=torch.int32, device="cuda")
    tv.tree_verify_attention(q, k, v, bt, P, mask, ref, st_ref, ws)

    for call in range(2):
        out = torch.full_like(q, float("nan"))
        st = torch.full((B,), -9, dtype=torch.int32, device="cuda")
        tv.tree_verify_attention_noalloc(q, k, v, bt, P, mask, out, st)
        torch.cuda.synchronize()
        assert (st == 0).all() and (st_ref == 0).all()
        err = (out.float() - ref.float()).abs()
        assert torch.isfinite(out.float()).all(), f"call {call}"
        assert err.max().item() <= 2e-2 and err.mean().item() <= 2e-3, f"call {call}"


def test_noalloc_scratch_covers_extreme_shapes():
    """Every shape the attention step supports fits the fixed scratch, so the
    entry point's size check (TV_ERR_WORKSPACE) never turns a valid call away."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import eagle_speculative_decoding_parent_gb300 as tv
    cap = tv.tree_verify_attention_noalloc_capacity()
    for B, N, Hq, Hkv, d, max_blocks in [(1, 64, 64, 1, 128, 1 << 16), (4096, 64, 128, 8, 128, 4096),
                                          (4096, 1, 8, 8, 64, 1), (1, 1, 1, 1, 64, 1)]:
        need = tv.tree_verify_attention_workspace(B, N, Hq, Hkv, d, max_blocks, 16, torch.bfloat16)
        assert 0 < need <= cap, (B, N, Hq, Hkv, d, max_blocks, need, cap)
