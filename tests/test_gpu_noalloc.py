"""tree_verify_attention_noalloc against tree_verify_attention (GPU).

The no-allocation entry point serves callers that cannot give the library a
scratch buffer (an engine that owns all device memory and does not allocate
while decoding, or a plugin host without an allocator): it takes its scratch
from a fixed array inside the library instead.  It runs the same kernels with
the same schedule as the workspace-taking entry point, so its outputs must be
bit-identical to that entry point's, on every call: each call reuses the one
array, which still holds the previous call's partial results and counters.

The shapes cover both attention schedules: one sequence and a small batch
take the cluster schedule (only the scheduler counters live in the scratch),
and a Qwen2-7B-shaped batch takes the balanced split, whose partial results
and merge kernel use the array well beyond its counters.  The calls are
interleaved so that every call after the first starts from scratch left dirty
by a call of another shape.

"""
import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

SHAPES = [
    ("llama3_8b_tree60", {}, 1),                                   # cluster schedule, B = 1
    ("llama3_8b_b32_tree26", {"B": 2, "P_hi": 3000}, 1),           # cluster, ragged prefixes
    ("qwen2_7b_32k_tree63", {"P_lo": 3000, "P_hi": 5000}, 2),      # balanced split + merge
]


def _dev(a, bf16=False):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if bf16:
        t = t.view(torch.int16).view(torch.bfloat16)
    return t.cuda()


def _inputs(name, overrides):
    import oracle
    w = W.make(name, parts=("attn",), **overrides)
    spec = w["spec"]
    mask_np, _, _ = oracle.tree_mask(w["parents"])
    d = dict(q=_dev(w["q"], spec.bf16), k=_dev(w["k_cache"], spec.bf16),
             v=_dev(w["v_cache"], spec.bf16), bt=_dev(w["block_table"]),
             P=_dev(w["prefix_lens"]), mask=torch.from_numpy(mask_np.view(np.int64)).cuda())
    return w, d


def test_noalloc_matches_workspace_entry_point():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import oracle
    import eagle_speculative_decoding_parent_gb300 as tv

    cap = tv.tree_verify_attention_noalloc_capacity()
    cases = []
    for name, overrides, kernels in SHAPES:
        w, d = _inputs(name, overrides)
        spec = w["spec"]
        B, N = w["parents"].shape
        shape = (B, N, spec.Hq, spec.Hkv, spec.d, d["bt"].shape[1], spec.bs)
        need = tv.tree_verify_attention_workspace(*shape, d["q"].dtype)
        assert need <= cap
        # the schedule this shape takes, with the caller-sized workspace and
        # with the no-allocation entry (which passes exactly `need` on)
        assert tv.tree_verify_attention_kernels(*shape, d["q"].dtype, need) == kernels, name
        ws = torch.zeros(max(need, 256), dtype=torch.uint8, device="cuda")
        ref = torch.empty_like(d["q"])
        st_ref = torch.full((B,), -9, dtype=torch.int32, device="cuda")
        tv.tree_verify_attention(d["q"], d["k"], d["v"], d["bt"], d["P"], d["mask"], ref,
                                 st_ref, ws)
        torch.cuda.synchronize()
        assert (st_ref == 0).all(), name
        cases.append((name, w, d, ref))

    # the workspace entry point's result against the double-precision oracle on
    # a few nodes of each shape (bf16: max-abs 2e-2, mean-abs 2e-3)
    for name, w, d, ref in cases:
        B, N = w["parents"].shape
        spec = w["spec"]
        sel = sorted({0, B * N - 1, (B * N) // 2, N - 1})
        want, rst = oracle.attention(w["q"], w["k_cache"], w["v_cache"], w["block_table"],
                                     w["prefix_lens"], oracle.tree_mask(w["parents"])[0],
                                     bf16=True, sel=sel, nthreads=8)
        assert (rst == 0).all()
        got = ref.float().cpu().numpy().reshape(B * N, spec.Hq, spec.d)[sel]
        err = np.abs(got.astype(np.float64) - want)
        assert err.max() <= 2e-2 and err.mean() <= 2e-3, (name, err.max(), err.mean())

    # interleaved no-allocation calls: each one after the first finds the
    # array as a call of another shape left it
    order = [0, 2, 1, 2, 0, 1]
    seen = {}
    for c in order:
        name, w, d, ref = cases[c]
        B = w["parents"].shape[0]
        out = torch.full_like(d["q"], float("nan"))
        st = torch.full((B,), -9, dtype=torch.int32, device="cuda")
        tv.tree_verify_attention_noalloc(d["q"], d["k"], d["v"], d["bt"], d["P"], d["mask"],
                                         out, st)
        torch.cuda.synchronize()
        seen[name] = seen.get(name, 0) + 1
        tag = f"{name} call {seen[name]}"
        assert (st == 0).all(), tag
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), tag
    assert all(v == 2 for v in seen.values())


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
