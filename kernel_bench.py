"""Times one entry point of the verification step alone, on a named workload.

bench.py times the whole step; this times a single C-ABI call (or, for the
draft tree, the calls that build one tree) with the same hygiene: inputs
resident in HBM, L2 flushed by a write of twice its size before every timed
call, a spin kernel queued ahead so the events hold device time only, CUDA
events on the launching stream.  It is also the command the per-kernel ncu
summaries are captured on (select the kernel with ``ncu -k``).

  python kernel_bench.py --entry accept --workload llama3_8b_b32_tree26
  python kernel_bench.py --entry accept_walk --workload llama3_8b_b32_tree26
  python kernel_bench.py --entry accept --workload llama3_8b_b32_tree26 --mode stochastic
  python kernel_bench.py --entry mask|compact|append --workload NAME
  python kernel_bench.py --entry draft --B 32 --V 128256 --topk 10 --layers 6 --N 60

Prints one JSON line: the entry point, the workload, the mean and minimum
device time per call (microseconds) and the bytes the operation needs by its
definition, with the rate they give.
"""
from __future__ import annotations

import argparse
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

SLEEP_CYCLES = 400_000
ENTRIES = ("mask", "attention", "accept", "accept_walk", "compact", "append", "draft")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--entry", required=True, choices=ENTRIES)
    ap.add_argument("--workload", default=W.DEFAULT_BENCH, choices=list(W.SPECS))
    ap.add_argument("--mode", choices=["greedy", "stochastic"], default=None,
                    help="acceptance rule (default: the workload's own)")
    ap.add_argument("--reps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    # draft tree shape
    ap.add_argument("--B", type=int, default=32)
    ap.add_argument("--V", type=int, default=128256)
    ap.add_argument("--topk", type=int, default=10)
    ap.add_argument("--layers", type=int, default=6)
    ap.add_argument("--N", type=int, default=60)
    return ap.parse_args()


def timed(fn, reps, warmup, flush, stream, sleep_cycles=SLEEP_CYCLES):
    import torch
    for _ in range(max(3, warmup)):
        flush.fill_(1)
        fn()
    torch.cuda.synchronize()
    ts = []
    for k in range(reps):
        flush.fill_(k & 0xFF)
        torch.cuda._sleep(sleep_cycles)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b) * 1e3)
    return float(np.mean(ts)), float(np.min(ts))


def main():
    args = parse()
    import torch
    import eagle_speculative_decoding_parent_gb300 as tv

    dev = torch.device("cuda")
    stream = torch.cuda.current_stream()
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    i32 = dict(dtype=torch.int32, device=dev)

    def put(a, as_bf16=False):
        t = torch.from_numpy(np.ascontiguousarray(a))
        if as_bf16:
            t = t.view(torch.int16).view(torch.bfloat16)
        return t.to(dev)

    line = {"entry": args.entry}
    if args.entry == "draft":
        B, V, k, L, N = args.B, args.V, args.topk, args.layers, args.N
        rng = np.random.default_rng(0)
        rows = [put((3.0 * rng.standard_normal((B, 1 if l == 0 else k, V))).astype(np.float32))
                for l in range(L)]
        roots = put(rng.integers(0, V, size=B).astype(np.int32))
        ws = torch.zeros(tv.draft_tree_workspace(B, k, L), dtype=torch.uint8, device=dev)
        status = torch.zeros(B, **i32)
        ft = torch.zeros((B, k), **i32)
        fs = torch.zeros((B, k), **i32)
        par = torch.zeros((B, N), **i32)
        tok = torch.zeros((B, N), **i32)
        sc = torch.zeros((B, N), dtype=torch.float32, device=dev)

        def tree():
            ws.zero_()
            for layer in range(L):
                last = layer == L - 1
                tv.draft_tree_expand(rows[layer], layer, L, status, ws, topk=k, root_tokens=roots,
                                     N=N, front_tokens=ft, front_src=fs,
                                     parents=par if last else None, tokens=tok if last else None,
                                     scores=sc if last else None)
        # the spin covers the host's enqueue of all the tree's calls, so the
        # events hold device time only
        mean, best = timed(tree, args.reps, args.warmup, flush, stream, sleep_cycles=8_000_000)
        assert (status == 0).all().item()
        need = sum(r.numel() for r in rows) * 4
        line.update(workload=f"draft tree B={B} V={V} topk={k} layers={L} N={N}",
                    us_per_tree=mean, us_min=best, us_per_layer=mean / L,
                    bytes_needed=need, bytes_definition="every draft logit read once (B*F*V*4 per layer)",
                    gbs=need / (mean * 1e-6) / 1e9, note="includes one 1-launch workspace clear")
        print(json.dumps(line), flush=True)
        return

    over = {"mode": args.mode} if args.mode else {}
    parts = ("attn", "accept") if args.entry in ("attention", "compact", "append") else ("accept",)
    if args.entry == "mask":
        parts = ()
    w = W.make(args.workload, parts=parts, **over)
    s = w["spec"]
    B, N = w["parents"].shape
    par = put(w["parents"])
    line["workload"] = s.name + (f" ({args.mode} acceptance)" if args.mode else "")
    mask = torch.zeros((B, N), dtype=torch.int64, device=dev)
    depth = torch.zeros((B, N), **i32)
    st = torch.zeros(B, **i32)
    tv.tree_mask_build(par, mask, depth, st)

    if args.entry == "mask":
        fn = lambda: tv.tree_mask_build(par, mask, depth, st)  # noqa: E731
        need, what = B * N * 4 + B * N * 12, "parents read, mask and depth written"
    elif args.entry == "attention":
        q, kc, vc = (put(w[x], s.bf16) for x in ("q", "k_cache", "v_cache"))
        bt, P = put(w["block_table"]), put(w["prefix_lens"])
        out = torch.zeros_like(q)
        ws = torch.zeros(max(256, tv.tree_verify_attention_workspace(
            B, N, s.Hq, s.Hkv, s.d, bt.shape[1], s.bs, q.dtype)), dtype=torch.uint8, device=dev)
        fn = lambda: tv.tree_verify_attention(q, kc, vc, bt, P, mask, out, st, ws)  # noqa: E731
        e = 2 if s.bf16 else 4
        need = int(np.sum(w["prefix_lens"].astype(np.int64) + N)) * s.Hkv * s.d * e * 2
        what = "K+V rows read (prefix + tree, once per kv head)"
    elif args.entry in ("accept", "accept_walk"):
        greedy = s.mode == "greedy"
        mode = tv.GREEDY if greedy else tv.STOCHASTIC
        if args.entry == "accept_walk" and not greedy:
            raise SystemExit("accept_walk is the greedy rule without a workspace")
        mp = W.max_path_len(w["parents"])
        tok = put(w["draft_tokens"])
        target = put(w["logits"] if greedy else w["p"])
        draft = None if greedy else put(w["q_probs"])
        acc = torch.zeros(B, **i32)
        path = torch.zeros((B, mp), **i32)
        out_tok = torch.zeros((B, mp), **i32)
        wsz = tv.tree_accept_workspace(mode, B, N, s.V)
        if args.entry == "accept_walk" and wsz > 0:
            raise SystemExit("this shape takes the greedy row scan (it needs a workspace); "
                             "the walk serves the shapes whose workspace query returns 0")
        ws = torch.zeros(max(256, wsz), dtype=torch.uint8, device=dev) if wsz > 0 else None
        seed = w.get("seed", 0)
        fn = lambda: tv.tree_accept(mode, par, tok, target, draft, acc, path, out_tok, st,  # noqa: E731
                                    seed=seed, offset=0, workspace=ws)
        fn()
        torch.cuda.synchronize()
        a = acc.cpu().numpy().astype(np.int64)
        if greedy:
            need, what = int(np.sum(a + 1)) * s.V * 4, "target rows on the accepted path"
        else:
            # the rule's reads: every test on the path needs p and q at one token;
            # the first rejection's residual needs both rows whole (one p row when
            # every test passes)
            K = N - 1
            need = int(np.sum(np.where(a >= K, 1, 2))) * s.V * 4
            what = "rows of the residual at the first rejection (the target row when all pass)"
        line["rows_all_nodes_bytes"] = B * N * s.V * 4 * (1 if greedy else 2)
        line["mean_accept_len"] = float(a.mean())
        line["kernel"] = ("accept_walk_kernel" if wsz == 0 else "accept_rows_kernel") if greedy \
            else "accept_stochastic_kernel"
    elif args.entry == "compact":
        kc, vc = put(w["k_cache"], s.bf16), put(w["v_cache"], s.bf16)
        bt, P = put(w["block_table"]), put(w["prefix_lens"])
        mp = W.max_path_len(w["parents"])
        # an accepted path per sequence: its deepest leaf's root path (the
        # planted greedy path when the workload plants one)
        path_np = np.zeros((B, mp), np.int32)
        acc_np = np.zeros(B, np.int32)
        for b in range(B):
            j, chain = N - 1, []
            while j >= 0:
                chain.append(j)
                j = int(w["parents"][b, j])
            chain = chain[::-1][:mp]
            path_np[b, :len(chain)] = chain
            acc_np[b] = len(chain) - 1
        path, acc = put(path_np), put(acc_np)
        new_lens = torch.zeros(B, **i32)
        fn = lambda: tv.kv_compact(kc, vc, bt, P, path, acc, new_lens, st)  # noqa: E731
        e = 2 if s.bf16 else 4
        need = int(np.sum(acc_np + 1)) * s.Hkv * s.d * e * 2 * 2
        what = "accepted rows (root included): K and V read, then written"
    else:  # append
        kc, vc = put(w["k_cache"], s.bf16), put(w["v_cache"], s.bf16)
        bt, P = put(w["block_table"]), put(w["prefix_lens"])
        dt = torch.bfloat16 if s.bf16 else torch.float32
        kn = torch.randn((B, N, s.Hkv, s.d), device=dev).to(dt)
        vn = torch.randn((B, N, s.Hkv, s.d), device=dev).to(dt)
        fn = lambda: tv.tree_kv_append(kn, vn, depth, kc, vc, bt, P, st,  # noqa: E731
                                       rope_theta=500000.0)
        e = 2 if s.bf16 else 4
        need = B * N * s.Hkv * s.d * e * 2 * 2
        what = "new K and V rows read and written into the cache"

    mean, best = timed(fn, args.reps, args.warmup, flush, stream)
    torch.cuda.synchronize()
    assert (st == 0).all().item(), st.cpu().numpy()
    line.update(us=mean, us_min=best, bytes_needed=need, bytes_definition=what,
                gbs=need / (mean * 1e-6) / 1e9)
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
