"""Benchmark: one EAGLE tree-verification step on GB300.

A step is the whole hot path on one batch: tree_mask_build ->
tree_verify_attention -> tree_accept -> kv_compact, through the C ABI of
libtreeverify.  Inputs are synthetic (seeded, see workloads/) and resident in
HBM; L2 is flushed (a write of twice its size) before every timed step, and
each step is timed with CUDA events on the stream the kernels run on.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle on the same workload

Prints one JSON line (rank 0).  Under torchrun each rank runs its own copy of
the batch (the path shards by sequence, no collective on the data path) and
the slowest rank's time is reported.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "tree-verify tokens/s (attn+accept+compact)"
SLEEP_CYCLES = 400_000  # ~0.2 ms of GPU time queued ahead of each timed step
UNIT = "tokens/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=W.DEFAULT_BENCH, choices=list(W.SPECS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def slowest_rank(ms: float, world: int, device="cuda") -> float:
    """The largest of every rank's `ms` (an all-reduce MAX); `ms` itself alone."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world: int, B: int, N: int, ms_per_step: float) -> float:
    """Tokens per second of the whole job: every rank verifies its own B x N nodes
    per step, and the job's step time is the slowest rank's."""
    return world * B * N / (ms_per_step * 1e-3)


# ---------------------------------------------------------------- algorithmic work

def attn_kv_bytes(w) -> int:
    """Algorithmic bytes of one attention launch: the K and V rows of every
    sequence (prefix plus the tree's own positions), once per kv head."""
    s = w["spec"]
    e = 2 if s.bf16 else 4
    return int(np.sum(w["prefix_lens"].astype(np.int64) + w["parents"].shape[1])) * \
        s.Hkv * s.d * e * 2


def attn_qo_bytes(w) -> int:
    """Q read and O written by one attention launch (reported beside the K/V
    bytes; about 1 % of them on the batched workloads)."""
    s = w["spec"]
    e = 2 if s.bf16 else 4
    B, N = w["parents"].shape
    return B * N * s.Hq * s.d * e * 2


def accept_bytes(w, accept_len) -> int:
    """Rows the acceptance rule needs: greedy, the accepted path's rows
    (depth + 1 per sequence); stochastic, the two rows of the residual at the
    first rejection (one target row when everything is accepted)."""
    s = w["spec"]
    V = s.V
    if s.mode == "greedy":
        return int(np.sum(accept_len.astype(np.int64) + 1)) * V * 4
    K = w["parents"].shape[1] - 1
    rows = np.where(accept_len >= K, 1, 2)
    return int(rows.sum()) * V * 4


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (FileNotFoundError, OSError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- CPU oracle

def oracle_step(orc, w, nodes_frac=1.0, nthreads=1):
    """The oracle on one step of the workload; attention on a leading fraction
    of the nodes.  Returns (seconds, tokens covered)."""
    s = w["spec"]
    B, N = w["parents"].shape
    mp = W.max_path_len(w["parents"])
    t0 = time.perf_counter()
    mask, _, _ = orc.tree_mask(w["parents"])
    n_sel = max(1, int(round(B * N * nodes_frac)))
    sel = None if n_sel >= B * N else list(range(n_sel))
    orc.attention(w["q"], w["k_cache"], w["v_cache"], w["block_table"], w["prefix_lens"], mask,
                  bf16=s.bf16, sel=sel, nthreads=nthreads)
    if s.mode == "greedy":
        acc, path, _, _ = orc.accept_greedy(w["parents"], w["draft_tokens"], w["logits"], mp)
    else:
        acc, path, _, _ = orc.accept_stochastic(w["parents"], w["draft_tokens"], w["p"],
                                                w["q_probs"], w["seed"], w["offset"], mp)
    kc, vc = w["k_cache"].copy(), w["v_cache"].copy()
    orc.kv_compact(kc, vc, w["block_table"], w["prefix_lens"], path, acc)
    dt = time.perf_counter() - t0
    return dt, B * N * (n_sel / (B * N))


def pick_fraction(orc, w, budget_s, nthreads):
    """Fraction of nodes whose oracle step takes about budget_s seconds: the
    step's cost is fitted as a fixed part (mask, acceptance, compaction) plus a
    part per attention node, from one node and from four nodes per thread."""
    total = w["parents"].size
    n1, n2 = 1, min(total, 4 * nthreads)
    t1, _ = oracle_step(orc, w, nodes_frac=n1 / total, nthreads=nthreads)
    t2, _ = oracle_step(orc, w, nodes_frac=n2 / total, nthreads=nthreads)
    per_node = max((t2 - t1) / max(n2 - n1, 1), 1e-6)
    fixed = max(t1 - per_node, 0.0)
    return float(min(1.0, max(budget_s - fixed, per_node) / (per_node * total)))


def cpu_baseline(w, budget_s=12.0):
    import oracle as orc
    orc.build()
    nthreads = os.cpu_count() or 1
    frac = pick_fraction(orc, w, budget_s, nthreads)
    t, tokens = oracle_step(orc, w, frac, nthreads)
    steps = 1
    while frac >= 1.0 and t < budget_s and t / steps < budget_s - t:  # whole steps, repeated
        dt, tok = oracle_step(orc, w, frac, nthreads)
        t, tokens, steps = t + dt, tokens + tok, steps + 1
    B, N = w["parents"].shape
    return {"value": tokens / t, "unit": UNIT, "cores": nthreads, "kind": "oracle",
            "sample": f"{frac * 100:.1f}% of the {B * N} tree nodes in attention (all nodes "
                      f"in mask/accept/compaction), {steps} step(s), {t:.1f} s"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle as orc
    orc.build()
    w = W.make(args.workload)
    nthreads = os.cpu_count() or 1
    frac = pick_fraction(orc, w, 6.0, nthreads)
    for _ in range(min(args.warmup, 1)):
        oracle_step(orc, w, frac, nthreads)
    total_t, total_tok = 0.0, 0.0
    for _ in range(args.steps):
        t, tok = oracle_step(orc, w, frac, nthreads)
        total_t += t
        total_tok += tok
    value = total_tok / total_t
    s = w["spec"]
    B, N = w["parents"].shape
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * total_t / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": nthreads, "kind": "oracle",
                             "sample": f"{frac * 100:.1f}% of the {B * N} tree nodes in attention "
                                       f"per step (all nodes in mask/accept/compaction)"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def workload_config(w):
    s = w["spec"]
    B, N = w["parents"].shape
    P = w["prefix_lens"]
    return {"workload": s.name, "batch": B, "tree_nodes": N, "prefix_min": int(P.min()),
            "prefix_max": int(P.max()), "q_heads": s.Hq, "kv_heads": s.Hkv, "head_dim": s.d,
            "block_size": s.bs, "vocab": s.V, "accept": s.mode,
            "kv_dtype": "bf16" if s.bf16 else "f32", "l2": "flushed before every step"}


# ---------------------------------------------------------------- measured traffic

def measured_traffic(kernel_file: str, workload: str):
    """DRAM bytes per launch from a committed ncu capture, when the kernel
    source still matches the capture."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    try:
        rec = json.load(open(path)).get(workload, {}).get(kernel_file)
    except (OSError, ValueError):
        return None
    if not rec:
        return None
    src = os.path.join(ROOT, "eagle_speculative_decoding_parent_gb300", "csrc", kernel_file)
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    return rec["bytes_per_launch"] if rec.get("source_sha") == sha else None


# ---------------------------------------------------------------- GPU arm

def run_ours(args):
    import torch
    import torch.distributed as dist

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    import eagle_speculative_decoding_parent_gb300 as tv
    from eagle_speculative_decoding_parent_gb300.pipeline import VerifyStep

    w = W.make(args.workload)
    s = w["spec"]
    B, N = w["parents"].shape
    mp = W.max_path_len(w["parents"])
    bf = s.bf16
    mode = tv.GREEDY if s.mode == "greedy" else tv.STOCHASTIC

    def dev(a, as_bf16=False):
        t = torch.from_numpy(np.ascontiguousarray(a))
        if as_bf16:
            t = t.view(torch.int16).view(torch.bfloat16)
        return t.cuda()

    d = {k: dev(w[k]) for k in ("parents", "prefix_lens", "block_table", "draft_tokens")}
    for k in ("q", "k_cache", "v_cache"):
        d[k] = dev(w[k], bf)
    target = dev(w["logits"] if mode == tv.GREEDY else w["p"])
    draft = None if mode == tv.GREEDY else dev(w["q_probs"])
    seed, offset = w.get("seed", 0), w.get("offset", 0)
    dtype = d["q"].dtype
    step = VerifyStep(B=B, N=N, Hq=s.Hq, Hkv=s.Hkv, d=s.d, max_blocks=w["block_table"].shape[1],
                      bs=s.bs, dtype=dtype, max_path=mp, V=s.V, mode=mode)
    # kernels per step: mask and compaction launch one each; attention one, or two
    # when it takes the balanced schedule (a merge kernel follows); acceptance one,
    # or two for the stochastic rule on trees of more than two nodes (chains, then
    # branching trees)
    accept_kernels = 2 if (mode == tv.STOCHASTIC and N > 2) else 1
    attn_kernels = tv.tree_verify_attention_kernels(
        B, N, s.Hq, s.Hkv, s.d, w["block_table"].shape[1], s.bs, dtype,
        step.workspace.numel())
    stream = torch.cuda.current_stream()
    l2 = torch.cuda.get_device_properties(local).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device="cuda")

    def one_step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        step.mask_build(d["parents"])
        if ev is not None:
            ev[1].record(stream)
        step.attention(d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["prefix_lens"])
        if ev is not None:
            ev[2].record(stream)
        step.accept(mode, d["parents"], d["draft_tokens"], target, draft, seed, offset)
        if ev is not None:
            ev[3].record(stream)
        step.compact(d["k_cache"], d["v_cache"], d["block_table"], d["prefix_lens"])
        if ev is not None:
            ev[4].record(stream)

    for _ in range(max(3, args.warmup)):
        flush.fill_(1)
        one_step()
    torch.cuda.synchronize()

    # timed region: the four kernels of each step back to back (no events
    # between them, so each kernel may start while the previous one drains)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    sampler = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    wall0 = time.perf_counter()
    for k in range(args.steps):
        flush.fill_(k & 0xFF)
        # keep the GPU busy while the host enqueues the step, so the event
        # intervals hold device time only (no host launch gaps)
        torch.cuda._sleep(SLEEP_CYCLES)
        evs[k][0].record(stream)
        one_step()
        evs[k][1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    step_ms = np.array([evs[k][0].elapsed_time(evs[k][1]) for k in range(args.steps)])
    total_ms = float(step_ms.sum())

    # per-kernel durations (events between the kernels), same inputs and flush
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    for k in range(args.steps):
        flush.fill_(k & 0xFF)
        torch.cuda._sleep(SLEEP_CYCLES)
        one_step(kev[k])
    torch.cuda.synchronize()
    per = np.array([[kev[k][j].elapsed_time(kev[k][j + 1]) for j in range(4)]
                    for k in range(args.steps)])  # ms: mask, attn, accept, compact
    total_ms = slowest_rank(total_ms, world)
    ms_per_step = total_ms / args.steps
    value = whole_job_rate(world, B, N, ms_per_step)
    acc_len = step.accept_len.cpu().numpy()
    names = ["tree_mask_build", "tree_verify_attention", "tree_accept", "kv_compact"]
    mean_ms = per.mean(axis=0)

    # roofline of the dominant kernel
    dom = int(np.argmax(mean_ms))
    peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) \
        if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")) else None
    peak = peaks["hbm_gbs"] if peaks else 6800.0
    alg = {1: attn_kv_bytes(w), 2: accept_bytes(w, acc_len)}.get(dom)
    G = s.Hq // s.Hkv
    tc = bf and s.d == 128 and G <= 128  # the tensor-memory attention kernel
    files = {0: "tree_mask.cu", 1: ("attn_tc.cu" if tc else "attn_bf16.cu") if bf else "attn_f32.cu",
             2: "accept.cu", 3: "kv_compact.cu"}
    if alg is None:
        # mask / compaction: bytes moved by the definition
        alg = (B * N * 4 + B * N * 12) if dom == 0 else \
            int(np.sum(acc_len + 1)) * s.Hkv * s.d * (2 if bf else 4) * 4
    achieved = alg / (mean_ms[dom] * 1e-3) / 1e9
    roofline = {"kernel": names[dom], "bound": "hbm", "achieved": achieved, "peak": peak,
                "unit": "GB/s", "frac": achieved / peak,
                "peak_source": "measured" if peaks else "fallback",
                "traffic": measured_traffic(files[dom], s.name),
                "algorithmic_bytes_per_launch": alg,
                "bytes_definition": {1: "K+V rows read (prefix + tree, once per kv head)",
                                     2: "rows the acceptance rule needs"}.get(dom, "definition")}
    attn_gbs = attn_kv_bytes(w) / (mean_ms[1] * 1e-3) / 1e9
    attn_gbs_qo = (attn_kv_bytes(w) + attn_qo_bytes(w)) / (mean_ms[1] * 1e-3) / 1e9

    # end to end through the C ABI with host buffers (pinned), copies timed
    inputs = {"q": w["q"], "parents": w["parents"], "draft_tokens": w["draft_tokens"],
              "block_table": w["block_table"], "prefix_lens": w["prefix_lens"],
              "target": w["logits"] if mode == tv.GREEDY else w["p"]}
    if mode != tv.GREEDY:
        inputs["draft"] = w["q_probs"]
    host_in = {k: torch.from_numpy(np.ascontiguousarray(v)).pin_memory() for k, v in inputs.items()}
    if bf:
        host_in["q"] = host_in["q"].view(torch.int16).view(torch.bfloat16)
    dev_in = {"q": d["q"], "parents": d["parents"], "draft_tokens": d["draft_tokens"],
              "block_table": d["block_table"], "prefix_lens": d["prefix_lens"], "target": target}
    if draft is not None:
        dev_in["draft"] = draft
    outs = {"out": step.out, "accept_len": step.accept_len, "out_tokens": step.out_tokens,
            "new_lens": step.new_lens}
    host_out = {k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in outs.items()}
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out.values())

    def e2e_step():
        for k, t in host_in.items():
            dev_in[k].copy_(t, non_blocking=True)
        one_step()
        for k, t in outs.items():
            host_out[k].copy_(t, non_blocking=True)

    for _ in range(3):
        flush.fill_(2)
        e2e_step()
    torch.cuda.synchronize()
    e_ms = []
    for k in range(args.steps):
        flush.fill_(k & 0xFF)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        e2e_step()
        b.record(stream)
        b.synchronize()
        e_ms.append(a.elapsed_time(b))
    e2e_ms = slowest_rank(float(np.mean(e_ms)), world)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms_per_step,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16" if bf else "f32", "data": "synthetic",
                "config": workload_config(w),
                "roofline": roofline,
                "cpu_baseline": cpu,
                "e2e": {"value": whole_job_rate(world, B, N, e2e_ms), "unit": UNIT,
                        "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
                "gpu_launches": (2 + accept_kernels + attn_kernels) * args.steps,
                "clocks": clocks,
                "kernel_ms": {n: float(m) for n, m in zip(names, mean_ms)},
                "attention_kv_gbs": attn_gbs,
                "attention_kv_qo_gbs": attn_gbs_qo,
                "accepted_tokens_per_s": world * float(np.sum(acc_len + 1)) / (ms_per_step * 1e-3),
                "mean_accept_len": float(np.mean(acc_len)),
                "wall_s_timed_region": wall}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
