"""Helpers shared by the GPU parity tests: move a synthetic workload to the
device and bring results back as numpy arrays."""
import numpy as np
import torch

from workloads import bf16_bits_to_f32


def dev(a, bf16=False):
    if bf16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host_f32(t):
    if t.dtype == torch.bfloat16:
        return bf16_bits_to_f32(t.view(torch.int16).cpu().numpy().view(np.uint16))
    return t.cpu().numpy()


def to_device(w):
    spec = w["spec"]
    d = {k: dev(w[k]) for k in ("parents", "prefix_lens", "block_table") if k in w}
    for k in ("q", "k_cache", "v_cache"):
        if k in w:
            d[k] = dev(w[k], bf16=spec.bf16)
    for k in ("draft_tokens", "logits", "p", "q_probs"):
        if k in w:
            d[k] = dev(w[k])
    return d
