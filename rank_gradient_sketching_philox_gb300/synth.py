"""Seeded synthetic inputs: the workloads' shapes and value distributions.

This module holds no arithmetic of the sketching method.  It draws W, X and D
with torch's own generators (CPU for parity cases, CUDA for large benchmark
buffers) and describes the layer stacks the method is run on.  The same
tensors feed both the GPU library and the CPU oracle.

Distributions: W ~ N(0, 0.02) (standard deviation), X ~ N(0, 1), D ~ N(0, 1e-3),
all stored as BF16.  The long-response workload makes about 5% of the token rows
of D ten times larger (heavy-tailed rows).
"""
from dataclasses import dataclass, field
from typing import List, Tuple

import torch

W_STD = 0.02
X_STD = 1.0
D_STD = 1e-3


def normal_bf16(shape, std, seed, device="cpu"):
    """BF16 tensor of N(0, std^2) draws from a generator seeded with ``seed``."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    t = torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32)
    return (t * std).to(torch.bfloat16)


def heavy_tail_rows(D, frac, factor, seed):
    """Scale a seeded random subset (each row with probability ``frac``) of the
    token rows of D by ``factor``; returns a new tensor."""
    g = torch.Generator(device=D.device)
    g.manual_seed(int(seed))
    pick = torch.rand(D.shape[0], generator=g, device=D.device) < frac
    scale = torch.where(pick, torch.tensor(float(factor), device=D.device),
                        torch.tensor(1.0, device=D.device))
    return (D.float() * scale[:, None]).to(torch.bfloat16)


def seed_w(layer):
    return 1000 + layer


def seed_x(layer, microbatch):
    return 1_000_000 + 1000 * layer + 2 * microbatch


def seed_d(layer, microbatch):
    return 1_000_000 + 1000 * layer + 2 * microbatch + 1


def layer_weight(d, k, layer, device="cpu"):
    return normal_bf16((d, k), W_STD, seed_w(layer), device)


def layer_x(T, k, layer, microbatch, device="cpu"):
    return normal_bf16((T, k), X_STD, seed_x(layer, microbatch), device)


def layer_d(T, d, layer, microbatch, device="cpu", heavy_tail=False):
    D = normal_bf16((T, d), D_STD, seed_d(layer, microbatch), device)
    if heavy_tail:
        D = heavy_tail_rows(D, 0.05, 10.0, seed_d(layer, microbatch) + 7_000_000)
    return D


@dataclass
class Workload:
    """A stack of linear layers, each (d, k) = (out width, in width)."""
    name: str
    layers: List[Tuple[str, int, int]]
    ranks: List[int]
    tokens_per_step: int
    microbatch: int
    projection: str          # "rademacher-fixed", "qr-refreshed", or "both"
    update: str              # "normsgd" or "sgd"
    step_size: float         # tau for normsgd, alpha*eta for sgd
    heavy_tail: bool = False
    notes: str = ""

    @property
    def microbatches(self):
        return max(1, self.tokens_per_step // self.microbatch)

    @property
    def weights(self):
        return sum(d * k for _, d, k in self.layers)


def _block(prefix, hidden, kv, inter):
    return [(prefix + "q", hidden, hidden), (prefix + "k", kv, hidden), (prefix + "v", kv, hidden),
            (prefix + "o", hidden, hidden), (prefix + "gate", inter, hidden),
            (prefix + "up", inter, hidden), (prefix + "down", hidden, inter)]


def input_groups(layers):
    """Indices of the layers that read the same input X, in order: q, k and v
    of a block read the attention input, gate and up the MLP input; every
    other layer reads its own."""
    groups, open_ = [], {}
    for li, (name, _, _) in enumerate(layers):
        prefix, _, kind = name.rpartition(".")
        key = (prefix, "attn") if kind in ("q", "k", "v") else (prefix, "mlp") if kind in ("gate", "up") else None
        if key is None:
            groups.append([li])
        elif key in open_:
            groups[open_[key]].append(li)
        else:
            open_[key] = len(groups)
            groups.append([li])
    return groups


def qwen3_stack(blocks, hidden, kv, inter):
    layers = []
    for b in range(blocks):
        layers += _block("b%d." % b, hidden, kv, inter)
    return layers


WORKLOADS = {
    "single-linear-256x512": Workload(
        "single-linear-256x512", [("w", 256, 512)], [16], 512, 128, "both", "normsgd", 1e-3),
    "logra-4096x4096": Workload(
        "logra-4096x4096", [("w", 4096, 4096)], [64], 32768, 4096, "rademacher-fixed", "sgd", 1e-4),
    "qwen3-1.7b-stack": Workload(
        "qwen3-1.7b-stack", qwen3_stack(28, 2048, 1024, 6144), [64, 128, 256], 32768, 4096,
        "qr-refreshed", "normsgd", 1e-3),
    "qwen3-8b-stack": Workload(
        "qwen3-8b-stack", qwen3_stack(36, 4096, 1024, 12288), [64], 32768, 4096,
        "qr-refreshed", "normsgd", 1e-3),
    "long-response-sweep": Workload(
        "long-response-sweep", [("sq", 8192, 8192), ("up", 28672, 8192)], [4, 16, 64, 256],
        131072, 16384, "both", "normsgd", 1e-3, heavy_tail=True,
        notes="tokens per step swept over 1024, 8192, 65536, 131072; microbatch = min(T, 16384)"),
}
