"""Policy sync by sketch: ship the d x r factor and the seed, not the weights.

A trainer that updates W <- W - alpha*eta * U P^T can send U (scaled by
alpha*eta) and the Philox seed to its rollout workers; each worker
regenerates P from (seed, layer, step) and applies the same update to its
own copy of W ("LoGRA: Scaling LLM Reinforcement Learning with Low-Rank
Gradient Sketches", Key Contributions: the sketch and the seed are what
travels; "LoGRA: Low-Rank Gradient Sketches", "Why the Update Is Low-Rank and
Cheap to Sync").  When the trainer applies the same payload the same way,
the two W agree bit for bit: both run the identical rebuild, the identical
fused multiply-add and the identical stochastic-rounding stream.

The payload is 4*d*r bytes of U plus 16 bytes of (seed, layer, step) against
2*d*k bytes of BF16 weights.
"""
import torch

from . import binding


def payload(C, alpha_eta):
    """U = fl32(alpha_eta * C): the factor to send (d x r fp32)."""
    if C.dtype != torch.float32:
        raise TypeError("C must be float32")
    return C * torch.tensor(alpha_eta, dtype=torch.float32, device=C.device)


def payload_bytes(d, r):
    """Bytes on the wire per layer: U (4 d r) plus seed (8), layer (4) and step (4)."""
    return 4 * d * r + 16


def apply(W, U, P, seed, layer, step, dev_status=None, stream=None):
    """W <- SR_bf16(W - U P^T) with the (seed, layer, step) rounding stream; the
    scale is already in U.  Trainer and workers both call this."""
    return binding.apply_update_sgd(W, U, P, 1.0, seed, layer, step, dev_status=dev_status, stream=stream)
