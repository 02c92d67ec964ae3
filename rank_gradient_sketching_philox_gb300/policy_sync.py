"""Policy sync by sketch: ship the d x r factor and the seed, not the weights.

A trainer that updates W <- W - alpha*eta * U P^T sends its rollout workers
the factor U, the step size alpha*eta and the Philox seed; each worker
regenerates P from (seed, layer, step) and applies the same update to its own
copy of W ("LoGRA: Scaling LLM Reinforcement Learning with Low-Rank Gradient
Sketches", Key Contributions: the sketch and the seed are what travels;
"LoGRA: Low-Rank Gradient Sketches", "Why the Update Is Low-Rank and Cheap to
Sync").  The step size travels as a number and is applied inside the update
kernel (v = fmaf(-alpha*eta, H, w)), so no arithmetic happens outside the
library and the trainer and every worker run the identical rebuild, fused
multiply-add and stochastic-rounding stream: their W agree bit for bit.

The payload is 4*d*r bytes of U plus 20 bytes of (alpha*eta, seed, layer,
step) against 2*d*k bytes of BF16 weights.
"""
from typing import NamedTuple

import torch

from . import binding


class Message(NamedTuple):
    """What one layer's update sends: U (d x r fp32), alpha*eta, and the
    projection's (seed, layer, step)."""
    U: torch.Tensor
    alpha_eta: float
    seed: int
    layer: int
    step: int


def message(C, alpha_eta, seed, layer, step):
    """The message of an SGD update W <- W - alpha_eta * C P^T: the sketch C
    itself (U = C in LoGRA's basic SGD) and the scalars; nothing is computed."""
    if C.dtype != torch.float32:
        raise TypeError("C must be float32")
    return Message(C, float(alpha_eta), int(seed), int(layer), int(step))


def payload_bytes(d, r):
    """Bytes on the wire per layer: U (4 d r) plus alpha*eta (4), seed (8),
    layer (4) and step (4)."""
    return 4 * d * r + 20


def apply(W, msg, P, dev_status=None, stream=None):
    """W <- SR_bf16(W - alpha_eta U P^T) with the message's rounding stream.
    P is the regenerated projection of (msg.seed, msg.layer, msg.step).  The
    trainer and every worker call this with the same message."""
    return binding.apply_update_sgd(W, msg.U, P, msg.alpha_eta, msg.seed, msg.layer, msg.step,
                                    dev_status=dev_status, stream=stream)
