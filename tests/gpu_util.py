"""Helpers for the GPU parity tests (comparison metrics and conversions)."""
import numpy as np
import torch


def bits(t):
    """BF16 tensor -> np.uint16 bit patterns (on the host)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def from_bits(a, device):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)


def rel_fro(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def bf16_ulp_distance(a_bits, b_bits):
    """Distance in BF16 steps between two arrays of BF16 bit patterns (sign-aware)."""
    def key(x):
        x = np.asarray(x, np.uint16).astype(np.int32)
        mag = x & 0x7FFF
        return np.where(x & 0x8000, -mag, mag)
    return np.abs(key(a_bits) - key(b_bits))


def w_parity(got_bits, ref_bits):
    """Return (fraction bit-identical, max BF16-step distance)."""
    got_bits = np.asarray(got_bits, np.uint16)
    ref_bits = np.asarray(ref_bits, np.uint16)
    dist = bf16_ulp_distance(got_bits, ref_bits)
    return float(np.mean(got_bits == ref_bits)), int(dist.max()) if dist.size else 0
