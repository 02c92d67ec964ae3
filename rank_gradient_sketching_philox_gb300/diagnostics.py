"""Reconstruction diagnostic: how well the rebuilt update H = C P^T points along
the dense gradient G = D^T X, over ranks and projection kinds.

The sketch C = D^T (X P) and the projection come from the library (the same
kernels as training); the dense G is formed only here, as the thing H is
compared with.  Both G and H = C P^T are formed in float64 from the library's
C and P, so the measured cosine carries no rounding of this module's own.  ("LoGRA: Scaling LLM Reinforcement Learning with Low-Rank
Gradient Sketches", Experimental Findings: reconstruction cosine over ranks;
"LoGRA: Low-Rank Gradient Sketches", "Why Refreshing the Projection Enables New
Update Directions": averaging over refreshed projections recovers more of G.)

For one step the expected values are closed forms: a Rademacher projection
(entries +-1/sqrt(r)) gives E||H - G||^2 = ((k - 1)/r) ||G||^2 and E<G, H> =
||G||^2, so cos(G, H) ~ 1/sqrt(1 + (k - 1)/r); a QR frame scaled by sqrt(k/r)
gives E||H||^2 = (k/r) ||G||^2, so cos(G, H) ~ sqrt(r/k).  Averaging H over S
refreshed projections divides the excess by S: cos ~ 1/sqrt(1 + excess/S),
while a fixed projection stays where one step put it.
"""
import math

import torch

from . import binding


def expected_cosine(kind, k, r, steps=1):
    """Closed-form cos(G, mean H) for `steps` refreshed projections."""
    excess = (k - 1) / r if kind == binding.PROJ_RADEMACHER else k / r - 1.0
    return 1.0 / math.sqrt(1.0 + excess / steps)


def reconstruction(Ds, Xs, r, kind, steps=1, refreshed=True, seed=0, layer=0):
    """cos(G, H_mean) and ||H_mean - G|| / ||G|| for microbatches Ds (T x d BF16)
    and Xs (T x k BF16), with H_mean the mean of C_s P_s^T over `steps` steps
    (P refreshed each step, or the step-0 projection every time)."""
    dev = Xs[0].device
    d, k = Ds[0].shape[1], Xs[0].shape[1]
    G = sum(D.double().t() @ X.double() for D, X in zip(Ds, Xs))
    H = torch.zeros(d, k, dtype=torch.float64, device=dev)
    P = torch.empty(k, r, dtype=torch.float32, device=dev)
    C = torch.empty(d, r, dtype=torch.float32, device=dev)
    for s in range(steps):
        binding.sample_projection(kind, seed, layer, s if refreshed else 0, P)
        for m, (D, X) in enumerate(zip(Ds, Xs)):
            # row stride a multiple of 8 elements, as the library requires
            XP = torch.empty(X.shape[0], (r + 7) // 8 * 8, dtype=torch.bfloat16, device=dev)[:, :r]
            binding.project_inputs(X, P, XP)
            binding.accumulate(D, XP, C, overwrite=(m == 0))
        H += C.double() @ P.double().t()
    H /= steps
    gn = torch.linalg.norm(G)
    cos = float((G * H).sum() / (gn * torch.linalg.norm(H)))
    rel = float(torch.linalg.norm(H - G) / gn)
    return cos, rel


def sweep(Ds, Xs, ranks=(4, 16, 64, 256), steps=8):
    """Rows (kind, r, refreshed, steps, cos, expected cos, relative error) over
    ranks, both projection kinds, fixed and refreshed projections."""
    k = Xs[0].shape[1]
    rows = []
    for kind in (binding.PROJ_RADEMACHER, binding.PROJ_GAUSSIAN_QR):
        for r in ranks:
            if kind == binding.PROJ_GAUSSIAN_QR and r > k:
                continue
            for refreshed in (False, True):
                cos, rel = reconstruction(Ds, Xs, r, kind, steps=steps, refreshed=refreshed)
                rows.append({"kind": "rademacher" if kind == binding.PROJ_RADEMACHER else "qr", "r": r,
                             "refreshed": refreshed, "steps": steps, "cos": cos,
                             "expected_cos": expected_cosine(kind, k, r, steps if refreshed else 1),
                             "rel_err": rel})
    return rows
