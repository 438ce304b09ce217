"""Helpers shared by the GPU tests: move seeded workload inputs to the device
and compare GPU results with oracle values at the stated tolerances."""
import numpy as np
import torch

TOL = {"f32": 1e-5, "bf16": 2e-2}


def to_dev(inp, device="cuda"):
    if inp.wl.dtype == "bf16":
        A = torch.from_numpy(inp.A_dev.view(np.int16)).view(torch.bfloat16)
        G = torch.from_numpy(inp.G_dev.view(np.int16)).view(torch.bfloat16)
    else:
        A = torch.from_numpy(inp.A_dev)
        G = torch.from_numpy(inp.G_dev)
    return A.to(device).contiguous(), G.to(device).contiguous()


def host(x):
    return x.detach().double().cpu().numpy()


def assert_rel(got, ref, tol, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rel = np.abs(got - ref) / np.maximum(np.abs(ref), 1e-300)
    assert np.all(rel <= tol), f"{what}: max rel err {rel.max():.3e} > {tol} (got {got}, ref {ref})"


def grad_magnitude(A, G, s):
    """sum_i s_i |A_i|^T |G_i|: the sum of absolute terms behind each entry of
    the clipped sum, which bounds the rounding error of a fp32 accumulation
    (|error| <= K eps * sum |terms| for a dot product of length K)."""
    mag = None
    for i in range(A.shape[0]):
        t = s[i] * (np.abs(A[i]).astype(np.float64).T @ np.abs(G[i]).astype(np.float64))
        mag = t if mag is None else mag + t
    return mag


def assert_grad(got, ref, tol, sigmaC, what="grad", mag=None):
    """Normwise max|err| / max|ref| <= tol, and per entry
    |err| <= tol * (|ref| + sigma C + magnitude of the summed terms)."""
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - ref)
    normwise = err.max() / np.abs(ref).max()
    assert normwise <= tol, f"{what}: normwise error {normwise:.3e} > {tol}"
    bound = tol * (np.abs(ref) + sigmaC + (0.0 if mag is None else mag))
    bad = err > bound
    assert not bad.any(), f"{what}: {bad.sum()} entries outside tol*(|ref|+sigma*C)"


def assert_flags(got, n_ref, C, tol, what="flags"):
    got = np.asarray(got).astype(bool)
    away = np.abs(n_ref - C) > 4 * tol * C
    assert np.array_equal(got[away], (n_ref > C)[away]), what
