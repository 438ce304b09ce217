"""Helpers shared by the GPU tests: move seeded workload inputs to the device
and compare GPU results with oracle values at the stated tolerances."""
import numpy as np
import torch

TOL = {"f32": 1e-5, "bf16": 2e-2}

# |GPU noise - oracle noise| per entry, in units of sigma C.  The gradient
# kernels draw the Gaussian mechanism's normals with the SFU's log2, sine and
# cosine (a series for the log near 1); test_gradient_noise_is_the_oracle_stream
# bounds the difference from the oracle's fp64 Box-Muller over a full
# 2048 x 8192 draw (1.7e-6 at most there).
NOISE_TOL = 5e-6

# A gradient check whose allowance exceeds this fraction of the clipped sum's
# largest entry could pass a wrong GEMM; every check asserts it stays below.
MAX_ALLOWANCE = 0.05

U32 = 2.0 ** -24   # unit roundoff of fp32


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
    (|error| <= K u * sum |terms| for a sum of K terms, u = 2^-24)."""
    mag = None
    for i in range(A.shape[0]):
        t = s[i] * (np.abs(A[i]).astype(np.float64).T @ np.abs(G[i]).astype(np.float64))
        mag = t if mag is None else mag + t
    return mag


def assert_grad(got, S, tol, K, mag, noise=None, sigmaC=0.0, slack=0.0, what="grad"):
    """Compare a GPU gradient with the oracle's clipped sum S = sum_i s_i M_i,
    after taking away the oracle's noise sigma C z (`noise`, None for sigma = 0),
    so that the check sees the GEMM however large the noise is:

      normwise   max|got - noise - S| <= tol max|S| + NOISE_TOL sigma C
      per entry  |got - noise - S| <= tol |S| + 4 K u mag + NOISE_TOL sigma C

    K = B T is the accumulation length and mag = sum_i s_i |A_i|^T |G_i|: an
    fp32 sum of K terms is off by at most about K u sum|terms| (the factor 4
    covers the per-sample scaling, the final additions and a tensor core that
    truncates instead of rounding).  `slack` (scalar or per entry) is added to
    both bounds for a result that went through another rounding (an update of
    parameters).  The normwise allowance must stay below MAX_ALLOWANCE of
    max|S|: a check that noise or a loose bound swamps fails here instead of
    passing whatever the GEMM returned."""
    got = np.asarray(got, dtype=np.float64)
    resid = got - (0.0 if noise is None else noise)
    err = np.abs(resid - S)
    smax = float(np.abs(S).max())
    slack_max = float(np.max(slack))
    allow = tol * smax + NOISE_TOL * sigmaC + slack_max
    assert smax > 0.0, f"{what}: the clipped sum is zero, nothing to compare"
    assert allow <= MAX_ALLOWANCE * smax, (
        f"{what}: allowance {allow:.3e} is {allow / smax:.3f} of max|S| = {smax:.3e}")
    assert err.max() <= allow, (
        f"{what}: normwise error {err.max() / smax:.3e} of max|S| (allowed {allow / smax:.3e})")
    bound = tol * np.abs(S) + 4.0 * K * U32 * mag + NOISE_TOL * sigmaC + slack
    bad = err > bound
    assert not bad.any(), (
        f"{what}: {bad.sum()} entries outside tol|S| + 4 K u mag + NOISE_TOL sigma C "
        f"(worst {np.max(err / bound):.2f} of its bound)")


def assert_flags(got, n_ref, C, tol, what="flags"):
    got = np.asarray(got).astype(bool)
    away = np.abs(n_ref - C) > 4 * tol * C
    assert np.array_equal(got[away], (n_ref > C)[away]), what
