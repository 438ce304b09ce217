"""fp64 CPU oracle of the per-linear-layer DP-SGD clipping path.

TEST INFRASTRUCTURE ONLY: imported by the tests, by the package smoke check and
by the benchmark's CPU-baseline / reference arm, never by the product path.  It
shares no code with the CUDA library: it has its own Philox, its own
Box-Muller, its own bf16 rounding and uses numpy's fp64 matmul and Householder
QR (LAPACK) as library steps.

Sources (cited by title and section throughout):
  GL  "DP-SGD (differentially private stochastic gradient descent)" glossary
      entry, jisaku.com -- section "DP-SGD algorithm", steps 1-5.
  RC  "Technical summary: efficient DP-SGD for LLMs with randomized clipping"
      (gist.science summary of arXiv 2605.24879) -- sections "Problem
      definition", "Core mechanism" (trace identity; item 1 Hutch; item 2
      Hutch++), "Algorithmic flow" (Algorithm 1, steps 1-5), "Key contributions
      1: complexity reduction".
  PH  J. Salmon, M. Moraes, R. Dror, D. Shaw, "Parallel random numbers: as easy
      as 1, 2, 3", SC'11 -- the Philox-4x32 bijection with 10 rounds.
  FB  "Technical summary: FIBER -- a differentially private optimizer with
      filter-aware innovation bias correction" (gist.science summary of arXiv
      2605.03425) -- section "Method: FIBER", A (innovation-space filtering)
      and C (filter-aware second-moment calibration).

Notation (RC, Core mechanism): for sample i, A_i is the T x d matrix of layer
inputs (activations), G_i the T x p matrix of output gradients, the per-sample
weight gradient is M_i = A_i^T G_i (d x p) and O_i = G_i^T A_i A_i^T G_i (p x p)
so that ||M_i||_F^2 = trace(O_i).

Readings where the pages are silent or garbled (each is listed with its reason
in the design notes):
  * Hutch is normalised by 1/k: q_i = (1/k) sum_j P_j^T O_i P_j (the summary
    prints the sum without the factor; 1/k is the only unbiased reading for
    N(0,1) probes).
  * One probe matrix P per call, shared by every sample (memory term kp has no
    B factor, RC Key contributions 1).
  * Hutch++ with a budget of k matrix products: r = floor(k/3) sketch columns S,
    r head columns Q, m = k - 2r tail probes scaled by 1/m.
  * Probes and noise come from Philox-4x32-10 (PH), key = 64-bit seed, counter
    = (element_index // 4, stream, offset low word, offset high word), lane =
    element_index % 4; streams 0 = P, 1 = S, 2 = G', 3 = noise.  Box-Muller:
    u = ((x >> 8) + 1) 2^-24 in (0, 1], v = (x >> 8) 2^-24 in [0, 1),
    lanes 0/1 = sqrt(-2 ln u(w0)) cos/sin(2 pi v(w1)), lanes 2/3 the same from
    words 2 and 3.
  * bf16 workloads use probes rounded to bfloat16 (nearest even).
  * Rademacher probes (the {+-1} sketches the summary names as future work,
    "Empirical results" / claims): element e is +1 when the top bit of word
    e % 4 of Philox block e // 4 is clear, -1 when it is set (same counters
    as the normals).
  * Noise N(0, sigma^2 C^2 I) is added once to the clipped sum; the 1/|B| of
    the SGD update (GL step 5) is not applied.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "STREAM_P", "STREAM_S", "STREAM_GP", "STREAM_NOISE",
    "philox4x32_10", "philox_normals", "philox_rademacher", "round_bf16", "probe_rows",
    "per_sample_grads", "sqnorms_direct", "sqnorms_trace", "sqnorms_ghost",
    "sqnorms_outer_bruteforce",
    "hutch_probe", "sqnorms_hutch", "hutchpp_split", "hutchpp_probes",
    "sqnorms_hutchpp", "clip_scales", "noise_matrix", "clipped_noisy_grad",
    "STREAM_BIAS_NOISE", "per_sample_bias_grads", "bias_sqnorms", "clipped_noisy_bias_grad",
    "sgd_update", "fiber_attenuation", "fiber_filter_step", "fiber_adamw_step",
]

STREAM_P, STREAM_S, STREAM_GP, STREAM_NOISE = 0, 1, 2, 3
STREAM_BIAS_NOISE = 4   # the bias gradient's noise (a stream of its own)

_MASK32 = np.uint64(0xFFFFFFFF)
# PH: Philox-4x32 multipliers and the Weyl key increments (golden ratio and
# sqrt(3) - 1, as 32-bit fractions).
_PHILOX_M0 = np.uint64(0xD2511F53)
_PHILOX_M1 = np.uint64(0xCD9E8D57)
_PHILOX_W0 = np.uint64(0x9E3779B9)
_PHILOX_W1 = np.uint64(0xBB67AE85)


def philox4x32_10(ctr, key):
    """Philox-4x32 with 10 rounds (PH).  `ctr`: 4 arrays (or ints) of 32-bit
    counter words, `key`: 2 32-bit key words.  Returns a uint32 array [..., 4].

    One round maps (c0, c1, c2, c3) with key (k0, k1) to
    (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2), hi(M0 c0) ^ c3 ^ k1, lo(M0 c0));
    the key is bumped by the Weyl increments before every round but the first.
    """
    c0, c1, c2, c3 = (np.asarray(c, dtype=np.uint64) & _MASK32 for c in ctr)
    k0 = np.uint64(int(key[0]) & 0xFFFFFFFF)
    k1 = np.uint64(int(key[1]) & 0xFFFFFFFF)
    for rnd in range(10):
        if rnd:
            k0 = (k0 + _PHILOX_W0) & _MASK32
            k1 = (k1 + _PHILOX_W1) & _MASK32
        prod0 = _PHILOX_M0 * c0          # both factors < 2^32: exact in uint64
        prod1 = _PHILOX_M1 * c2
        hi0, lo0 = prod0 >> np.uint64(32), prod0 & _MASK32
        hi1, lo1 = prod1 >> np.uint64(32), prod1 & _MASK32
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return np.stack(np.broadcast_arrays(c0, c1, c2, c3), axis=-1).astype(np.uint32)


def philox_normals(n: int, seed: int, stream: int, offset: int, start: int = 0) -> np.ndarray:
    """Standard normals z[start : start + n] of one Philox stream, in fp64.

    Element e uses Philox block e // 4 (counter (e // 4, stream, offset_lo,
    offset_hi), key (seed_lo, seed_hi)) and lane e % 4, through the Box-Muller
    transform on the block's four words.
    """
    e = np.arange(start, start + n, dtype=np.uint64)
    blocks = np.unique(e >> np.uint64(2))
    words = philox4x32_10(
        (blocks, np.full_like(blocks, stream), np.full_like(blocks, offset & 0xFFFFFFFF),
         np.full_like(blocks, (offset >> 32) & 0xFFFFFFFF)),
        (seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF)).astype(np.float64)
    top24 = np.floor(words / 256.0)                    # x >> 8, exact in fp64
    u0 = (top24[:, 0] + 1.0) * 2.0 ** -24              # (0, 1]
    v1 = top24[:, 1] * 2.0 ** -24                      # [0, 1)
    u2 = (top24[:, 2] + 1.0) * 2.0 ** -24
    v3 = top24[:, 3] * 2.0 ** -24
    r0 = np.sqrt(-2.0 * np.log(u0))
    r2 = np.sqrt(-2.0 * np.log(u2))
    z = np.stack([r0 * np.cos(2 * np.pi * v1), r0 * np.sin(2 * np.pi * v1),
                  r2 * np.cos(2 * np.pi * v3), r2 * np.sin(2 * np.pi * v3)], axis=1)
    idx = (e - (blocks[0] << np.uint64(2))).astype(np.int64)
    return z.reshape(-1)[idx]


def philox_rademacher(n: int, seed: int, stream: int, offset: int, start: int = 0) -> np.ndarray:
    """Rademacher values r[start : start + n] of one Philox stream (fp64):
    +1 or -1 from the top bit of word e % 4 of Philox block e // 4."""
    e = np.arange(start, start + n, dtype=np.uint64)
    blocks = np.unique(e >> np.uint64(2))
    words = philox4x32_10(
        (blocks, np.full_like(blocks, stream), np.full_like(blocks, offset & 0xFFFFFFFF),
         np.full_like(blocks, (offset >> 32) & 0xFFFFFFFF)),
        (seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF))
    top = (words >> np.uint32(31)).astype(np.float64)       # 0 or 1
    vals = 1.0 - 2.0 * top
    idx = (e - (blocks[0] << np.uint64(2))).astype(np.int64)
    return vals.reshape(-1)[idx]


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round fp64 values to the nearest bfloat16 value (8 significant bits,
    ties to even), returned as fp64.  Values here are finite and normal."""
    x = np.asarray(x, dtype=np.float64)
    mant, expo = np.frexp(x)                 # x = mant * 2**expo, |mant| in [0.5, 1)
    return np.ldexp(np.rint(mant * 256.0), expo - 8)


def probe_rows(rows: int, cols: int, seed: int, stream: int, offset: int, dtype: str,
               kind: str = "gaussian") -> np.ndarray:
    """rows x cols matrix of stream `stream`, element (j, c) at index j*cols + c.
    Gaussian probes of bf16 workloads are rounded to bfloat16; Rademacher
    values are exact in every format."""
    if kind == "rademacher":
        return philox_rademacher(rows * cols, seed, stream, offset).reshape(rows, cols)
    if kind != "gaussian":
        raise ValueError(f"unknown probe kind {kind!r}")
    z = philox_normals(rows * cols, seed, stream, offset).reshape(rows, cols)
    return round_bf16(z) if dtype == "bf16" else z


# --------------------------------------------------------------------------
# Exact per-sample squared norms (RC, Core mechanism: trace identity; RC,
# Problem definition: FGC materialises per-sample gradients, GC uses Grams).
# --------------------------------------------------------------------------

def per_sample_grads(A: np.ndarray, G: np.ndarray):
    """Yield M_i = A_i^T G_i (d x p, fp64) for every sample i (RC, Core
    mechanism: the per-sample gradient of a linear layer)."""
    for i in range(A.shape[0]):
        yield A[i].astype(np.float64).T @ G[i].astype(np.float64)


def sqnorms_direct(A, G) -> np.ndarray:
    """||A_i^T G_i||_F^2 by materialising each per-sample gradient."""
    return np.array([np.sum(M * M) for M in per_sample_grads(A, G)])


def sqnorms_trace(A, G) -> np.ndarray:
    """trace(O_i) with O_i = G_i^T A_i A_i^T G_i formed explicitly (p x p)."""
    out = []
    for i in range(A.shape[0]):
        a, g = A[i].astype(np.float64), G[i].astype(np.float64)
        O = g.T @ (a @ a.T) @ g
        out.append(np.trace(O))
    return np.array(out)


def sqnorms_ghost(A, G) -> np.ndarray:
    """Ghost form sum((A_i A_i^T) o (G_i G_i^T)), Hadamard product of the two
    T x T Gram matrices (equal to trace(O_i) by cyclicity of the trace)."""
    out = []
    for i in range(A.shape[0]):
        a, g = A[i].astype(np.float64), G[i].astype(np.float64)
        out.append(np.sum((a @ a.T) * (g @ g.T)))
    return np.array(out)


def sqnorms_outer_bruteforce(A, G) -> np.ndarray:
    """Tiny inputs only: build M_i entry by entry as sum_t a_t[r] g_t[c] with
    Python loops, then square-sum.  Independent of any matmul routine."""
    B, T, d = A.shape
    p = G.shape[2]
    out = []
    for i in range(B):
        total = 0.0
        for r in range(d):
            for c in range(p):
                m = 0.0
                for t in range(T):
                    m += float(A[i, t, r]) * float(G[i, t, c])
                total += m * m
        out.append(total)
    return np.array(out)


# --------------------------------------------------------------------------
# Hutch (RC, Core mechanism, item 1)
# --------------------------------------------------------------------------

def hutch_probe(p: int, k: int, seed: int, offset: int, dtype: str,
                kind: str = "gaussian") -> np.ndarray:
    """The p x k probe matrix P (stored by the GPU path as k rows of length p,
    element (j, c) at j*p + c of stream 0); Gaussian or Rademacher."""
    return probe_rows(k, p, seed, STREAM_P, offset, dtype, kind).T


def sqnorms_hutch(A, G, P: np.ndarray, Ms=None) -> np.ndarray:
    """Hutchinson estimate of trace(O_i) with the probe columns P_j:
    q_i = (1/k) sum_j P_j^T O_i P_j, where P_j^T O_i P_j = ||M_i P_j||^2
    since O_i = M_i^T M_i."""
    k = P.shape[1]
    Ms = per_sample_grads(A, G) if Ms is None else Ms
    out = []
    for M in Ms:
        total = 0.0
        for j in range(k):
            v = M @ P[:, j]
            total += float(v @ v)
        out.append(total / k)
    return np.array(out)


# --------------------------------------------------------------------------
# Hutch++ (RC, Core mechanism, item 2: QR low-rank head + Hutchinson tail)
# --------------------------------------------------------------------------

def hutchpp_split(k: int):
    """Budget of k products with O: r = floor(k/3) sketch columns, r head
    columns, m = k - 2r tail probes."""
    r = k // 3
    m = k - 2 * r
    if r < 1 or m < 1:
        raise ValueError("Hutch++ needs k >= 3")
    return r, m


def hutchpp_probes(p: int, k: int, seed: int, offset: int, dtype: str, kind: str = "gaussian"):
    """S (p x r, stream 1) and G' (p x m, stream 2), stored row-per-column like P."""
    r, m = hutchpp_split(k)
    S = probe_rows(r, p, seed, STREAM_S, offset, dtype, kind).T
    Gp = probe_rows(m, p, seed, STREAM_GP, offset, dtype, kind).T
    return S, Gp


def sqnorms_hutchpp(A, G, S: np.ndarray, Gp: np.ndarray, Ms=None, qr=None) -> np.ndarray:
    """Hutch++ estimate of trace(O_i), per sample:
      Y = O_i S, Q = orthonormal basis of range(Y) (Householder QR),
      head = trace(Q^T O_i Q),
      W = (I - Q Q^T) G', tail = trace(W^T O_i W) / m,
      q_i = head + tail.
    Products with O_i are taken as M_i^T (M_i X)."""
    qr = (lambda Y: np.linalg.qr(Y, mode="reduced")[0]) if qr is None else qr
    m = Gp.shape[1]
    Ms = per_sample_grads(A, G) if Ms is None else Ms
    out = []
    for M in Ms:
        Y = M.T @ (M @ S)
        Q = qr(Y)
        MQ = M @ Q
        head = float(np.sum(MQ * MQ))
        W = Gp - Q @ (Q.T @ Gp)
        MW = M @ W
        tail = float(np.sum(MW * MW)) / m
        out.append(head + tail)
    return np.array(out)


# --------------------------------------------------------------------------
# Clipping and noise (GL, DP-SGD algorithm steps 3-4; RC, Algorithmic flow
# steps 4-5)
# --------------------------------------------------------------------------

def clip_scales(q: np.ndarray, C: float):
    """s_i = min(C / n_i, 1) with n_i = sqrt(q_i) (RC step 4), which equals
    the 1 / max(1, n_i / C) of GL step 3.  n_i = 0 gives s_i = 1.  The flag
    marks samples whose estimated norm exceeds C (those actually scaled)."""
    q = np.asarray(q, dtype=np.float64)
    n = np.sqrt(np.maximum(q, 0.0))
    with np.errstate(divide="ignore"):
        s = np.where(n > 0, np.minimum(1.0, C / np.where(n > 0, n, 1.0)), 1.0)
    return s, n > C


def noise_matrix(d: int, p: int, seed: int, offset: int) -> np.ndarray:
    """d x p standard normals from stream 3, entry (r, c) at index r*p + c."""
    return philox_normals(d * p, seed, STREAM_NOISE, offset).reshape(d, p)


def clipped_noisy_grad(A, G, q, C: float, sigma: float, seed: int, offset: int, Ms=None):
    """sum_i s_i M_i + N(0, sigma^2 C^2 I) (GL step 4 on the clipped per-sample
    gradients; RC steps 4-5: the second backward of the loss rescaled by s_i
    gives, for one linear layer, sum_i s_i A_i^T G_i).  Returns (D, s, flags),
    D being d x p."""
    s, flags = clip_scales(q, C)
    Ms = per_sample_grads(A, G) if Ms is None else Ms
    D = None
    for si, M in zip(s, Ms):
        D = si * M if D is None else D + si * M
    if D is None:
        # an empty lot (Poisson sampling can draw none, GL step 1): the sum of
        # no clipped gradients is zero and only the noise remains
        D = np.zeros((A.shape[2], G.shape[2]))
    if sigma != 0.0:
        D = D + (sigma * C) * noise_matrix(D.shape[0], D.shape[1], seed, offset)
    return D, s, flags


# ----------------------------------------------------------------------------
# Bias of the linear layer (RC, Algorithmic flow steps 3-5 for the whole
# per-sample gradient; GL step 3 clips the gradient of every parameter).
# For y_t = x_t W + b the derivative of the output w.r.t. b is the identity at
# every token, so the per-sample bias gradient sums the output gradients over
# the sample's tokens.  It is the weight gradient of an extra input feature
# that is 1 at every token.

def per_sample_bias_grads(G: np.ndarray) -> np.ndarray:
    """b_i = sum_t G_i[t, :] for every sample (B x p, fp64)."""
    return G.astype(np.float64).sum(axis=1)


def bias_sqnorms(G: np.ndarray) -> np.ndarray:
    """||b_i||^2 per sample: the bias's share of the per-sample squared norm."""
    b = per_sample_bias_grads(G)
    return np.sum(b * b, axis=1)


def clipped_noisy_bias_grad(G, q, C: float, sigma: float, seed: int, offset: int, bs=None):
    """sum_i s_i b_i + N(0, sigma^2 C^2 I_p), the same s_i as the weights (q is
    the per-sample squared norm of the whole gradient), noise from stream 4
    with column c at element index c.  Returns (Db, s, flags), Db of length p."""
    s, flags = clip_scales(q, C)
    bs = per_sample_bias_grads(G) if bs is None else bs
    Db = np.zeros(bs.shape[1])
    for si, b in zip(s, bs):
        Db = Db + si * b
    if sigma != 0.0:
        Db = Db + (sigma * C) * philox_normals(bs.shape[1], seed, STREAM_BIAS_NOISE, offset)
    return Db, s, flags


# ----------------------------------------------------------------------------
# Parameter update (GL step 5): theta <- theta - eta * g~ / L, g~ the noisy sum
# of clipped per-sample gradients and L the lot size of the average.  With
# Poisson sampling (each example joins the lot with probability L / N) the
# drawn lot size varies from step to step and L is its expectation, so the
# noise scale relative to the update does not depend on the draw.

def sgd_update(theta: np.ndarray, g_noisy: np.ndarray, lr: float, denom: float) -> np.ndarray:
    """theta - lr * g_noisy / denom, in fp64."""
    return np.asarray(theta, np.float64) - (lr / denom) * np.asarray(g_noisy, np.float64)


# ----------------------------------------------------------------------------
# FIBER (FB, Method A and C): the privatized gradient g_t is filtered in
# innovation space and fed to AdamW, whose second moment is calibrated by the
# filtered noise variance.
#   innovation   nu_t = g_t - gf_{t-1}
#   residual     r_t  = (1 - omega) r_{t-1} + omega nu_t
#   integration  gf_t = gf_{t-1} + r_t
# A stable linear filter; for white noise of variance s2 at its input the
# output variance in steady state is A(omega) s2, A = (2 - omega)/(4 - 3 omega).
# AdamW on gf_t (decoupled weight decay), with the bias-corrected second
# moment reduced by the attenuated noise variance:
#   vbar_t = max(vhat_t - A(omega) s2, eps_v).
# Readings (FB is silent): the filter and moment states start at zero; the
# update is theta -= lr (mhat / (sqrt(vbar) + eps) + wd theta), the AdamW form;
# g_t is the privatized gradient the optimizer sees (the noisy clipped sum
# divided by the lot size), its noise variance per coordinate s2 = (sigma C / L)^2.

def fiber_attenuation(omega: float) -> float:
    """A(omega) = (2 - omega) / (4 - 3 omega), in [0.5, 1] for 0 < omega <= 1."""
    return (2.0 - omega) / (4.0 - 3.0 * omega)


def fiber_filter_step(g, gf, r, omega: float):
    """One step of the innovation filter: returns (gf_t, r_t)."""
    nu = np.asarray(g, np.float64) - gf
    r = (1.0 - omega) * r + omega * nu
    return gf + r, r


def fiber_adamw_step(theta, g, state, t: int, lr: float, beta1: float, beta2: float, eps: float,
                     eps_v: float, wd: float, omega: float, noise_var: float):
    """One FIBER step at step number t >= 1.  state = (gf, r, m, v), every
    array shaped like theta; returns (theta_t, state_t), all fp64."""
    gf, r, m, v = state
    gf, r = fiber_filter_step(g, gf, r, omega)
    m = beta1 * m + (1.0 - beta1) * gf
    v = beta2 * v + (1.0 - beta2) * gf * gf
    mhat = m / (1.0 - beta1 ** t)
    vhat = v / (1.0 - beta2 ** t)
    vbar = np.maximum(vhat - fiber_attenuation(omega) * noise_var, eps_v)
    theta = np.asarray(theta, np.float64)
    theta = theta - lr * (mhat / (np.sqrt(vbar) + eps) + wd * theta)
    return theta, (gf, r, m, v)
