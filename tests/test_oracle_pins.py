"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Nothing here compares the oracle with itself: each check is a published
known-answer vector, a closed form, an invariant, a special case that reduces
to a library routine, or brute force on tiny inputs.
"""
import math
import os

import numpy as np
import pytest
import scipy.stats
import torch

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def _tiny(B=3, T=7, d=5, p=6, seed=0, gscale=1.0):
    r = _rng(seed)
    return r.standard_normal((B, T, d)), gscale * r.standard_normal((B, T, p))


# --------------------------------------------------------------- Philox / RNG

def test_philox_known_answers():
    rows = []
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                rows.append([int(w, 16) for w in line.split()])
    assert len(rows) == 3
    for r in rows:
        out = O.philox4x32_10(r[0:4], r[4:6])
        assert [int(w) for w in out] == r[6:10]


def test_philox_vectorised_matches_scalar():
    ctr = (np.arange(5, dtype=np.uint64), 7, 11, 13)
    many = O.philox4x32_10(ctr, (3, 9))
    for i in range(5):
        assert np.array_equal(many[i], O.philox4x32_10((i, 7, 11, 13), (3, 9)))


def test_normals_law():
    z = O.philox_normals(1 << 20, seed=12345, stream=3, offset=0)
    n = z.size
    assert abs(z.mean()) < 5 / math.sqrt(n)
    assert abs(z.var() - 1.0) < 5 * math.sqrt(2.0 / n)
    assert scipy.stats.kstest(z, "norm").pvalue > 1e-4
    # the two normals drawn from one (u, v) pair are uncorrelated
    pairs = z.reshape(-1, 2)
    assert abs(np.corrcoef(pairs[:, 0], pairs[:, 1])[0, 1]) < 5 / math.sqrt(n / 2)
    # fourth moment of N(0,1) is 3
    assert abs(np.mean(z ** 4) - 3.0) < 0.05


def test_normals_slicing_streams_offsets():
    full = O.philox_normals(103, seed=5, stream=0, offset=9)
    part = O.philox_normals(50, seed=5, stream=0, offset=9, start=37)
    assert np.array_equal(full[37:87], part)
    other_stream = O.philox_normals(103, seed=5, stream=1, offset=9)
    other_offset = O.philox_normals(103, seed=5, stream=0, offset=10)
    other_seed = O.philox_normals(103, seed=6, stream=0, offset=9)
    for x in (other_stream, other_offset, other_seed):
        assert not np.any(x == full)
    # the high word of the 64-bit offset and seed matter
    assert not np.any(O.philox_normals(16, 5, 0, 1 << 32) == O.philox_normals(16, 5, 0, 0))
    assert not np.any(O.philox_normals(16, 5 + (1 << 32), 0, 0) == O.philox_normals(16, 5, 0, 0))


def test_round_bf16_against_torch_and_ties():
    x = _rng(1).standard_normal(200000).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(O.round_bf16(x.astype(np.float64)), ref)
    # ties go to even significands
    assert O.round_bf16(np.array([1 + 2 ** -8]))[0] == 1.0
    assert O.round_bf16(np.array([1 + 3 * 2 ** -8]))[0] == 1 + 2 ** -6
    assert O.round_bf16(np.array([-(1 + 3 * 2 ** -8)]))[0] == -(1 + 2 ** -6)


# --------------------------------------------------------------- exact norms

def test_trace_identity_three_ways():
    A, G = _tiny(B=4, T=9, d=6, p=11, seed=2)
    q_direct = O.sqnorms_direct(A, G)
    np.testing.assert_allclose(O.sqnorms_trace(A, G), q_direct, rtol=1e-12)
    np.testing.assert_allclose(O.sqnorms_ghost(A, G), q_direct, rtol=1e-12)


def test_direct_against_bruteforce_outer_products():
    A, G = _tiny(B=2, T=5, d=3, p=4, seed=3)
    np.testing.assert_allclose(O.sqnorms_direct(A, G), O.sqnorms_outer_bruteforce(A, G), rtol=1e-13)


def test_ghost_against_torch_per_sample_grads():
    A, G = _tiny(B=3, T=20, d=8, p=5, seed=4)
    At, Gt = torch.from_numpy(A), torch.from_numpy(G)
    Mt = torch.einsum("btd,btp->bdp", At, Gt)
    np.testing.assert_allclose(O.sqnorms_ghost(A, G), (Mt ** 2).sum((1, 2)).numpy(), rtol=1e-12)


def test_exact_norm_is_gradient_of_linear_layer():
    # Per-sample gradient of sum(Y * G_i) with Y = A_i W (W: d x p) is A_i^T G_i
    # (a single linear layer with output gradient G_i), via autograd.
    A, G = _tiny(B=2, T=6, d=4, p=3, seed=5)
    q = []
    for i in range(2):
        W = torch.zeros(4, 3, dtype=torch.float64, requires_grad=True)
        (torch.from_numpy(A[i]) @ W * torch.from_numpy(G[i])).sum().backward()
        q.append(float((W.grad ** 2).sum()))
    np.testing.assert_allclose(O.sqnorms_direct(A, G), q, rtol=1e-13)


# --------------------------------------------------------------- Hutch

def test_hutch_scaled_identity_probe_is_exact():
    A, G = _tiny(B=3, T=8, d=5, p=7, seed=6)
    P = math.sqrt(7) * np.eye(7)
    np.testing.assert_allclose(O.sqnorms_hutch(A, G, P), O.sqnorms_direct(A, G), rtol=1e-12)


def test_hutch_associativity():
    A, G = _tiny(B=2, T=10, d=6, p=9, seed=7)
    P = _rng(8).standard_normal((9, 4))
    ref = [np.sum((A[i].T @ (G[i] @ P)) ** 2) / 4 for i in range(2)]
    np.testing.assert_allclose(O.sqnorms_hutch(A, G, P), ref, rtol=1e-12)


def test_hutch_unbiased_with_closed_form_variance():
    A, G = _tiny(B=1, T=12, d=6, p=10, seed=9)
    M = A[0].T @ G[0]
    Omat = M.T @ M
    exact = np.trace(Omat)
    k, N = 4, 4000
    est = np.array([O.sqnorms_hutch(A, G, O.hutch_probe(10, k, 77, off, "f32"), Ms=[M])[0]
                    for off in range(N)])
    se = est.std(ddof=1) / math.sqrt(N)
    assert abs(est.mean() - exact) < 4 * se
    var_true = 2.0 * np.sum(Omat * Omat) / k      # Gaussian probes, symmetric O
    assert abs(est.var(ddof=1) / var_true - 1.0) < 0.15


def test_hutch_probe_layout():
    P = O.hutch_probe(6, 3, seed=1, offset=2, dtype="f32")
    z = O.philox_normals(18, seed=1, stream=O.STREAM_P, offset=2)
    assert P.shape == (6, 3)
    assert P[4, 2] == z[2 * 6 + 4]
    Pb = O.hutch_probe(6, 3, seed=1, offset=2, dtype="bf16")
    assert np.array_equal(Pb, O.round_bf16(P))


# --------------------------------------------------------------- Hutch++

def test_hutchpp_split():
    assert O.hutchpp_split(32) == (10, 12)
    assert O.hutchpp_split(8) == (2, 4)
    assert O.hutchpp_split(3) == (1, 1)
    with pytest.raises(ValueError):
        O.hutchpp_split(2)


def test_hutchpp_exact_when_rank_below_head():
    # rank(O_i) <= T <= r: the head captures all of O_i and the tail vanishes.
    A, G = _tiny(B=3, T=4, d=9, p=12, seed=10)
    S, Gp = O.hutchpp_probes(12, 15, seed=3, offset=0, dtype="f32")   # r = 5 >= T
    np.testing.assert_allclose(O.sqnorms_hutchpp(A, G, S, Gp), O.sqnorms_direct(A, G), rtol=1e-10)


def test_hutchpp_invariant_to_qr_method():
    A, G = _tiny(B=2, T=30, d=8, p=14, seed=11)
    S, Gp = O.hutchpp_probes(14, 9, seed=4, offset=1, dtype="f32")

    def gram_schmidt(Y):
        Q = np.zeros_like(Y)
        for j in range(Y.shape[1]):
            v = Y[:, j].copy()
            for _ in range(2):
                v -= Q[:, :j] @ (Q[:, :j].T @ v)
            Q[:, j] = v / np.linalg.norm(v)
        return Q

    def svd_basis(Y):
        return np.linalg.svd(Y, full_matrices=False)[0]

    ref = O.sqnorms_hutchpp(A, G, S, Gp)
    np.testing.assert_allclose(O.sqnorms_hutchpp(A, G, S, Gp, qr=gram_schmidt), ref, rtol=1e-10)
    np.testing.assert_allclose(O.sqnorms_hutchpp(A, G, S, Gp, qr=svd_basis), ref, rtol=1e-10)


def test_hutchpp_unbiased_and_beats_hutch_on_decaying_spectrum():
    r = _rng(12)
    T, d, p = 40, 10, 16
    # a per-sample gradient with a fast-decaying spectrum
    U, _ = np.linalg.qr(r.standard_normal((d, d)))
    V, _ = np.linalg.qr(r.standard_normal((p, p)))
    sv = 2.0 ** -np.arange(d)
    M = (U * sv) @ V[:, :d].T
    exact = np.sum(M * M)
    k, N = 9, 1500
    hpp, hut = [], []
    for off in range(N):
        S, Gp = O.hutchpp_probes(p, k, 21, off, "f32")
        hpp.append(O.sqnorms_hutchpp(None, None, S, Gp, Ms=[M])[0])
        hut.append(O.sqnorms_hutch(None, None, O.hutch_probe(p, k, 21, off, "f32"), Ms=[M])[0])
    hpp, hut = np.array(hpp), np.array(hut)
    assert abs(hpp.mean() - exact) < 4 * hpp.std(ddof=1) / math.sqrt(N)
    assert hpp.var() < 0.1 * hut.var()


# --------------------------------------------------------------- clipping

def test_clip_scale_invariants():
    q = np.array([0.0, 0.25, 1.0, 4.0, 1e6])
    s, flags = O.clip_scales(q, 1.0)
    assert list(s[:3]) == [1.0, 1.0, 1.0]
    assert s[3] == 0.5
    assert list(flags) == [False, False, False, True, True]
    n = np.sqrt(q)
    assert np.all((s > 0) & (s <= 1))
    assert np.all(s * n <= 1.0 * (1 + 1e-15))
    # GL step 3 form: 1 / max(1, n / C)
    C = 0.7
    s2, _ = O.clip_scales(q, C)
    np.testing.assert_allclose(s2, 1.0 / np.maximum(1.0, n / C), rtol=1e-15)


def test_grad_without_clipping_or_noise_is_plain_gemm():
    A, G = _tiny(B=3, T=11, d=5, p=4, seed=13)
    q = O.sqnorms_direct(A, G)
    D, s, flags = O.clipped_noisy_grad(A, G, q, C=1e30, sigma=0.0, seed=1, offset=0)
    ref = torch.matmul(torch.from_numpy(A.reshape(-1, 5)).T, torch.from_numpy(G.reshape(-1, 4))).numpy()
    np.testing.assert_allclose(D, ref, rtol=1e-12, atol=1e-12)
    assert np.all(s == 1.0) and not flags.any()


def test_grad_clipped_per_sample_norms_are_C():
    A, G = _tiny(B=3, T=11, d=5, p=4, seed=14, gscale=10.0)
    q = O.sqnorms_direct(A, G)
    C = 0.5
    _, s, flags = O.clipped_noisy_grad(A, G, q, C=C, sigma=0.0, seed=1, offset=0)
    assert flags.all()
    np.testing.assert_allclose(s * np.sqrt(q), C, rtol=1e-14)


def test_noise_law_and_determinism():
    A, G = _tiny(B=2, T=16, d=64, p=96, seed=15)
    q = O.sqnorms_direct(A, G)
    C, sigma = 0.5, 0.8
    D0, _, _ = O.clipped_noisy_grad(A, G, q, C, 0.0, seed=3, offset=4)
    D0b, _, _ = O.clipped_noisy_grad(A, G, q, C, 0.0, seed=99, offset=7)
    assert np.array_equal(D0, D0b)                 # sigma = 0 is deterministic
    D1, _, _ = O.clipped_noisy_grad(A, G, q, C, sigma, seed=3, offset=4)
    z = ((D1 - D0) / (sigma * C)).ravel()
    n = z.size
    assert abs(z.mean()) < 5 / math.sqrt(n)
    assert abs(z.var() - 1.0) < 5 * math.sqrt(2.0 / n)
    assert scipy.stats.kstest(z, "norm").pvalue > 1e-4
    D2, _, _ = O.clipped_noisy_grad(A, G, q, C, sigma, seed=3, offset=4)
    assert np.array_equal(D1, D2)                  # same (seed, offset): same noise


# --------------------------------------------------------------- Rademacher probes

def test_rademacher_values_and_balance():
    r = O.philox_rademacher(1 << 20, seed=77, stream=0, offset=3)
    assert set(np.unique(r)) == {-1.0, 1.0}
    n = r.size
    assert abs(r.mean()) < 5 / math.sqrt(n)
    pairs = r.reshape(-1, 2)
    assert abs(np.mean(pairs[:, 0] * pairs[:, 1])) < 5 / math.sqrt(n / 2)
    # same counters as the normals: the sign bit of the word behind each element
    part = O.philox_rademacher(50, seed=77, stream=0, offset=3, start=1001)
    assert np.array_equal(part, r[1001:1051])
    w = O.philox4x32_10((250, 0, 3, 0), (77, 0))          # block 250 = elements 1000..1003
    assert [1.0 - 2.0 * (int(x) >> 31) for x in w] == list(r[1000:1004])


def test_rademacher_hutch_exact_for_diagonal_O():
    # G_i = I (T = p) and A_i with orthogonal rows: O_i = A_i A_i^T is diagonal,
    # so every Rademacher probe z gives z^T O z = trace(O) exactly.
    p, d = 6, 9
    A = np.zeros((2, p, d))
    A[0, :, :p] = np.diag([1.0, 2.0, 0.5, 3.0, 1.5, 0.25])
    A[1, :, 2:2 + p] = np.diag([2.0, 1.0, 1.0, 0.5, 4.0, 1.0])
    G = np.stack([np.eye(p), np.eye(p)])
    exact = O.sqnorms_direct(A, G)
    for off in range(20):
        P = O.hutch_probe(p, 3, seed=5, offset=off, dtype="f32", kind="rademacher")
        np.testing.assert_allclose(O.sqnorms_hutch(A, G, P), exact, rtol=1e-13)
    # Gaussian probes are not exact there
    P = O.hutch_probe(p, 3, seed=5, offset=0, dtype="f32")
    assert not np.allclose(O.sqnorms_hutch(A, G, P), exact, rtol=1e-3)


def test_rademacher_hutch_unbiased_with_closed_form_variance():
    A, G = _tiny(B=1, T=12, d=6, p=10, seed=9)
    M = A[0].T @ G[0]
    Om = M.T @ M
    exact = np.trace(Om)
    k, N = 4, 4000
    est = np.array([O.sqnorms_hutch(None, None, O.hutch_probe(10, k, 78, off, "f32", "rademacher"),
                                    Ms=[M])[0] for off in range(N)])
    assert abs(est.mean() - exact) < 4 * est.std(ddof=1) / math.sqrt(N)
    var_true = 2.0 * (np.sum(Om * Om) - np.sum(np.diag(Om) ** 2)) / k
    assert abs(est.var(ddof=1) / var_true - 1.0) < 0.15


def test_rademacher_hutchpp_exact_at_low_rank_and_unbiased():
    A, G = _tiny(B=2, T=4, d=9, p=12, seed=10)
    S, Gp = O.hutchpp_probes(12, 15, seed=3, offset=0, dtype="f32", kind="rademacher")
    np.testing.assert_allclose(O.sqnorms_hutchpp(A, G, S, Gp), O.sqnorms_direct(A, G), rtol=1e-10)
    A, G = _tiny(B=1, T=30, d=7, p=11, seed=12)
    M = A[0].T @ G[0]
    est = np.array([O.sqnorms_hutchpp(None, None, *O.hutchpp_probes(11, 6, 31, off, "f32", "rademacher"),
                                      Ms=[M])[0] for off in range(1500)])
    assert abs(est.mean() - np.sum(M * M)) < 4 * est.std(ddof=1) / math.sqrt(1500)


# --------------------------------------------------------------- bias of the linear layer

def test_bias_grad_is_the_weight_grad_of_a_constant_input():
    # y = x W + b is y = [x, 1] [W; b]: the bias gradient is the last row of
    # the augmented layer's weight gradient A_aug^T G
    A, G = _tiny(B=3, T=9, d=4, p=7, seed=41)
    ones = np.ones(A.shape[:2] + (1,))
    A_aug = np.concatenate([A, ones], axis=2)
    b = O.per_sample_bias_grads(G)
    for i, M in enumerate(O.per_sample_grads(A_aug, G)):
        np.testing.assert_allclose(b[i], M[-1], rtol=1e-13, atol=1e-13)
    # and its squared norm is what the augmented layer adds to ||M_i||^2
    q_aug = O.sqnorms_direct(A_aug, G)
    np.testing.assert_allclose(q_aug, O.sqnorms_direct(A, G) + O.bias_sqnorms(G), rtol=1e-12)


def test_bias_grad_single_token_and_linearity():
    _, G = _tiny(B=2, T=1, d=1, p=5, seed=42)
    np.testing.assert_array_equal(O.per_sample_bias_grads(G), G[:, 0, :])
    _, G = _tiny(B=2, T=6, d=1, p=5, seed=43)
    np.testing.assert_allclose(O.per_sample_bias_grads(-2.5 * G), -2.5 * O.per_sample_bias_grads(G),
                               rtol=1e-14)


def test_clipped_bias_grad_special_cases():
    _, G = _tiny(B=4, T=5, d=1, p=8, seed=44)
    q = O.bias_sqnorms(G)
    # no clipping, no noise: the plain sum over samples and tokens
    Db, s, flags = O.clipped_noisy_bias_grad(G, q, 1e12, 0.0, 1, 0)
    np.testing.assert_allclose(Db, G.sum(axis=(0, 1)), rtol=1e-13)
    assert np.all(s == 1.0) and not flags.any()
    # clipping every sample to C: each clipped bias gradient has norm C
    C = 0.5 * float(np.sqrt(q.min()))
    _, s, flags = O.clipped_noisy_bias_grad(G, q, C, 0.0, 1, 0)
    b = O.per_sample_bias_grads(G)
    np.testing.assert_allclose(np.linalg.norm(s[:, None] * b, axis=1), C, rtol=1e-12)
    assert flags.all()


def test_bias_noise_is_its_own_stream():
    _, G = _tiny(B=1, T=1, d=1, p=4096, seed=45)
    z = O.clipped_noisy_bias_grad(0 * G, np.zeros(1), 1.0, 1.0, 77, 3)[0]
    np.testing.assert_array_equal(z, O.philox_normals(4096, 77, O.STREAM_BIAS_NOISE, 3))
    w = O.philox_normals(4096, 77, O.STREAM_NOISE, 3)
    assert not np.allclose(z, w)
    assert abs(z.mean()) < 4 / 64 and abs(z.var() - 1) < 4 * math.sqrt(2 / 4096)


# --------------------------------------------------------------- parameter update and Poisson lots

def test_update_without_clipping_or_noise_is_sgd_on_the_lot():
    # C -> inf, sigma = 0: theta - lr / L * (sum of per-sample gradients), and
    # the sum of the per-sample gradients of a linear layer is one GEMM over
    # the lot's tokens
    A, G = _tiny(B=4, T=6, d=5, p=3, seed=51)
    theta = _rng(52).standard_normal((5, 3))
    q = O.sqnorms_direct(A, G)
    D, _, _ = O.clipped_noisy_grad(A, G, q, 1e12, 0.0, 1, 0)
    got = O.sgd_update(theta, D, 0.1, 7.0)
    full = A.reshape(-1, 5).T @ G.reshape(-1, 3)
    np.testing.assert_allclose(got, theta - 0.1 / 7.0 * full, rtol=1e-13, atol=1e-14)
    np.testing.assert_array_equal(O.sgd_update(theta, D, 0.0, 7.0), theta)


def test_empty_poisson_lot_updates_by_noise_only():
    # a lot with no examples: the update is the noise alone, N(0, (lr sigma C / L)^2)
    d, p = 64, 48
    A = np.zeros((0, 5, d))
    G = np.zeros((0, 5, p))
    D, s, flags = O.clipped_noisy_grad(A, G, np.zeros(0), 2.0, 1.5, 9, 4)
    assert D.shape == (d, p) and s.shape == (0,) and flags.shape == (0,)
    theta = np.ones((d, p))
    step = (theta - O.sgd_update(theta, D, 0.3, 10.0)) / (0.3 / 10.0 * 1.5 * 2.0)
    n = d * p
    assert abs(step.mean()) < 4 / math.sqrt(n) and abs(step.var() - 1) < 4 * math.sqrt(2 / n)
    Db, _, _ = O.clipped_noisy_bias_grad(G, np.zeros(0), 2.0, 1.5, 9, 4, bs=np.zeros((0, p)))
    assert Db.shape == (p,) and np.all(Db != 0)


# --------------------------------------------------------------- FIBER filter and calibrated AdamW

@pytest.mark.parametrize("omega", [0.15, 0.5, 0.85, 1.0])
def test_fiber_filter_attenuates_white_noise_by_A(omega):
    # the closed form of the summary against a long simulation of the filter
    # on unit white noise (many independent coordinates, steady state)
    r = _rng(61)
    n, steps = 20000, 400
    gf = np.zeros(n)
    res = np.zeros(n)
    for _ in range(steps):
        gf, res = O.fiber_filter_step(r.standard_normal(n), gf, res, omega)
    var = gf.var()
    A = O.fiber_attenuation(omega)
    assert 0.5 <= A <= 1.0
    # chi-square spread of a sample variance over n coordinates
    assert abs(var - A) < 5 * A * math.sqrt(2.0 / n)


def test_fiber_filter_tracks_a_drifting_gradient():
    # the second-order (constant-velocity) recursion follows a linear drift with
    # no steady-state error, where an EMA of the state lags by a constant
    gf, res = np.zeros(1), np.zeros(1)
    ema = np.zeros(1)
    for t in range(1, 400):
        g = np.array([1.0 + 0.01 * t])
        gf, res = O.fiber_filter_step(g, gf, res, 0.2)
        ema = 0.8 * ema + 0.2 * g
    assert abs(gf[0] - g[0]) < 1e-6
    assert abs(ema[0] - g[0]) > 0.03


def test_fiber_with_unit_gain_and_no_noise_is_adamw():
    # omega = 1 passes the gradient through; noise_var = 0 and eps_v = 0 leave
    # AdamW: compare with torch.optim.AdamW in fp64 over a few steps
    r = _rng(62)
    theta0 = r.standard_normal(50)
    grads = [r.standard_normal(50) for _ in range(6)]
    p = torch.tensor(theta0, dtype=torch.float64, requires_grad=True)
    opt = torch.optim.AdamW([p], lr=0.01, betas=(0.9, 0.99), eps=1e-8, weight_decay=0.05)
    theta = theta0.copy()
    state = tuple(np.zeros(50) for _ in range(4))
    for t, g in enumerate(grads, start=1):
        p.grad = torch.tensor(g, dtype=torch.float64)
        opt.step()
        theta, state = O.fiber_adamw_step(theta, g, state, t, 0.01, 0.9, 0.99, 1e-8, 0.0, 0.05,
                                          1.0, 0.0)
    np.testing.assert_allclose(theta, p.detach().numpy(), rtol=1e-12, atol=1e-13)


def test_fiber_calibration_removes_the_filtered_noise():
    # pure DP noise of variance s2: the filtered second moment settles at
    # A(omega) s2, which the calibration removes (down to the floor eps_v)
    r = _rng(63)
    n, s2, omega = 20000, 0.04, 0.3
    theta = np.zeros(n)
    state = tuple(np.zeros(n) for _ in range(4))
    for t in range(1, 1201):
        g = math.sqrt(s2) * r.standard_normal(n)
        theta, state = O.fiber_adamw_step(theta, g, state, t, 0.0, 0.9, 0.999, 1e-8, 1e-12, 0.0,
                                          omega, s2)
    v = state[3] / (1 - 0.999 ** 1200)
    assert abs(v.mean() - O.fiber_attenuation(omega) * s2) < 0.05 * s2
