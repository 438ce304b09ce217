"""GPU path vs the fp64 oracle, element by element, through the C ABI.

Tolerances: relative 1e-5 for fp32 inputs and 2e-2 for bf16 inputs with fp32
accumulation (per-sample norms and scales; the gradient normwise and per
entry against tol * (|ref| + sigma C)); clip flags bit-exact wherever the
reference norm is more than 4 tol C away from C.
"""
import numpy as np
import pytest
import torch

import oracle as O
from dp_sgd_clipping_gb300 import workloads as W
from gpu_util import (NOISE_TOL, TOL, assert_flags, assert_grad, assert_rel, grad_magnitude, host,
                      to_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api():
    import __graft_entry__
    __graft_entry__.build()
    from dp_sgd_clipping_gb300 import api as _api
    return _api


def oracle_all(inp, k=None, want=("direct", "hutch", "hutchpp")):
    wl = inp.wl
    Ms = list(O.per_sample_grads(inp.A, inp.G))
    out = {"Ms": Ms, "direct": np.array([np.sum(M * M) for M in Ms])}
    k = wl.k if k is None else k
    if "hutch" in want:
        out["hutch"] = O.sqnorms_hutch(None, None, O.hutch_probe(wl.p, k, wl.seed, 0, wl.dtype), Ms=Ms)
    if "hutchpp" in want:
        S, Gp = O.hutchpp_probes(wl.p, k, wl.seed, 0, wl.dtype)
        out["hutchpp"] = O.sqnorms_hutchpp(None, None, S, Gp, Ms=Ms)
    return out


def oracle_grad_parts(inp, q32, C, sigma, Ms, offset):
    """The oracle's clipped sum S = sum_i s_i M_i, its noise sigma C z (None at
    sigma = 0), the scales, and mag = sum_i s_i |A_i|^T |G_i| for the bound."""
    wl = inp.wl
    S, s_ref, _ = O.clipped_noisy_grad(None, None, q32, C, 0.0, wl.seed, offset, Ms=Ms)
    noise = sigma * C * O.noise_matrix(wl.d, wl.p, wl.seed, offset) if sigma != 0.0 else None
    return S, noise, s_ref, grad_magnitude(inp.A, inp.G, s_ref)


def check_grad(api, inp, A, G, q, C, sigma, Ms, offset=0, stored=None):
    """The clipped noisy gradient at sigma and, when sigma > 0, again at
    sigma = 0, each compared with the oracle's clipped sum after taking the
    oracle's noise away (gpu_util.assert_grad).  stored: the StoredGradients
    of norms_direct_store; then the gradient comes from the stored per-sample
    tiles instead of a second GEMM."""
    wl = inp.wl
    tol = TOL[wl.dtype]
    qd = torch.tensor(q, dtype=torch.float32, device="cuda")
    q32 = qd.double().cpu().numpy()          # the sqnorms the GPU saw
    S, noise, s_ref, mag = oracle_grad_parts(inp, q32, C, sigma, Ms, offset)
    K = wl.B * wl.T
    grad = None
    for sg in ((sigma, 0.0) if sigma != 0.0 else (0.0,)):
        if stored is None:
            g, scales, clipped = api.clipped_noisy_grad(A, G, qd, C, sg, wl.seed, offset)
        else:
            g, scales, clipped = api.stored_clipped_noisy_grad(stored, qd, C, sg, wl.seed, offset)
        torch.cuda.synchronize()
        assert_rel(host(scales), s_ref, 1e-6, "scales")
        assert_flags(host(clipped), np.sqrt(q32), C, tol)
        assert_grad(host(g), S, tol, K, mag, noise if sg != 0.0 else None, sg * C,
                    what=f"grad (sigma={sg}, {'stored' if stored is not None else 'gemm'})")
        grad = g if grad is None else grad
    return grad


# ----------------------------------------------------------------------------- RNG

def test_philox_normals_match_oracle(api):
    n = (1 << 20) + 3
    z = api.philox_normal(n, seed=0xD5C11F, stream_id=3, offset=7)
    ref = O.philox_normals(n, 0xD5C11F, 3, 7)
    assert np.max(np.abs(host(z) - ref)) < 2e-5
    zb = api.philox_normal(n, seed=0xD5C11F, stream_id=0, offset=(1 << 33) + 5, dtype=torch.bfloat16)
    refb = O.round_bf16(O.philox_normals(n, 0xD5C11F, 0, (1 << 33) + 5))
    got = host(zb)
    same = got == refb
    assert same.mean() > 0.999
    # the rare differences are one bf16 step at a rounding boundary
    assert np.all(np.abs(got[~same] - refb[~same]) <= 2.0 ** -7 * np.abs(refb[~same]) + 1e-30)


def test_clip_scales_kernel(api):
    q = np.array([0.0, 1e-12, 0.24, 0.25, 0.26, 1.0, 4.0, 1e8], dtype=np.float32)
    s, c = api.clip_scales(torch.tensor(q, device="cuda"), 0.5)
    s_ref, c_ref = O.clip_scales(q.astype(np.float64), 0.5)
    assert_rel(host(s), s_ref, 1e-6, "scales")
    assert_flags(host(c), np.sqrt(q.astype(np.float64)), 0.5, 1e-6)


# ----------------------------------------------------------------------------- fp32 tiny

def test_tiny_f32_workload(api):
    inp = W.make_inputs(W.get(1))
    wl = inp.wl
    A, G = to_dev(inp)
    ref = oracle_all(inp)
    tol = TOL["f32"]
    assert_rel(host(api.norms_exact(A, G, method=2)), ref["direct"], tol, "direct")
    assert_rel(host(api.norms_exact(A, G, method=1)), ref["direct"], tol, "ghost")
    assert_rel(host(api.norms_exact(A, G, method=0)), ref["direct"], tol, "auto")
    q_h = api.norms_hutch(A, G, wl.k, wl.seed, 0)
    assert_rel(host(q_h), ref["hutch"], tol, "hutch")
    assert_rel(host(api.norms_hutchpp(A, G, wl.k, wl.seed, 0)), ref["hutchpp"], tol, "hutch++")
    # the workload as stated (every sample clips at C = 1), then C at the
    # median norm so that about half clip, then sigma = 0
    check_grad(api, inp, A, G, host(q_h), wl.C, wl.sigma, ref["Ms"])
    C_med = float(np.median(np.sqrt(ref["direct"])))
    check_grad(api, inp, A, G, ref["direct"], C_med, wl.sigma, ref["Ms"], offset=3)
    check_grad(api, inp, A, G, ref["direct"], C_med, 0.0, ref["Ms"])


# ----------------------------------------------------------------------------- bf16 ragged

RAGGED = [
    # B, T, d, p, k : several tiles of every kernel plus ragged tails
    (3, 300, 200, 328, 32),
    (2, 300, 200, 328, 12),
    (2, 40, 64, 72, 8),        # T below one token tile
    (1, 1, 8, 16, 4),          # single token, the narrowest rows
    (2, 520, 136, 520, 20),
]


@pytest.mark.parametrize("B,T,d,p,k", RAGGED)
def test_bf16_ragged_all_paths(api, B, T, d, p, k):
    wl = W.Workload(100 + T, f"ragged_{B}_{T}_{d}_{p}", B, T, d, p, "bf16", 1e-2, 0.5, 0.8, k,
                    ("exact", "hutch", "hutchpp", "grad"))
    inp = W.make_inputs(wl)
    A, G = to_dev(inp)
    ref = oracle_all(inp, k=k, want=("hutch", "hutchpp") if k >= 3 else ("hutch",))
    tol = TOL["bf16"]
    assert_rel(host(api.norms_exact(A, G, method=2)), ref["direct"], tol, "direct")
    assert_rel(host(api.norms_exact(A, G, method=1)), ref["direct"], tol, "ghost")
    q_h = api.norms_hutch(A, G, k, wl.seed, 0)
    assert_rel(host(q_h), ref["hutch"], tol, "hutch")
    if k >= 3:
        assert_rel(host(api.norms_hutchpp(A, G, k, wl.seed, 0)), ref["hutchpp"], tol, "hutch++")
    check_grad(api, inp, A, G, host(q_h), wl.C, wl.sigma, ref["Ms"])
    C_med = float(np.median(np.sqrt(ref["direct"])))
    check_grad(api, inp, A, G, ref["direct"], C_med, 0.0, ref["Ms"])


def test_hutchpp_exact_when_rank_deficient(api):
    # T = 6 tokens < r = 10 head columns: rank(O_i) <= 6, Hutch++ is exact.
    wl = W.Workload(120, "rankdef", 2, 6, 64, 96, "bf16", 1e-2, 1.0, 1.0, 32, ("hutchpp",))
    inp = W.make_inputs(wl)
    A, G = to_dev(inp)
    q = host(api.norms_hutchpp(A, G, 32, wl.seed, 0))
    assert_rel(q, O.sqnorms_direct(inp.A, inp.G), 2e-2, "hutch++ rank-deficient")


@pytest.mark.parametrize("case", ["bf16", "f32"])
def test_hutchpp_decaying_spectrum(api, case):
    # A_i^T G_i with 12 singular values decaying by 1/2 over a flat floor, the
    # inputs Hutch++ is meant for: the sketch O_i S spans directions whose
    # squared singular values fall by 1/4 each, so the Gram of the QR's first
    # pass has pivots down to ~1e-11 of the largest, and a head that keeps only
    # the well-conditioned ones leaves the rest to the tail estimate
    wl = W.Workload(185 if case == "bf16" else 186, f"decay_{case}", 2, 300, 200, 328, case, 1e-2,
                    1.0, 1.0, 32, ())
    inp = W.make_decaying_inputs(wl)
    A, G = to_dev(inp)
    Ms = list(O.per_sample_grads(inp.A, inp.G))
    sv = np.linalg.svd(Ms[0], compute_uv=False)
    assert 0.4 < sv[9] / sv[8] < 0.8 and sv[5] / sv[0] < 0.04     # the spectrum decays
    S, Gp = O.hutchpp_probes(wl.p, wl.k, wl.seed, 0, wl.dtype)
    ref = O.sqnorms_hutchpp(None, None, S, Gp, Ms=Ms)
    assert_rel(host(api.norms_hutchpp(A, G, wl.k, wl.seed, 0)), ref, TOL[wl.dtype],
               "hutch++ decaying spectrum")
    P = O.hutch_probe(wl.p, wl.k, wl.seed, 0, wl.dtype)
    assert_rel(host(api.norms_hutch(A, G, wl.k, wl.seed, 0)),
               O.sqnorms_hutch(None, None, P, Ms=Ms), TOL[wl.dtype], "hutch decaying spectrum")


def test_zero_gradients(api):
    wl = W.Workload(121, "zeros", 2, 130, 64, 64, "bf16", 1e-2, 1.0, 1.0, 8, ())
    A = torch.zeros(2, 130, 64, dtype=torch.bfloat16, device="cuda")
    G = torch.zeros_like(A)
    for q in (api.norms_exact(A, G, method=1), api.norms_exact(A, G, method=2),
              api.norms_hutch(A, G, 8, 1, 0), api.norms_hutchpp(A, G, 8, 1, 0)):
        assert np.all(host(q) == 0.0)
    grad, s, c = api.clipped_noisy_grad(A, G, torch.zeros(2, device="cuda"), 1.0, 0.0, 1, 0)
    assert np.all(host(grad) == 0.0) and np.all(host(s) == 1.0) and not host(c).any()


def test_results_are_deterministic(api):
    wl = W.Workload(122, "det", 3, 700, 256, 512, "bf16", 1e-2, 0.5, 1.0, 32, ())
    A, G = to_dev(W.make_inputs(wl))
    for f in (lambda: api.norms_hutch(A, G, 32, 5, 1), lambda: api.norms_hutchpp(A, G, 32, 5, 1),
              lambda: api.norms_exact(A, G, method=1), lambda: api.norms_exact(A, G, method=2)):
        assert torch.equal(f(), f())
    q = api.norms_hutch(A, G, 32, 5, 1)
    g1 = api.clipped_noisy_grad(A, G, q, 0.5, 1.0, 9, 4)[0]
    g2 = api.clipped_noisy_grad(A, G, q, 0.5, 1.0, 9, 4)[0]
    assert torch.equal(g1, g2)


@pytest.mark.parametrize("shape", [(3, 1000, 512, 1536), (4, 4096, 2048, 8192)])
def test_back_to_back_calls_share_a_workspace(api, shape):
    # Each kernel of an estimator call overlaps its prologue with the end of
    # the previous kernel, and the next call's first kernel clears the
    # workspace's tickets while nothing else is in flight.  Calls queued back
    # to back on one workspace, with other seeds and inputs each time, must
    # give what the same calls give alone on a workspace filled with NaN
    # bytes: a read of an intermediate before it is stored, or of a ticket
    # before it is cleared, sees another call's values or the NaN fill.
    B, T, d, p = shape
    wl = W.Workload(123, "b2b", B, T, d, p, "bf16", 1e-2, 1.0, 1.0, 32, ())
    g = torch.Generator(device="cuda").manual_seed(11)
    pairs = [(torch.randn(B, T, d, device="cuda", generator=g).to(torch.bfloat16),
              (torch.randn(B, T, p, device="cuda", generator=g) * 1e-2).to(torch.bfloat16))
             for _ in range(2)]
    from dp_sgd_clipping_gb300 import _lib as L
    for op, fn in ((L.OP_NORMS_HUTCH, api.norms_hutch), (L.OP_NORMS_HUTCHPP, api.norms_hutchpp)):
        nb = api.workspace_bytes(op, B, T, d, p, L.BF16, wl.k)
        calls = [(pairs[c % 2], seed) for c, seed in enumerate(range(1, 7))]
        alone = []
        for (A, G), seed in calls:
            ws = torch.full((nb,), 0xFF, dtype=torch.uint8, device="cuda")
            alone.append(fn(A, G, wl.k, seed, 0, ws=ws))
            torch.cuda.synchronize()
        ws = torch.full((nb,), 0xFF, dtype=torch.uint8, device="cuda")
        torch.cuda.synchronize()
        queued = [fn(A, G, wl.k, seed, 0, ws=ws) for (A, G), seed in calls]
        torch.cuda.synchronize()
        for a, q in zip(alone, queued):
            assert torch.isfinite(a).all()
            assert torch.equal(a, q), (op, host(a), host(q))


# ----------------------------------------------------------------------------- standard workloads

def test_exact_workload_ghost_vs_direct(api):
    inp = W.make_inputs(W.get(2))
    wl = inp.wl
    A, G = to_dev(inp)
    ref = oracle_all(inp, want=())
    tol = TOL["bf16"]
    q_g = host(api.norms_exact(A, G, method=1))
    q_d = host(api.norms_exact(A, G, method=2))
    assert_rel(q_g, ref["direct"], tol, "ghost")
    assert_rel(q_d, ref["direct"], tol, "direct")
    assert_rel(q_g, q_d, 1e-3, "ghost vs direct")
    check_grad(api, inp, A, G, q_d, wl.C, wl.sigma, ref["Ms"])
    C_med = float(np.median(np.sqrt(ref["direct"])))
    check_grad(api, inp, A, G, ref["direct"], C_med, 0.0, ref["Ms"])


@pytest.mark.parametrize("B,T,d,p", [(1, 3328, 2048, 4096), (1, 3300, 2040, 4088),
                                     (5, 1500, 2040, 2040), (1, 4352, 2048, 4096),
                                     (2, 2560, 2048, 4096), (1, 4096, 1024, 2048)])
def test_ghost_last_round_cuts(api, B, T, d, p):
    # More 256-token units than pairs, so the last round is cut: on 76 pairs
    # (one GB300) the first two shapes leave 15 units whose A Gram block is
    # formed once and shared by two p-slices (the second with a partial
    # token tile, a partial last K-block over d and a shorter second slice),
    # the third 29 such units of two samples (one p-slice each), the fourth
    # 1 unit cut into 8 slices that each recompute it, the fifth 34 units cut
    # in two, the sixth 60 whole units.  A unit carries about 1/100 of a
    # sample's norm (1/21 in the third), so the check is at 2e-4, against the
    # oracle and the direct form.
    wl = W.Workload(124, f"ghost_cut_{B}_{T}_{d}_{p}", B, T, d, p, "bf16", 1e-2, 1.0, 1.0, 8, ())
    inp = W.make_inputs(wl)
    A, G = to_dev(inp)
    ref = O.sqnorms_direct(inp.A, inp.G)
    q_g = host(api.norms_exact(A, G, method=1))
    assert_rel(q_g, ref, 2e-4, "ghost")
    assert_rel(q_g, host(api.norms_exact(A, G, method=2)), 2e-4, "ghost vs direct")


@pytest.mark.slow
@pytest.mark.parametrize("wid", [3, 4, 5])
def test_full_size_workloads(api, wid):
    inp = W.make_inputs(W.get(wid))
    wl = inp.wl
    A, G = to_dev(inp)
    want = tuple(r for r in wl.runs if r in ("hutch", "hutchpp"))
    ref = oracle_all(inp, want=want)
    tol = TOL["bf16"]
    q_h = api.norms_hutch(A, G, wl.k, wl.seed, 0)
    assert_rel(host(q_h), ref["hutch"], tol, "hutch")
    if "hutchpp" in wl.runs:
        assert_rel(host(api.norms_hutchpp(A, G, wl.k, wl.seed, 0)), ref["hutchpp"], tol, "hutch++")
    if "direct" in wl.runs:
        assert_rel(host(api.norms_exact(A, G, method=2)), ref["direct"], tol, "direct")
    check_grad(api, inp, A, G, host(q_h), wl.C, wl.sigma, ref["Ms"])
    # the stored variant of the exact norms and of the gradient
    q_s, stored = api.norms_direct_store(A, G)
    assert_rel(host(q_s), ref["direct"], tol, "direct (stored)")
    check_grad(api, inp, A, G, host(q_h), wl.C, wl.sigma, ref["Ms"], stored=stored)


# ----------------------------------------------------------------------------- failure path

def test_bounded_wait_reports_timeout_and_context_survives(api):
    from dp_sgd_clipping_gb300 import _lib as L
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    api.selftest_wait_timeout(ws, 20000)
    assert api.workspace_status(ws) == L.ERR_TIMEOUT
    # the context is still usable afterwards
    z = api.philox_normal(1024, 1, 0, 0)
    torch.cuda.synchronize()
    assert torch.isfinite(z).all()
    ws2 = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    A = torch.ones(1, 8, 8, dtype=torch.bfloat16, device="cuda")
    q = api.norms_hutch(A, A, 4, 1, 0, ws=ws2)
    assert api.workspace_status(ws2) == 0
    assert torch.isfinite(q).all()


# ----------------------------------------------------------------------------- shape boundaries

def _run_all(api, wl, paths=("direct", "ghost", "hutch", "hutchpp", "grad")):
    inp = W.make_inputs(wl)
    A, G = to_dev(inp)
    want = tuple(x for x in ("hutch", "hutchpp") if x in paths and (x != "hutchpp" or wl.k >= 3))
    ref = oracle_all(inp, want=want)
    tol = TOL[wl.dtype]
    if "direct" in paths:
        assert_rel(host(api.norms_exact(A, G, method=2)), ref["direct"], tol, "direct")
    if "ghost" in paths:
        assert_rel(host(api.norms_exact(A, G, method=1)), ref["direct"], tol, "ghost")
    if "hutch" in paths:
        assert_rel(host(api.norms_hutch(A, G, wl.k, wl.seed, 0)), ref["hutch"], tol, "hutch")
    if "hutchpp" in want:
        assert_rel(host(api.norms_hutchpp(A, G, wl.k, wl.seed, 0)), ref["hutchpp"], tol, "hutch++")
    if "grad" in paths:
        C_med = float(np.median(np.sqrt(ref["direct"])))
        check_grad(api, inp, A, G, ref["direct"], C_med, wl.sigma, ref["Ms"], offset=5)


@pytest.mark.parametrize("k", [1, 2, 15, 16, 17, 31, 32])
def test_hutch_probe_widths(api, k):
    # k <= 16 runs the 16-column skinny kernels, k > 16 the 32-column ones
    wl = W.Workload(140 + k, f"kwidth_{k}", 2, 200, 64, 136, "bf16", 1e-2, 1.0, 1.0, k, ())
    _run_all(api, wl, paths=("hutch",))


@pytest.mark.parametrize("B,T,d,p", [(5, 2048, 2048, 1024), (3, 2304, 2304, 1280),
                                     (2, 3072, 3072, 1536), (1, 5120, 5120, 1792)])
def test_skinny_split_counts(api, B, T, d, p):
    # the K-split of the skinny GEMMs is a cluster of 3, 5, 6 or 7 CTAs here
    # (and 7 or 8 on Hutch++'s pass over G), so rows are finished by CTAs
    # that own unequal row counts; the standard workloads give 1, 2, 4 and 8
    wl = W.Workload(190 + B, f"splits_{B}_{T}_{d}_{p}", B, T, d, p, "bf16", 1e-2, 1.0, 1.0, 32, ())
    _run_all(api, wl, paths=("hutch", "hutchpp"))


@pytest.mark.parametrize("k", [3, 4, 5, 46, 47, 48])
def test_hutchpp_budgets(api, k):
    # r = k // 3 head columns, m = k - 2r tail probes; k = 48 fills all 32 columns
    wl = W.Workload(160 + k, f"hpp_{k}", 2, 260, 96, 192, "bf16", 1e-2, 1.0, 1.0, k, ())
    _run_all(api, wl, paths=("hutchpp",))


@pytest.mark.parametrize("wid", [1, 2, 170, 176])
def test_stored_direct(api, wid):
    # exact norms that keep every A_i^T G_i, then the clipped sum from them:
    # fp32 with d*p not a multiple of 4 (padded per-sample blocks, ragged
    # end), bf16 over several tiles with ragged tails; half the samples clip
    shapes = {170: W.Workload(170, "f32_odd", 3, 37, 29, 50, "f32", 1.0, 1.0, 1.0, 7, ()),
              176: W.Workload(176, "stored_ragged", 5, 300, 200, 328, "bf16", 1e-2, 1.0, 0.7, 8, ())}
    wl = shapes[wid] if wid in shapes else W.get(wid)
    inp = W.make_inputs(wl)
    A, G = to_dev(inp)
    ref = oracle_all(inp, want=())
    tol = TOL[wl.dtype]
    q, stored = api.norms_direct_store(A, G)
    assert_rel(host(q), ref["direct"], tol, "direct (stored)")
    # accumulate: a second layer with the same inputs doubles the sum
    q2 = q.clone()
    api.norms_direct_store(A, G, sqnorms=q2, accumulate=True, ws=stored.ws)
    assert_rel(host(q2), 2 * ref["direct"], tol, "direct (stored, accumulated)")
    C_med = float(np.median(np.sqrt(ref["direct"])))
    check_grad(api, inp, A, G, ref["direct"], C_med, wl.sigma, ref["Ms"], offset=9, stored=stored)


@pytest.mark.parametrize("wid", [170, 177, 4])
def test_bias_grads(api, wid):
    # per-sample bias gradients sum_t G_i[t, :], their share of the norm and
    # the clipped noisy bias gradient; 1100 tokens = two full 512-token chunks
    # and a ragged one, p = 328 a full and a partial 256-column block
    shapes = {170: W.Workload(170, "f32_odd", 3, 37, 29, 50, "f32", 1.0, 1.0, 1.0, 7, ()),
              177: W.Workload(177, "bias_ragged", 3, 1100, 8, 328, "bf16", 1e-2, 1.0, 0.9, 8, ())}
    wl = shapes[wid] if wid in shapes else W.get(wid)
    inp = W.make_inputs(wl)
    A, G = to_dev(inp)
    tol = TOL[wl.dtype]
    b_ref = O.per_sample_bias_grads(inp.G)
    q_b, bg = api.bias_grads(G)
    b = host(bg)
    assert np.max(np.abs(b - b_ref)) <= tol * np.max(np.abs(b_ref))
    assert_rel(host(q_b), O.bias_sqnorms(inp.G), tol, "bias sqnorms")
    # the whole per-sample norm: weights (exact) + bias, accumulated on device
    q_w = api.norms_exact(A, G, method=2 if wl.dtype == "bf16" else 0)
    q_tot = q_w.clone()
    api.bias_grads(G, sqnorms=q_tot, accumulate=True, want_grads=False)
    q_ref = O.sqnorms_direct(inp.A, inp.G) + O.bias_sqnorms(inp.G)
    assert_rel(host(q_tot), q_ref, tol, "weights + bias sqnorms")
    C = float(np.median(np.sqrt(q_ref)))
    q32 = host(q_tot).astype(np.float64)
    Sb, nb, s_ref, bmag = bias_parts(inp, b_ref, q32, C, wl.sigma, 11)
    for sg in (wl.sigma, 0.0):
        Db = host(api.clipped_noisy_bias_grad(bg, q_tot, C, sg, wl.seed, 11))
        assert_grad(Db, Sb, tol, wl.B * wl.T, bmag, nb if sg else None, sg * C,
                    what=f"bias grad (sigma={sg})")


def bias_parts(inp, b_ref, q32, C, sigma, offset):
    """The oracle's clipped bias sum sum_i s_i b_i, its noise (stream 4), the
    scales and mag = sum_i s_i sum_t |G_i[t, :]| for the bound."""
    wl = inp.wl
    Sb, s_ref, _ = O.clipped_noisy_bias_grad(None, q32, C, 0.0, wl.seed, offset, bs=b_ref)
    noise = (sigma * C * O.philox_normals(wl.p, wl.seed, O.STREAM_BIAS_NOISE, offset)
             if sigma != 0.0 else None)
    absb = np.abs(inp.G).astype(np.float64).sum(axis=1)
    return Sb, noise, s_ref, np.sum(s_ref[:, None] * absb, axis=0)


def _check_update(theta0, theta1, scale, S, noise, tol, K, mag, sigmaC, what):
    """theta1 = theta0 - scale * g: the step taken, divided by scale, is the
    gradient the kernel applied, compared with the oracle's clipped sum after
    taking its noise away.  The parameters are rounded to fp32 once more,
    hence a slack of two of their ulps (in gradient units)."""
    g_eff = (theta0.astype(np.float64) - theta1) / scale
    slack = 2.0 * np.spacing(np.abs(theta1).astype(np.float32)).astype(np.float64) / scale
    assert_grad(g_eff, S, tol, K, mag, noise, sigmaC, slack=slack, what=what)


@pytest.mark.parametrize("path", ["gemm_bf16", "gemm_f32", "stored_bf16"])
def test_fused_sgd_update(api, path):
    # weights and bias updated in place by the gradient calls, with and
    # without the gradient itself being stored; the parameters start at the
    # size of one step so that their rounding does not hide the clipped sum
    if path == "gemm_f32":
        wl = W.Workload(170, "f32_odd", 3, 37, 29, 50, "f32", 1.0, 1.0, 1.0, 7, ())
    else:
        wl = W.Workload(176, "stored_ragged", 5, 300, 200, 328, "bf16", 1e-2, 1.0, 0.7, 8, ())
    inp = W.make_inputs(wl)
    A, G = to_dev(inp)
    tol = TOL[wl.dtype]
    K = wl.B * wl.T
    Ms = list(O.per_sample_grads(inp.A, inp.G))
    q_ref = O.sqnorms_direct(inp.A, inp.G) + O.bias_sqnorms(inp.G)
    C = float(np.median(np.sqrt(q_ref)))
    qd = torch.tensor(q_ref, dtype=torch.float32, device="cuda")
    q32 = host(qd).astype(np.float64)
    S, noise, s_ref, mag = oracle_grad_parts(inp, q32, C, wl.sigma, Ms, 5)
    lr, L = 0.3, 7.0
    scale = lr / L
    rng = np.random.default_rng(3)
    for store in (True, False):
        theta0 = (scale * np.abs(S).max() * rng.standard_normal((wl.d, wl.p))).astype(np.float32)
        theta = torch.tensor(theta0, device="cuda")
        upd = api.SGDUpdate(theta, lr, L, store_grad=store)
        if path == "stored_bf16":
            _, stored = api.norms_direct_store(A, G)
            g, _, _ = api.stored_clipped_noisy_grad(stored, qd, C, wl.sigma, wl.seed, 5, update=upd)
        else:
            g, _, _ = api.clipped_noisy_grad(A, G, qd, C, wl.sigma, wl.seed, 5, update=upd)
        _check_update(theta0, host(theta), scale, S, noise, tol, K, mag, wl.sigma * C,
                      f"{path} update (grad stored: {store})")
        if store:
            assert_grad(host(g), S, tol, K, mag, noise, wl.sigma * C, what=f"{path} grad")
        elif path != "gemm_f32":
            assert g is None
    # the bias
    q_b, bg = api.bias_grads(G)
    b_ref = O.per_sample_bias_grads(inp.G)
    Sb, nb, _, bmag = bias_parts(inp, b_ref, q32, C, wl.sigma, 5)
    beta0 = (scale * np.abs(Sb).max() * rng.standard_normal(wl.p)).astype(np.float32)
    beta = torch.tensor(beta0, device="cuda")
    api.clipped_noisy_bias_grad(bg, qd, C, wl.sigma, wl.seed, 5,
                                update=api.SGDUpdate(beta, lr, L, store_grad=False))
    _check_update(beta0, host(beta), scale, Sb, nb, tol, K, bmag, wl.sigma * C, f"{path} bias update")


def test_empty_poisson_lot(api):
    # B = 0: the gradient is the noise alone (streams 3 and 4), the update too
    d, p, C, sigma, lr, L = 40, 24, 2.0, 1.5, 0.3, 10.0
    A = torch.zeros(0, 5, d, dtype=torch.bfloat16, device="cuda")
    G = torch.zeros(0, 5, p, dtype=torch.bfloat16, device="cuda")
    q = torch.zeros(0, device="cuda")
    theta = torch.ones(d, p, device="cuda")
    g, _, _ = api.clipped_noisy_grad(A, G, q, C, sigma, 9, 4, update=api.SGDUpdate(theta, lr, L))
    D_ref, _, _ = O.clipped_noisy_grad(np.zeros((0, 5, d)), np.zeros((0, 5, p)), np.zeros(0), C,
                                       sigma, 9, 4)
    assert np.max(np.abs(host(g) - D_ref)) < 1e-4
    np.testing.assert_allclose(host(theta), O.sgd_update(np.ones((d, p)), D_ref, lr, L), atol=1e-5)
    beta = torch.zeros(p, device="cuda")
    gb = api.clipped_noisy_bias_grad(torch.zeros(0, p, device="cuda"), q, C, sigma, 9, 4,
                                     update=api.SGDUpdate(beta, lr, L))
    Db_ref, _, _ = O.clipped_noisy_bias_grad(None, np.zeros(0), C, sigma, 9, 4, bs=np.zeros((0, p)))
    assert np.max(np.abs(host(gb) - Db_ref)) < 1e-4
    np.testing.assert_allclose(host(beta), -lr / L * Db_ref, atol=1e-5)


def test_gradient_noise_is_the_oracle_stream(api):
    # With A = 0 (G = 0 for the bias) the clipped sum vanishes and each path
    # returns sigma C z, z the Philox normals of its stream at element r p + c
    # (stream 3) or c (stream 4).  The kernels draw them with the SFU's log2,
    # sine and cosine (and a series for the log near 1): every value within
    # NOISE_TOL of the fp64 transform.
    # The bf16 GEMM case draws a whole up_proj gradient (2048 x 8192 normals),
    # the size at which NOISE_TOL is used by the gradient checks.
    C, sigma, seed, off = 2.0, 1.5, 0x5EED, 11
    tol = NOISE_TOL * sigma * C
    for dtype, (B, T, d, p) in ((torch.bfloat16, (3, 70, 200, 328)),
                                (torch.bfloat16, (1, 16, 2048, 8192)),
                                (torch.float32, (2, 9, 24, 40))):
        A = torch.zeros(B, T, d, dtype=dtype, device="cuda")
        G = torch.randn(B, T, p, device="cuda").to(dtype)
        q = torch.ones(B, device="cuda")
        z = O.philox_normals(d * p, seed, 3, off).reshape(d, p)
        g, _, _ = api.clipped_noisy_grad(A, G, q, C, sigma, seed, off)
        err = np.max(np.abs(host(g) - sigma * C * z))
        assert err < tol, f"{dtype} {d}x{p} gemm: {err / (sigma * C):.2e} sigma C"
        q2, stored = api.norms_direct_store(A, G)
        gs, _, _ = api.stored_clipped_noisy_grad(stored, q, C, sigma, seed, off)
        err = np.max(np.abs(host(gs) - sigma * C * z))
        assert err < tol, f"{dtype} {d}x{p} stored: {err / (sigma * C):.2e} sigma C"
    p = 520
    zb = O.philox_normals(p, seed, 4, off)
    _, bg = api.bias_grads(torch.zeros(2, 33, p, dtype=torch.bfloat16, device="cuda"))
    gb = api.clipped_noisy_bias_grad(bg, torch.ones(2, device="cuda"), C, sigma, seed, off)
    err = np.max(np.abs(host(gb) - sigma * C * zb))
    assert err < tol, f"bias: {err / (sigma * C):.2e} sigma C"


FIBER_HP = dict(lr=0.05, beta1=0.9, beta2=0.99, eps=1e-6, eps_v=1e-10, weight_decay=0.01,
                omega=0.4)


def _fiber_oracle_steps(theta0, grads, denom, noise_var, hp):
    theta = theta0.astype(np.float64)
    st = tuple(np.zeros_like(theta) for _ in range(4))
    out = []
    for t, g in enumerate(grads, start=1):
        theta, st = O.fiber_adamw_step(theta, np.asarray(g, np.float64) / denom, st, t, hp["lr"],
                                       hp["beta1"], hp["beta2"], hp["eps"], hp["eps_v"],
                                       hp["weight_decay"], hp["omega"], noise_var)
        out.append((theta, st))
    return out


def _check_fiber(opt, ref, theta0, rtol=2e-4):
    theta_ref, (gf, r, m, v) = ref
    scale = np.abs(theta_ref - theta0).max()
    assert np.max(np.abs(host(opt.param) - theta_ref)) <= rtol * scale + 1e-6 * np.abs(theta0).max()
    for got, want in ((opt.filt, gf), (opt.resid, r), (opt.m, m), (opt.v, v)):
        assert np.max(np.abs(host(got) - want)) <= rtol * np.abs(want).max() + 1e-30


def test_fiber_step_matches_oracle(api):
    # the standalone step over several steps, 1003 elements (a ragged end)
    rng = np.random.default_rng(7)
    n, denom, nv = 1003, 4.0, 0.02
    theta0 = rng.standard_normal(n).astype(np.float32)
    grads = [4.0 * rng.standard_normal(n).astype(np.float32) for _ in range(4)]
    opt = api.FiberAdamW(torch.tensor(theta0, device="cuda"), denom=denom, noise_var=nv,
                         **FIBER_HP)
    ref = _fiber_oracle_steps(theta0, grads, denom, nv, FIBER_HP)
    for t, g in enumerate(grads):
        api.fiber_step(torch.tensor(g, device="cuda"), opt)
        _check_fiber(opt, ref[t], theta0)


@pytest.mark.parametrize("path", ["gemm_bf16", "gemm_f32", "stored_bf16", "bias", "empty"])
def test_fiber_fused(api, path):
    # the FIBER step applied where the gradient is formed; the oracle's step is
    # fed the gradient the GPU formed (its parity is tested above), so this
    # checks the fused step itself over two steps of carried state
    if path == "gemm_f32":
        wl = W.Workload(170, "f32_odd", 3, 37, 29, 50, "f32", 1.0, 1.0, 1.0, 7, ())
    else:
        wl = W.Workload(176, "stored_ragged", 5, 300, 200, 328, "bf16", 1e-2, 1.0, 0.7, 8, ())
    inp = W.make_inputs(wl)
    A, G = to_dev(inp)
    if path == "empty":
        A, G = A[:0], G[:0]
    q = torch.tensor(O.sqnorms_direct(inp.A, inp.G) + O.bias_sqnorms(inp.G), dtype=torch.float32,
                     device="cuda")
    C = float(np.median(np.sqrt(host(q))))
    denom = 5.0
    nv = (wl.sigma * C / denom) ** 2
    shape = (wl.p,) if path == "bias" else (wl.d, wl.p)
    theta0 = np.random.default_rng(8).standard_normal(shape).astype(np.float32)
    opt = api.FiberAdamW(torch.tensor(theta0, device="cuda"), denom=denom, noise_var=nv,
                         **FIBER_HP)
    grads = []
    if path == "stored_bf16":
        _, stored = api.norms_direct_store(A, G)
    if path == "bias":
        _, bg = api.bias_grads(G)
    q32 = host(q)
    tol, K = TOL[wl.dtype], wl.B * wl.T
    Ms = list(O.per_sample_grads(inp.A, inp.G)) if path not in ("bias", "empty") else None
    for step in range(2):
        if path == "stored_bf16":
            g, _, _ = api.stored_clipped_noisy_grad(stored, q, C, wl.sigma, wl.seed, step, fiber=opt)
        elif path == "bias":
            g = api.clipped_noisy_bias_grad(bg, q, C, wl.sigma, wl.seed, step, fiber=opt)
        else:
            g, _, _ = api.clipped_noisy_grad(A, G, q[:A.shape[0]], C, wl.sigma, wl.seed, step,
                                             fiber=opt)
        grads.append(host(g).copy())
        # the gradient the step was fed, against the oracle's clipped sum
        if path == "bias":
            Sb, nb, _, bmag = bias_parts(inp, O.per_sample_bias_grads(inp.G), q32, C, wl.sigma,
                                         step)
            assert_grad(grads[-1], Sb, tol, K, bmag, nb, wl.sigma * C, what="fiber bias grad")
        elif path != "empty":
            S, noise, _, mag = oracle_grad_parts(inp, q32, C, wl.sigma, Ms, step)
            assert_grad(grads[-1], S, tol, K, mag, noise, wl.sigma * C, what=f"fiber {path} grad")
        ref = _fiber_oracle_steps(theta0, grads, denom, nv, FIBER_HP)[-1]
        _check_fiber(opt, ref, theta0)


@pytest.mark.parametrize("case", ["bf16", "f32_rankdef"])
def test_hutchpp_wide_layer(api, case):
    # p = 20000 (17001) rows: each CTA of the sample's cluster owns more rows
    # than it keeps resident, so V and G' are staged tile by tile in every pass;
    # with T = 7 < r = 10 the head also drops dependent columns on that path.
    if case == "bf16":
        wl = W.Workload(174, "hpp_wide", 2, 40, 24, 20000, "bf16", 1e-2, 1.0, 1.0, 32, ())
    else:
        wl = W.Workload(175, "hpp_wide_f32", 2, 7, 24, 17001, "f32", 1.0, 1.0, 1.0, 32, ())
    _run_all(api, wl, paths=("hutchpp",))


def test_f32_odd_shapes(api):
    wl = W.Workload(170, "f32_odd", 3, 37, 29, 50, "f32", 1.0, 1.0, 1.0, 7, ())
    _run_all(api, wl)


def test_many_samples_per_tile(api):
    # 33 samples: the gradient's tiles are split over many CTAs by sample
    wl = W.Workload(171, "many_samples", 33, 24, 64, 64, "bf16", 1e-2, 0.5, 1.0, 8, ())
    _run_all(api, wl)


def test_long_sequence_narrow_layer(api):
    wl = W.Workload(172, "long_narrow", 1, 5000, 8, 16, "bf16", 1e-2, 0.5, 1.0, 6, ())
    _run_all(api, wl)


def test_grad_tail_split_over_k(api):
    # 64 pair tiles on 76 CTA pairs: no full wave, every tile is cut into
    # bands over its samples and K-blocks and summed from partial tiles
    wl = W.Workload(173, "waves", 2, 1100, 1024, 4096, "bf16", 1e-3, 0.5, 0.0, 8, ())
    inp = W.make_inputs(wl)
    A, G = to_dev(inp)
    Ms = list(O.per_sample_grads(inp.A, inp.G))
    q = np.array([np.sum(M * M) for M in Ms])
    check_grad(api, inp, A, G, q, float(np.sqrt(q).min()), 0.0, Ms)


def test_grad_tail_bands(api):
    # 104 pair tiles: on 76 pairs one full wave and 28 tiles cut into bands
    # over three levels (pairs with up to three segments, tiles summed from
    # up to four partial sums); ragged T, d and p
    from dp_sgd_clipping_gb300 import _lib
    _, ntail, segs, contrib = _lib.grad_tail_schedule(76, 104, 2, 20)
    assert ntail == 28 and np.bincount(segs[:, 0]).max() == 2
    assert np.bincount(contrib[:, 0]).max() == 4
    wl = W.Workload(174, "tail_bands", 2, 1270, 248, 26616, "bf16", 1e-3, 0.5, 0.8, 8, ())
    inp = W.make_inputs(wl)
    A, G = to_dev(inp)
    Ms = list(O.per_sample_grads(inp.A, inp.G))
    q = np.array([np.sum(M * M) for M in Ms])
    check_grad(api, inp, A, G, q, float(np.sqrt(q).min()), wl.sigma, Ms)


def test_grad_tail_three_segments(api):
    # 180 pair tiles: on 76 pairs two full waves and 28 tiles whose bands go
    # three levels deep (pairs with three segments, run shortest first; tiles
    # summed from up to five partial sums); ragged T, d and p
    from dp_sgd_clipping_gb300 import _lib
    _, ntail, segs, contrib = _lib.grad_tail_schedule(76, 180, 2, 16)
    assert ntail == 28 and np.bincount(segs[:, 0]).max() == 3
    assert np.bincount(contrib[:, 0]).max() == 5
    wl = W.Workload(175, "tail_three_segments", 2, 1000, 248, 46072, "bf16", 1e-3, 0.5, 0.8, 8, ())
    inp = W.make_inputs(wl)
    A, G = to_dev(inp)
    Ms = list(O.per_sample_grads(inp.A, inp.G))
    q = np.array([np.sum(M * M) for M in Ms])
    check_grad(api, inp, A, G, q, float(np.sqrt(q).min()), wl.sigma, Ms)


# ----------------------------------------------------------------------------- Rademacher probes

def test_rademacher_fill_is_exact(api):
    n = (1 << 18) + 5
    for dt in (torch.float32, torch.bfloat16):
        r = api.philox_rademacher(n, seed=4242, stream_id=0, offset=(1 << 35) + 9, dtype=dt)
        ref = O.philox_rademacher(n, 4242, 0, (1 << 35) + 9)
        assert np.array_equal(host(r), ref)


@pytest.mark.parametrize("case", ["bf16", "f32"])
def test_rademacher_estimators(api, case):
    if case == "bf16":
        wl = W.Workload(180, "rad_bf16", 3, 300, 200, 328, "bf16", 1e-2, 1.0, 1.0, 24, ())
    else:
        wl = W.get(1)
    inp = W.make_inputs(wl)
    A, G = to_dev(inp)
    Ms = list(O.per_sample_grads(inp.A, inp.G))
    P = O.hutch_probe(wl.p, wl.k, wl.seed, 2, wl.dtype, kind="rademacher")
    S, Gp = O.hutchpp_probes(wl.p, wl.k, wl.seed, 2, wl.dtype, kind="rademacher")
    tol = TOL[wl.dtype]
    assert_rel(host(api.norms_hutch(A, G, wl.k, wl.seed, 2, probe="rademacher")),
               O.sqnorms_hutch(None, None, P, Ms=Ms), tol, "hutch rademacher")
    assert_rel(host(api.norms_hutchpp(A, G, wl.k, wl.seed, 2, probe="rademacher")),
               O.sqnorms_hutchpp(None, None, S, Gp, Ms=Ms), tol, "hutch++ rademacher")
