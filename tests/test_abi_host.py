"""Host-only checks of the C ABI: the library loads, exports every declared
entry point, sizes workspaces, and rejects bad arguments with a status code
before it touches the GPU (none of these calls reaches a CUDA launch)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__.build()
    from dp_sgd_clipping_gb300 import _lib
    return _lib


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "dpclip.h")).read()
    return sorted(set(re.findall(r"\b(dpclip_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(L):
    names = declared_symbols()
    assert len(names) >= 15
    for n in names:
        assert hasattr(L.lib, n), n
        assert n in L.SIGNATURES, n


def test_status_strings_and_version(L):
    assert L.status_string(0) == "ok"
    assert "timed out" in L.status_string(L.ERR_TIMEOUT)
    assert L.lib.dpclip_version().decode().startswith("dpclip")


def test_workspace_sizes(L):
    ws = L.workspace_size
    n1 = ws(L.OP_NORMS_HUTCH, 4, 4096, 2048, 8192, L.BF16, 32)
    n2 = ws(L.OP_NORMS_HUTCH, 4, 4096, 2048, 8192, L.BF16, 8)
    assert n1 >= n2 > 0 and n1 % 256 == 0
    # O(BkT + kp) memory of the randomized estimator: far below one d x p gradient
    assert n1 < 2048 * 8192 * 4 / 4
    assert ws(L.OP_NORMS_HUTCHPP, 4, 4096, 2048, 8192, L.BF16, 32) > n1
    # gradient: tile tickets plus two partial 128x256 fp32 tiles per CTA of the
    # balanced tail (at most 160 CTAs)
    g = ws(L.OP_CLIPPED_NOISY_GRAD, 4, 4096, 2048, 8192, L.BF16, 0)
    assert 2 * 160 * 128 * 256 * 4 <= g <= 2 * 160 * 128 * 256 * 4 + 4096
    assert ws(L.OP_CLIPPED_NOISY_GRAD, 4, 64, 32, 48, L.F32, 0) == 256
    direct = ws(L.OP_NORMS_EXACT, 8, 512, 768, 768, L.BF16, L.EXACT_DIRECT)
    ghost = ws(L.OP_NORMS_EXACT, 8, 512, 768, 768, L.BF16, L.EXACT_GHOST)
    assert direct > 0 and ghost > 0
    assert ws(L.OP_NORMS_HUTCH, 4, 64, 32, 48, L.F32, 8) > 0
    assert ws(L.OP_NORMS_EXACT, 4, 64, 32, 48, L.F32, L.EXACT_GHOST) >= 4 * 64 * 64 * 4
    # stored direct norms: the control block, B fp32 d x p gradients (each
    # padded to a multiple of 4 floats), then the norm partials
    st = ws(L.OP_STORED_DIRECT, 4, 4096, 2048, 8192, L.BF16, 0)
    assert 256 + 4 * 2048 * 8192 * 4 < st < 256 + 4 * 2048 * 8192 * 4 + (1 << 20)
    assert ws(L.OP_STORED_DIRECT, 3, 37, 29, 50, L.F32, 0) >= 256 + 3 * 1452 * 4
    # bias: per (sample, 512-token chunk) column sums
    assert ws(L.OP_BIAS, 4, 4096, 0, 8192, L.BF16, 0) == (4 * 8 * 8192 + 4 * 32) * 4


def test_workspace_size_rejects(L):
    n = ctypes.c_size_t(0)
    f = L.lib.dpclip_workspace_size
    assert f(L.OP_NORMS_HUTCH, 0, 1, 8, 8, L.BF16, 8, ctypes.byref(n)) == L.ERR_INVALID_ARG
    assert f(L.OP_NORMS_HUTCH, 1, 1, 8, 8, 7, 8, ctypes.byref(n)) == L.ERR_INVALID_ARG
    assert f(L.OP_NORMS_HUTCH, 1, 1, 8, 8, L.BF16, 33, ctypes.byref(n)) == L.ERR_UNSUPPORTED
    assert f(L.OP_NORMS_HUTCH, 1, 1, 8, 8, L.BF16, 0, ctypes.byref(n)) == L.ERR_UNSUPPORTED
    assert f(L.OP_NORMS_HUTCHPP, 1, 1, 8, 8, L.BF16, 2, ctypes.byref(n)) == L.ERR_UNSUPPORTED
    assert f(L.OP_NORMS_HUTCHPP, 1, 1, 8, 8, L.BF16, 49, ctypes.byref(n)) == L.ERR_UNSUPPORTED
    assert f(L.OP_NORMS_EXACT, 1, 1, 8, 8, L.BF16, 9, ctypes.byref(n)) == L.ERR_INVALID_ARG
    assert f(99, 1, 1, 8, 8, L.BF16, 0, ctypes.byref(n)) == L.ERR_INVALID_ARG
    assert f(L.OP_NORMS_HUTCH, 1, 1, 8, 8, L.BF16, 8, None) == L.ERR_INVALID_ARG


FAKE = 1 << 40           # aligned, never dereferenced: every call below fails its checks first


def test_entry_points_reject_before_any_launch(L):
    lib = L.lib
    big = 1 << 30
    # null inputs
    assert lib.dpclip_norms_hutch(None, FAKE, 2, 8, 16, 16, L.BF16, 8, 1, 0, FAKE, FAKE, big,
                                  None) == L.ERR_INVALID_ARG
    assert lib.dpclip_norms_exact(FAKE, FAKE, 2, 8, 16, 16, L.BF16, 0, None, FAKE, big,
                                  None) == L.ERR_INVALID_ARG
    # bf16 rows must be 16-byte multiples
    assert lib.dpclip_norms_hutch(FAKE, FAKE, 2, 8, 12, 16, L.BF16, 8, 1, 0, FAKE, FAKE, big,
                                  None) == L.ERR_UNSUPPORTED
    # misaligned bf16 base pointer
    assert lib.dpclip_norms_hutchpp(FAKE + 2, FAKE, 2, 8, 16, 16, L.BF16, 9, 1, 0, FAKE, FAKE,
                                    big, None) == L.ERR_UNSUPPORTED
    # bad k
    assert lib.dpclip_norms_hutch(FAKE, FAKE, 2, 8, 16, 16, L.BF16, 40, 1, 0, FAKE, FAKE, big,
                                  None) == L.ERR_UNSUPPORTED
    # workspace missing / misaligned / too small
    assert lib.dpclip_norms_hutch(FAKE, FAKE, 2, 8, 16, 16, L.BF16, 8, 1, 0, FAKE, None, big,
                                  None) == L.ERR_WORKSPACE
    assert lib.dpclip_norms_hutch(FAKE, FAKE, 2, 8, 16, 16, L.BF16, 8, 1, 0, FAKE, FAKE + 16, big,
                                  None) == L.ERR_WORKSPACE
    assert lib.dpclip_norms_hutch(FAKE, FAKE, 2, 8, 16, 16, L.BF16, 8, 1, 0, FAKE, FAKE, 255,
                                  None) == L.ERR_WORKSPACE
    # gradient: bad C / sigma / null output
    g = lib.dpclip_clipped_noisy_grad
    assert g(FAKE, FAKE, 2, 8, 16, 16, L.BF16, FAKE, 0.0, 1.0, 1, 0, FAKE, None, None, FAKE, big,
             None) == L.ERR_INVALID_ARG
    assert g(FAKE, FAKE, 2, 8, 16, 16, L.BF16, FAKE, 1.0, -1.0, 1, 0, FAKE, None, None, FAKE, big,
             None) == L.ERR_INVALID_ARG
    assert g(FAKE, FAKE, 2, 8, 16, 16, L.BF16, FAKE, float("nan"), 1.0, 1, 0, FAKE, None, None,
             FAKE, big, None) == L.ERR_INVALID_ARG
    assert g(FAKE, FAKE, 2, 8, 16, 16, L.BF16, FAKE, 1.0, 1.0, 1, 0, None, None, None, FAKE, big,
             None) == L.ERR_INVALID_ARG
    # non-positive sizes
    for B, T, d, p in ((0, 8, 16, 16), (2, 0, 16, 16), (2, 8, -8, 16), (2, 8, 16, 0)):
        assert lib.dpclip_norms_exact(FAKE, FAKE, B, T, d, p, L.F32, 0, FAKE, FAKE, big,
                                      None) == L.ERR_INVALID_ARG
    assert lib.dpclip_philox_normal(None, 10, L.F32, 1, 0, 0, None) == L.ERR_INVALID_ARG
    assert lib.dpclip_philox_normal(FAKE + 2, 10, L.F32, 1, 0, 0, None) == L.ERR_UNSUPPORTED
    assert lib.dpclip_clip_scales(FAKE, 4, -1.0, FAKE, FAKE, None) == L.ERR_INVALID_ARG
    assert lib.dpclip_selftest_wait_timeout(FAKE, 256, 0, None) == L.ERR_INVALID_ARG
    assert lib.dpclip_workspace_status(None, None) == L.ERR_INVALID_ARG
    # unknown probe law
    assert lib.dpclip_norms_hutch_ex(FAKE, FAKE, 2, 8, 16, 16, L.BF16, 8, 7, 1, 0, FAKE, FAKE, big,
                                     None) == L.ERR_INVALID_ARG
    assert lib.dpclip_norms_hutchpp_ex(FAKE, FAKE, 2, 8, 16, 16, L.BF16, 9, -1, 1, 0, FAKE, FAKE,
                                       big, None) == L.ERR_INVALID_ARG
    assert lib.dpclip_philox_rademacher(None, 10, L.F32, 1, 0, 0, None) == L.ERR_INVALID_ARG
    # bias of the linear layer
    bg = lib.dpclip_bias_grads
    assert bg(FAKE, 2, 8, 16, L.BF16, 0, None, None, FAKE, big, None) == L.ERR_INVALID_ARG
    assert bg(FAKE, 2, 8, 12, L.BF16, 0, FAKE, FAKE, FAKE, big, None) == L.ERR_UNSUPPORTED
    assert bg(FAKE, 2, 8, 16, L.BF16, 3, FAKE, FAKE, FAKE, big, None) == L.ERR_INVALID_ARG
    assert bg(FAKE, 2, 8, 16, L.BF16, 0, FAKE, FAKE, FAKE, 0, None) == L.ERR_WORKSPACE
    cb = lib.dpclip_clipped_noisy_bias_grad
    assert cb(FAKE, 2, 16, FAKE, 0.0, 1.0, 1, 0, FAKE, None) == L.ERR_INVALID_ARG
    assert cb(None, 2, 16, FAKE, 1.0, 1.0, 1, 0, FAKE, None) == L.ERR_INVALID_ARG
    assert cb(FAKE, 20000, 16, FAKE, 1.0, 1.0, 1, 0, FAKE, None) == L.ERR_UNSUPPORTED
    # FIBER: bad gain, step, missing state
    fo = L.FiberAdamW(FAKE, FAKE, FAKE, FAKE, FAKE, 1e-3, 0.9, 0.999, 1e-8, 0.0, 0.0, 1.5, 0.0,
                      1.0, 1)
    assert lib.dpclip_fiber_adamw_step(FAKE, 16, ctypes.byref(fo), None) == L.ERR_INVALID_ARG
    fo.omega = 0.5
    fo.step = 0
    assert lib.dpclip_fiber_adamw_step(FAKE, 16, ctypes.byref(fo), None) == L.ERR_INVALID_ARG
    fo.step = 1
    fo.m = None
    assert lib.dpclip_fiber_adamw_step(FAKE, 16, ctypes.byref(fo), None) == L.ERR_INVALID_ARG
    fo.m = FAKE
    fo.v = FAKE + 4
    assert lib.dpclip_clipped_noisy_grad_fiber(FAKE, FAKE, 2, 8, 16, 16, L.BF16, FAKE, 1.0, 1.0, 1,
                                               0, None, None, None, ctypes.byref(fo), FAKE, big,
                                               None) == L.ERR_UNSUPPORTED
    assert lib.dpclip_stored_clipped_noisy_grad_fiber(2, 16, 16, FAKE, 1.0, 1.0, 1, 0, None, None,
                                                      None, None, FAKE, big,
                                                      None) == L.ERR_INVALID_ARG
    # stored direct norms and their gradient
    st = lib.dpclip_norms_direct_store
    assert st(FAKE, FAKE, 2, 8, 16, 16, L.BF16, 2, FAKE, FAKE, big, None) == L.ERR_INVALID_ARG
    assert st(FAKE, FAKE, 2, 8, 16, 16, L.BF16, 0, None, FAKE, big, None) == L.ERR_INVALID_ARG
    assert st(FAKE, FAKE, 2, 8, 16, 16, L.BF16, 0, FAKE, FAKE, 1024, None) == L.ERR_WORKSPACE
    sg = lib.dpclip_stored_clipped_noisy_grad
    assert sg(0, 16, 16, FAKE, 1.0, 1.0, 1, 0, FAKE, None, None, FAKE, big, None) == L.ERR_INVALID_ARG
    assert sg(2, 16, 16, FAKE, -1.0, 1.0, 1, 0, FAKE, None, None, FAKE, big, None) == L.ERR_INVALID_ARG
    assert sg(2, 16, 16, FAKE, 1.0, 1.0, 1, 0, FAKE + 4, None, None, FAKE, big,
              None) == L.ERR_UNSUPPORTED
    assert sg(2, 16, 16, FAKE, 1.0, 1.0, 1, 0, FAKE, None, None, FAKE, 256 + 2 * 256 * 4 - 1,
              None) == L.ERR_WORKSPACE


def test_product_path_does_not_import_oracle():
    pat = re.compile(r"^\s*(import\s+oracle|from\s+oracle|from\s+\.\.oracle)|oracle/|dpclip_oracle",
                     re.M)
    pkg = os.path.join(ROOT, "dp_sgd_clipping_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                assert not pat.search(open(os.path.join(dirpath, f)).read()), f
