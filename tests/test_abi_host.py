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
    # gradient: tile tickets plus three partial 128x256 fp32 tiles per CTA (the
    # segments of the tail schedule; at most 160 CTAs)
    g = ws(L.OP_CLIPPED_NOISY_GRAD, 4, 4096, 2048, 8192, L.BF16, 0)
    assert 3 * 160 * 128 * 256 * 4 <= g <= 3 * 160 * 128 * 256 * 4 + 4096
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
    # sizes past the index ranges: d * p beyond the Philox block index (2^34
    # elements), B * T beyond 2^30 tokens
    for B, T, d, p in ((1, 8, 1 << 18, 1 << 17), (1 << 16, 1 << 15, 16, 16)):
        assert lib.dpclip_norms_exact(FAKE, FAKE, B, T, d, p, L.BF16, 0, FAKE, FAKE, big,
                                      None) == L.ERR_UNSUPPORTED
        assert lib.dpclip_norms_hutch(FAKE, FAKE, B, T, d, p, L.BF16, 8, 1, 0, FAKE, FAKE, big,
                                      None) == L.ERR_UNSUPPORTED
        assert g(FAKE, FAKE, B, T, d, p, L.BF16, FAKE, 1.0, 1.0, 1, 0, FAKE, None, None, FAKE,
                 big, None) == L.ERR_UNSUPPORTED
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


# ----------------------------------------------------------------------------- gradient tail schedule

def _tail_cases():
    # (pairs, pair tiles, samples, 64-token blocks per sample)
    cases = [(76, 256, 4, 64), (76, 64, 4, 64), (76, 64, 1, 128), (74, 256, 4, 64),
             (76, 8 * 32, 1, 1), (80, 79, 1, 1), (80, 79, 4, 64), (76, 75, 2, 3),
             (3, 5, 2, 1), (1, 1, 1, 1), (76, 152, 8, 16), (76, 1, 33, 1)]
    for pairs in (2, 5, 13, 37, 64, 76, 80):
        for ntiles in (1, pairs - 1, pairs + 1, 2 * pairs + pairs // 3, 3 * pairs + 7):
            for B, tb in ((1, 1), (2, 5), (4, 64), (3, 100)):
                if ntiles >= 1:
                    cases.append((pairs, ntiles, B, tb))
    return cases


def test_grad_tail_schedule_covers_once(L):
    """Every (tile, K-block) of the tiles left after the full waves belongs
    to exactly one segment; each pair holds at most three partial tiles;
    slots are unique and below 3 per pair; the contributions of a tile are
    exactly the slots of its segments, added in slot order; and the busiest
    pair carries no more than a whole tile's time line."""
    import numpy as np
    for pairs, ntiles, B, tb in _tail_cases():
        waves, ntail, segs, contrib = L.grad_tail_schedule(pairs, ntiles, B, tb)
        assert waves == ntiles // pairs and ntail == ntiles % pairs
        Lt = B * tb
        if ntail == 0:
            assert len(segs) == 0 and len(contrib) == 0
            continue
        cover = np.zeros((ntail, Lt), dtype=np.int32)
        work = np.zeros(pairs, dtype=np.int64)
        count = np.zeros(pairs, dtype=np.int64)
        for c, t, t0, t1, sl in segs:
            assert 0 <= c < pairs and 0 <= t < ntail and 0 <= t0 < t1 <= Lt
            cover[t, t0:t1] += 1
            work[c] += t1 - t0
            count[c] += 1
        assert (cover == 1).all(), (pairs, ntiles, B, tb)
        assert count.max() <= 3
        slots = segs[:, 4]
        assert len(set(slots.tolist())) == len(slots) and slots.min() >= 0
        assert slots.max() < 3 * pairs
        assert list(segs[:, 0]) == sorted(segs[:, 0])
        for t in range(ntail):
            mine = sorted(segs[segs[:, 1] == t][:, 4].tolist())
            listed = contrib[contrib[:, 0] == t][:, 1].tolist()
            assert listed == mine, (pairs, ntiles, B, tb, t)
        assert work.max() <= Lt


def test_grad_tail_schedule_balance(L):
    """Where the time line is long, the busiest pair of the tail stays near
    the fair share ntail * L / pairs; on the up_proj shape (256 pair tiles,
    76 pairs, 4 samples of 64 blocks) it is within two K-blocks of it, and
    most pairs hold a single segment."""
    import numpy as np
    _, ntail, segs, _ = L.grad_tail_schedule(76, 256, 4, 64)
    assert ntail == 28
    work = np.bincount(segs[:, 0], weights=segs[:, 3] - segs[:, 2], minlength=76)
    fair = 28 * 256 / 76
    assert work.max() <= fair + 2
    assert np.sum(np.bincount(segs[:, 0], minlength=76) == 1) >= 50
    for pairs, ntiles, B, tb in _tail_cases():
        if B * tb < 64:
            continue
        _, ntail, segs, _ = L.grad_tail_schedule(pairs, ntiles, B, tb)
        if ntail == 0:
            continue
        work = np.bincount(segs[:, 0], weights=segs[:, 3] - segs[:, 2], minlength=pairs)
        assert work.max() <= 1.35 * ntail * B * tb / pairs + 1, (pairs, ntiles, B, tb)


def test_grad_tail_schedule_rejects(L):
    import ctypes as C
    w, n, ns, nc = C.c_int(), C.c_int(), C.c_int(), C.c_int()
    for args in ((0, 4, 1, 1), (81, 4, 1, 1), (4, 0, 1, 1), (4, 4, 0, 1), (4, 4, 1, 0)):
        st = L.lib.dpclip_grad_tail_schedule(*args, C.byref(w), C.byref(n), None, 0, C.byref(ns),
                                             None, 0, C.byref(nc))
        assert st == L.ERR_INVALID_ARG


def _ghost_items(nfull, tail_units, split, pbc, shared, pblocks, dblocks):
    """The sub-units of the ghost kernel's last round, in item order: (tail
    unit, first K-block over d count, p-block range), as the kernel deals
    them (one X sub-unit first when shared)."""
    items = []
    per = split + shared
    for t in range(tail_units * per):
        tu, c = divmod(t, per)
        kx = dblocks
        if shared:
            if c == 0:
                items.append((tu, dblocks, 0, 0))
                continue
            kx, c = 0, c - 1
        pb0 = c * pbc
        items.append((tu, kx, pb0, min(pb0 + pbc, pblocks)))
    return items


def test_ghost_schedule_covers_once(L):
    """Every unit of the ghost form's last round has each of its p-blocks in
    exactly one sub-unit and its A Gram block formed by exactly one sub-unit
    per p-slice (recomputed) or once for all (shared); with a shared Gram
    block each pair holds at most one sub-unit of that round, so no pair
    both waits for a Gram block and owes one; and the chosen cut costs no
    more K-blocks than dealing the units whole."""
    for pairs in (1, 2, 7, 40, 76, 80):
        for B, T in ((1, 300), (2, 2048), (4, 4096), (3, 4352), (1, 16384)):
            for d, p in ((64, 64), (256, 512), (1024, 2048), (2048, 8192), (2048, 2048), (4096, 512)):
                units = B * ((T + 255) // 256) * ((T + 255) // 256 + 1) // 2
                grid = min(pairs, units)
                nfull, split, pbc, shared = L.ghost_schedule(pairs, B, T, d, p)
                db, pb = (d + 63) // 64, (p + 63) // 64
                assert nfull == units // grid * grid
                tail = units - nfull
                assert split >= 1 and (split - 1) * pbc < pb <= split * pbc
                assert shared in (0, 1)
                if tail == 0:
                    assert (split, pbc, shared) == (1, pb, 0)
                    continue
                items = _ghost_items(nfull, tail, split, pbc, shared, pb, db)
                for tu in range(tail):
                    mine = [it for it in items if it[0] == tu]
                    cover = [0] * pb
                    for _, kx, b0, b1 in mine:
                        for k in range(b0, b1):
                            cover[k] += 1
                    assert cover == [1] * pb
                    gram = [kx for _, kx, _, _ in mine]
                    if shared:
                        assert gram.count(db) == 1 and gram.count(0) == split
                    else:
                        assert gram == [db] * split
                if shared:
                    assert len(items) <= grid
                    cost = max(db, pbc) + 10
                else:
                    cost = -(-len(items) // grid) * (db + pbc)
                assert cost <= db + pb, (pairs, B, T, d, p)


def test_ghost_schedule_up_proj(L):
    # 544 units on 76 pairs: 7 whole rounds, 12 units left, each one Gram
    # sub-unit over d (32 K-blocks) and four 32-block slices of p, all 60 of
    # them at once on their own pairs; on q_proj (p = 2048) six 6-block
    # slices that each recompute the Gram block cost less than sharing it
    assert L.ghost_schedule(76, 4, 4096, 2048, 8192) == (532, 4, 32, 1)
    assert L.ghost_schedule(76, 4, 4096, 2048, 2048) == (532, 6, 6, 0)


def test_ghost_schedule_rejects(L):
    import ctypes as C
    o = [C.c_int() for _ in range(4)]
    for args in ((0, 1, 64, 64, 64), (81, 1, 64, 64, 64), (4, 0, 64, 64, 64), (4, 1, 0, 64, 64),
                 (4, 1, 64, 0, 64), (4, 1, 64, 64, 0)):
        assert L.lib.dpclip_ghost_schedule(*args, *[C.byref(x) for x in o]) == L.ERR_INVALID_ARG
    assert L.lib.dpclip_ghost_schedule(4, 1, 64, 64, 64, None, *[C.byref(x) for x in o[1:]]) == \
        L.ERR_INVALID_ARG
