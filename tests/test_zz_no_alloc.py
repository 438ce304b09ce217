"""dpclip_norms_hutch_noalloc: the Hutch norms for callers that cannot allocate
device memory where they need them (a framework callback that forbids device
allocation after set-up, a process whose memory belongs to another allocator,
a latency-critical loop).  It uses a library-owned scratch array instead of a
caller workspace.  Compared, through the C ABI, with dpclip_norms_hutch on the
same inputs, two calls in a row, bit for bit (both run the same deterministic
kernels), with the scratch array's status read after each call.  This file is
collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

from dp_sgd_clipping_gb300 import workloads as W
from gpu_util import host, to_dev


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__.build()
    from dp_sgd_clipping_gb300 import _lib
    return _lib


def _noalloc(L, A, G, dtype, k, seed, offset):
    B, T, d = A.shape
    p = G.shape[2]
    out = torch.full((B,), float("nan"), dtype=torch.float32, device=A.device)
    st = L.lib.dpclip_norms_hutch_noalloc(A.data_ptr(), G.data_ptr(), B, T, d, p, dtype, k, seed,
                                          offset, out.data_ptr(),
                                          torch.cuda.current_stream().cuda_stream)
    assert st == L.OK, L.status_string(st)
    return out


def test_noalloc_rejects_sizes_beyond_its_scratch(L):
    fake = 1 << 40      # never dereferenced: the size check comes first
    # B*T = 524288 tokens at k = 32: the sketch alone needs 64 MiB
    n = ctypes.c_size_t(0)
    L.lib.dpclip_workspace_size(L.OP_NORMS_HUTCH, 64, 8192, 2048, 8192, L.BF16, 32, ctypes.byref(n))
    assert n.value > L.NOALLOC_SCRATCH_BYTES
    assert L.lib.dpclip_norms_hutch_noalloc(fake, fake, 64, 8192, 2048, 8192, L.BF16, 32, 1, 0,
                                            fake, None) == L.ERR_WORKSPACE
    assert L.lib.dpclip_norms_hutch_noalloc(None, fake, 2, 8, 16, 16, L.BF16, 8, 1, 0, fake,
                                            None) == L.ERR_INVALID_ARG


@pytest.mark.gpu
@pytest.mark.parametrize("case", ["bf16", "f32", "up_proj"])
def test_noalloc_matches_workspace_entry_point(L, case):
    from dp_sgd_clipping_gb300 import api
    if case == "bf16":
        wl = W.Workload(130, "noalloc_bf16", 3, 300, 200, 328, "bf16", 1e-2, 1.0, 1.0, 32, ())
    elif case == "f32":
        wl = W.get(1)
    else:
        wl = W.get(4)          # the up_proj workload (2.5 MiB of scratch)
    A, G = to_dev(W.make_inputs(wl))
    dt = L.BF16 if wl.dtype == "bf16" else L.F32
    stream = torch.cuda.current_stream().cuda_stream
    for offset in (0, 7):    # two calls in a row on the shared scratch
        got = _noalloc(L, A, G, dt, wl.k, wl.seed, offset)
        # no bounded wait expired on the device during that call
        assert L.lib.dpclip_noalloc_status(stream) == L.OK
        ref = api.norms_hutch(A, G, wl.k, wl.seed, offset)
        torch.cuda.synchronize()
        assert np.all(np.isfinite(host(got)))
        # the same kernels on the same inputs in the same order: the same bits
        assert torch.equal(got, ref), f"noalloc vs workspace entry point, offset {offset}"
