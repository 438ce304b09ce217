"""ctypes loader of libdpclip.so and the raw C-ABI (names as in include/dpclip.h).

Loading needs no GPU; the library refuses to fall back to anything else: if
the shared object is missing the import of this module raises.
"""
from __future__ import annotations

import ctypes
import os

from . import _build

OK = 0
ERR_INVALID_ARG = -1
ERR_UNSUPPORTED = -2
ERR_WORKSPACE = -3
ERR_CUDA = -4
ERR_TIMEOUT = -5

F32 = 0
BF16 = 1

EXACT_AUTO, EXACT_GHOST, EXACT_DIRECT = 0, 1, 2
PROBE_GAUSSIAN, PROBE_RADEMACHER = 0, 1
PROBES = {"gaussian": PROBE_GAUSSIAN, "rademacher": PROBE_RADEMACHER}
OP_NORMS_EXACT, OP_NORMS_HUTCH, OP_NORMS_HUTCHPP, OP_CLIPPED_NOISY_GRAD = 0, 1, 2, 3
OP_STORED_DIRECT = 4
OP_BIAS = 5
HUTCH_MAX_K = 32
HUTCHPP_MAX_K = 48
NOALLOC_SCRATCH_BYTES = 16 << 20

_c = ctypes
_vp, _i, _u64, _u32, _i64, _f = _c.c_void_p, _c.c_int, _c.c_uint64, _c.c_uint32, _c.c_int64, _c.c_float
_sz = _c.c_size_t



class SgdUpdate(_c.Structure):
    """struct dpclip_sgd_update: param -= (lr / denom) * g, in place."""
    _fields_ = [("param", _c.c_void_p), ("lr", _c.c_float), ("denom", _c.c_float),
                ("store_grad", _c.c_int)]


_up = _c.POINTER(SgdUpdate)


class FiberAdamW(_c.Structure):
    """struct dpclip_fiber_adamw: the FIBER step's tensors and hyper-parameters."""
    _fields_ = [("param", _c.c_void_p), ("filt", _c.c_void_p), ("resid", _c.c_void_p),
                ("m", _c.c_void_p), ("v", _c.c_void_p), ("lr", _c.c_float),
                ("beta1", _c.c_float), ("beta2", _c.c_float), ("eps", _c.c_float),
                ("eps_v", _c.c_float), ("weight_decay", _c.c_float), ("omega", _c.c_float),
                ("noise_var", _c.c_float), ("denom", _c.c_float), ("step", _c.c_int)]


_fp = _c.POINTER(FiberAdamW)

# symbol -> (restype, argtypes)
SIGNATURES = {
    "dpclip_workspace_size": (_i, [_i, _i, _i, _i, _i, _i, _i, _c.POINTER(_sz)]),
    "dpclip_norms_exact": (_i, [_vp, _vp, _i, _i, _i, _i, _i, _i, _vp, _vp, _sz, _vp]),
    "dpclip_norms_hutch": (_i, [_vp, _vp, _i, _i, _i, _i, _i, _i, _u64, _u64, _vp, _vp, _sz, _vp]),
    "dpclip_norms_hutchpp": (_i, [_vp, _vp, _i, _i, _i, _i, _i, _i, _u64, _u64, _vp, _vp, _sz, _vp]),
    "dpclip_norms_hutch_ex": (_i, [_vp, _vp, _i, _i, _i, _i, _i, _i, _i, _u64, _u64, _vp, _vp, _sz,
                                   _vp]),
    "dpclip_norms_hutchpp_ex": (_i, [_vp, _vp, _i, _i, _i, _i, _i, _i, _i, _u64, _u64, _vp, _vp,
                                     _sz, _vp]),
    "dpclip_philox_rademacher": (_i, [_vp, _i64, _i, _u64, _u32, _u64, _vp]),
    "dpclip_clipped_noisy_grad": (_i, [_vp, _vp, _i, _i, _i, _i, _i, _vp, _f, _f, _u64, _u64,
                                       _vp, _vp, _vp, _vp, _sz, _vp]),
    "dpclip_clip_scales": (_i, [_vp, _i, _f, _vp, _vp, _vp]),
    "dpclip_clipped_noisy_grad_ex": (_i, [_vp, _vp, _i, _i, _i, _i, _i, _vp, _f, _f, _u64, _u64,
                                          _vp, _vp, _vp, _up, _vp, _sz, _vp]),
    "dpclip_stored_clipped_noisy_grad_ex": (_i, [_i, _i, _i, _vp, _f, _f, _u64, _u64, _vp, _vp,
                                                 _vp, _up, _vp, _sz, _vp]),
    "dpclip_clipped_noisy_bias_grad_ex": (_i, [_vp, _i, _i, _vp, _f, _f, _u64, _u64, _vp, _up,
                                               _vp]),
    "dpclip_fiber_adamw_step": (_i, [_vp, _i64, _fp, _vp]),
    "dpclip_clipped_noisy_grad_fiber": (_i, [_vp, _vp, _i, _i, _i, _i, _i, _vp, _f, _f, _u64,
                                             _u64, _vp, _vp, _vp, _fp, _vp, _sz, _vp]),
    "dpclip_stored_clipped_noisy_grad_fiber": (_i, [_i, _i, _i, _vp, _f, _f, _u64, _u64, _vp,
                                                    _vp, _vp, _fp, _vp, _sz, _vp]),
    "dpclip_clipped_noisy_bias_grad_fiber": (_i, [_vp, _i, _i, _vp, _f, _f, _u64, _u64, _vp, _fp,
                                                  _vp]),
    "dpclip_bias_grads": (_i, [_vp, _i, _i, _i, _i, _i, _vp, _vp, _vp, _sz, _vp]),
    "dpclip_clipped_noisy_bias_grad": (_i, [_vp, _i, _i, _vp, _f, _f, _u64, _u64, _vp, _vp]),
    "dpclip_norms_direct_store": (_i, [_vp, _vp, _i, _i, _i, _i, _i, _i, _vp, _vp, _sz, _vp]),
    "dpclip_stored_clipped_noisy_grad": (_i, [_i, _i, _i, _vp, _f, _f, _u64, _u64, _vp, _vp, _vp,
                                              _vp, _sz, _vp]),
    "dpclip_norms_hutch_noalloc": (_i, [_vp, _vp, _i, _i, _i, _i, _i, _i, _u64, _u64, _vp, _vp]),
    "dpclip_noalloc_status": (_i, [_vp]),
    "dpclip_philox_normal": (_i, [_vp, _i64, _i, _u64, _u32, _u64, _vp]),
    "dpclip_workspace_status": (_i, [_vp, _vp]),
    "dpclip_selftest_wait_timeout": (_i, [_vp, _sz, _i, _vp]),
    "dpclip_grad_tail_schedule": (_i, [_i, _i, _i, _i, _c.POINTER(_i), _c.POINTER(_i), _vp, _i,
                                       _c.POINTER(_i), _vp, _i, _c.POINTER(_i)]),
    "dpclip_ghost_schedule": (_i, [_i, _i, _i, _i, _i, _c.POINTER(_i), _c.POINTER(_i),
                                   _c.POINTER(_i), _c.POINTER(_i)]),
    "dpclip_status_string": (_c.c_char_p, [_i]),
    "dpclip_version": (_c.c_char_p, []),
}


class DpclipError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn} failed: {msg} (status {status})")
        self.status = status


def lib_path() -> str:
    return _build.LIB


def _load():
    path = lib_path()
    if not os.path.exists(path):
        raise ImportError(
            f"libdpclip.so is not built ({path}); run "
            "`python -c 'import __graft_entry__ as g; g.build()'` first")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


def grad_tail_schedule(pairs: int, ntiles: int, B: int, tblocks: int):
    """The gradient's tail schedule (host only): (waves, ntail, segments,
    contributions), segments as rows (pair, tail tile, t0, t1, slot) and
    contributions as rows (tail tile, slot)."""
    import numpy as np
    waves, ntail, ns, nc = _c.c_int(), _c.c_int(), _c.c_int(), _c.c_int()
    seg_cap = contrib_cap = 0
    while True:
        segs = np.zeros((max(seg_cap, 1), 5), dtype=np.int64)
        contrib = np.zeros((max(contrib_cap, 1), 2), dtype=np.int64)
        st = lib.dpclip_grad_tail_schedule(pairs, ntiles, B, tblocks, _c.byref(waves),
                                           _c.byref(ntail), segs.ctypes.data, seg_cap,
                                           _c.byref(ns), contrib.ctypes.data, contrib_cap,
                                           _c.byref(nc))
        if st != 0:
            raise DpclipError("dpclip_grad_tail_schedule", st, status_string(st))
        if ns.value <= seg_cap and nc.value <= contrib_cap:
            return waves.value, ntail.value, segs[:ns.value], contrib[:nc.value]
        seg_cap, contrib_cap = ns.value, nc.value


def ghost_schedule(pairs: int, B: int, T: int, d: int, p: int):
    """The ghost form's work split (host only): (nfull, tail_split,
    pb_per_split, tail_shared)."""
    out = [_c.c_int() for _ in range(4)]
    st = lib.dpclip_ghost_schedule(pairs, B, T, d, p, *[_c.byref(o) for o in out])
    if st != 0:
        raise DpclipError("dpclip_ghost_schedule", st, status_string(st))
    return tuple(o.value for o in out)


def status_string(status: int) -> str:
    return lib.dpclip_status_string(status).decode()


def check(fn: str, status: int) -> None:
    if status != OK:
        raise DpclipError(fn, status, status_string(status))


def workspace_size(op: int, B: int, T: int, d: int, p: int, dtype: int, param: int) -> int:
    n = _sz(0)
    check("dpclip_workspace_size", lib.dpclip_workspace_size(op, B, T, d, p, dtype, param,
                                                             ctypes.byref(n)))
    return n.value
