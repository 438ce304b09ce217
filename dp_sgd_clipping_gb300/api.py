"""Torch-facing wrappers of the C-ABI.

Argument marshalling only: tensors are checked for device, dtype and
contiguity, a workspace is taken from the PyTorch caching allocator (or the
caller's), and the C entry point is called on the current CUDA stream.  Every
step of the computation runs in libdpclip's kernels.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib as L

__all__ = ["norms_exact", "norms_hutch", "norms_hutchpp", "clipped_noisy_grad", "clip_scales",
           "norms_direct_store", "stored_clipped_noisy_grad", "StoredGradients",
           "bias_grads", "clipped_noisy_bias_grad", "SGDUpdate", "FiberAdamW", "fiber_step",
           "philox_normal", "philox_rademacher", "workspace_bytes", "workspace_status",
           "selftest_wait_timeout"]

_DT = {torch.float32: L.F32, torch.bfloat16: L.BF16}


def _stream(stream=None) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _check_pair(A: torch.Tensor, G: torch.Tensor):
    if not (A.is_cuda and G.is_cuda):
        raise ValueError("A and G must be CUDA tensors")
    if A.dtype != G.dtype or A.dtype not in _DT:
        raise ValueError("A and G must both be float32 or both bfloat16")
    if A.dim() != 3 or G.dim() != 3 or A.shape[:2] != G.shape[:2]:
        raise ValueError("A must be [B, T, d] and G [B, T, p]")
    if not (A.is_contiguous() and G.is_contiguous()):
        raise ValueError("A and G must be contiguous")
    B, T, d = A.shape
    return B, T, d, G.shape[2], _DT[A.dtype]


def workspace_bytes(op: int, B: int, T: int, d: int, p: int, dtype: int, param: int) -> int:
    return L.workspace_size(op, B, T, d, p, dtype, param)


def _workspace(nbytes: int, device, ws):
    if ws is None:
        return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
    if ws.numel() * ws.element_size() < nbytes:
        raise ValueError(f"workspace too small: {ws.numel() * ws.element_size()} < {nbytes}")
    return ws


def norms_exact(A, G, method: int = L.EXACT_AUTO, out=None, ws=None, stream=None):
    B, T, d, p, dt = _check_pair(A, G)
    nb = workspace_bytes(L.OP_NORMS_EXACT, B, T, d, p, dt, method)
    ws = _workspace(nb, A.device, ws)
    out = torch.empty(B, dtype=torch.float32, device=A.device) if out is None else out
    L.check("dpclip_norms_exact", L.lib.dpclip_norms_exact(
        A.data_ptr(), G.data_ptr(), B, T, d, p, dt, method, out.data_ptr(), ws.data_ptr(),
        ws.numel() * ws.element_size(), _stream(stream)))
    return out


def norms_hutch(A, G, k: int, seed: int, offset: int = 0, out=None, ws=None, stream=None,
                probe: str = "gaussian"):
    B, T, d, p, dt = _check_pair(A, G)
    nb = workspace_bytes(L.OP_NORMS_HUTCH, B, T, d, p, dt, k)
    ws = _workspace(nb, A.device, ws)
    out = torch.empty(B, dtype=torch.float32, device=A.device) if out is None else out
    L.check("dpclip_norms_hutch_ex", L.lib.dpclip_norms_hutch_ex(
        A.data_ptr(), G.data_ptr(), B, T, d, p, dt, k, L.PROBES[probe], seed, offset,
        out.data_ptr(), ws.data_ptr(), ws.numel() * ws.element_size(), _stream(stream)))
    return out


def norms_hutchpp(A, G, k: int, seed: int, offset: int = 0, out=None, ws=None, stream=None,
                  probe: str = "gaussian"):
    B, T, d, p, dt = _check_pair(A, G)
    nb = workspace_bytes(L.OP_NORMS_HUTCHPP, B, T, d, p, dt, k)
    ws = _workspace(nb, A.device, ws)
    out = torch.empty(B, dtype=torch.float32, device=A.device) if out is None else out
    L.check("dpclip_norms_hutchpp_ex", L.lib.dpclip_norms_hutchpp_ex(
        A.data_ptr(), G.data_ptr(), B, T, d, p, dt, k, L.PROBES[probe], seed, offset,
        out.data_ptr(), ws.data_ptr(), ws.numel() * ws.element_size(), _stream(stream)))
    return out


class SGDUpdate:
    """A parameter update fused into a gradient call: param -= (lr / denom) g,
    in place.  param is the layer's fp32 tensor in the gradient's layout
    ([d, p] weights or [p] bias); denom is the lot size L of the average (its
    expectation for Poisson-sampled lots).  store_grad=False skips writing g."""

    def __init__(self, param, lr: float, denom: float, store_grad: bool = True):
        if param.dtype != torch.float32 or not param.is_cuda or not param.is_contiguous():
            raise ValueError("param must be a contiguous CUDA float32 tensor")
        self.param, self.lr, self.denom, self.store_grad = param, lr, denom, store_grad

    def _c(self):
        return L.SgdUpdate(self.param.data_ptr(), float(self.lr), float(self.denom),
                           int(bool(self.store_grad)))


class FiberAdamW:
    """FIBER optimizer state of one parameter tensor and its hyper-parameters
    (dpclip_fiber_adamw): the innovation filter (filt, resid) and AdamW moments
    (m, v) start at zero; `step` advances by one on every call that applies
    the step.  noise_var is the DP noise variance per coordinate of g = D / L,
    (sigma C / L)^2 for this library's noisy sum."""

    def __init__(self, param, lr: float, denom: float, noise_var: float, omega: float = 0.5,
                 beta1: float = 0.9, beta2: float = 0.999, eps: float = 1e-8, eps_v: float = 1e-12,
                 weight_decay: float = 0.0):
        if param.dtype != torch.float32 or not param.is_cuda or not param.is_contiguous():
            raise ValueError("param must be a contiguous CUDA float32 tensor")
        self.param = param
        self.filt, self.resid, self.m, self.v = (torch.zeros_like(param) for _ in range(4))
        self.lr, self.denom, self.noise_var, self.omega = lr, denom, noise_var, omega
        self.beta1, self.beta2, self.eps, self.eps_v, self.weight_decay = (beta1, beta2, eps, eps_v,
                                                                          weight_decay)
        self.step = 0

    def _c(self):
        self.step += 1
        return L.FiberAdamW(self.param.data_ptr(), self.filt.data_ptr(), self.resid.data_ptr(),
                            self.m.data_ptr(), self.v.data_ptr(), float(self.lr), float(self.beta1),
                            float(self.beta2), float(self.eps), float(self.eps_v),
                            float(self.weight_decay), float(self.omega), float(self.noise_var),
                            float(self.denom), int(self.step))


def fiber_step(grad, opt: FiberAdamW, stream=None):
    """One FIBER step of `opt` from a gradient already formed (fp32, param's shape)."""
    L.check("dpclip_fiber_adamw_step", L.lib.dpclip_fiber_adamw_step(
        grad.data_ptr(), grad.numel(), ctypes.pointer(opt._c()), _stream(stream)))


def _upd(update):
    return None if update is None else ctypes.pointer(update._c())


def clipped_noisy_grad(A, G, sqnorms, C: float, sigma: float, seed: int, offset: int = 0,
                       grad=None, scales=None, clipped=None, ws=None, stream=None,
                       want_scales: bool = True, update: SGDUpdate = None,
                       fiber: FiberAdamW = None, store_grad: bool = True):
    """Returns (grad [d, p] fp32, scales [B] fp32, clipped [B] uint8); with
    `update` (an SGD step) or `fiber` (a FIBER step), also applies it.  A lot
    of B = 0 samples ([0, T, d] tensors) gives the noise alone."""
    B, T, d, p, dt = _check_pair(A, G)
    if B > 0 and (sqnorms.dtype != torch.float32 or sqnorms.numel() != B or not sqnorms.is_cuda):
        raise ValueError("sqnorms must be a CUDA float32 tensor of B entries")
    nb = workspace_bytes(L.OP_CLIPPED_NOISY_GRAD, max(B, 1), T, d, p, dt, 0)
    ws = _workspace(nb, A.device, ws)
    # the GEMM path writes the gradient before a FIBER step, so it always stores it
    wants = update.store_grad if update is not None else True
    if grad is None and (wants or dt == L.F32):
        grad = torch.empty(d, p, dtype=torch.float32, device=A.device)
    if want_scales:
        scales = torch.empty(B, dtype=torch.float32, device=A.device) if scales is None else scales
        clipped = torch.empty(B, dtype=torch.uint8, device=A.device) if clipped is None else clipped
    if fiber is not None:
        L.check("dpclip_clipped_noisy_grad_fiber", L.lib.dpclip_clipped_noisy_grad_fiber(
            A.data_ptr() if B else None, G.data_ptr() if B else None, B, T, d, p, dt,
            sqnorms.data_ptr() if B else None, float(C), float(sigma), seed, offset,
            grad.data_ptr() if grad is not None else None,
            scales.data_ptr() if scales is not None and B else None,
            clipped.data_ptr() if clipped is not None and B else None,
            ctypes.pointer(fiber._c()), ws.data_ptr(), ws.numel() * ws.element_size(),
            _stream(stream)))
        return grad, scales, clipped
    L.check("dpclip_clipped_noisy_grad_ex", L.lib.dpclip_clipped_noisy_grad_ex(
        A.data_ptr() if B else None, G.data_ptr() if B else None, B, T, d, p, dt,
        sqnorms.data_ptr() if B else None, float(C), float(sigma), seed, offset,
        grad.data_ptr() if grad is not None else None,
        scales.data_ptr() if scales is not None and B else None,
        clipped.data_ptr() if clipped is not None and B else None, _upd(update), ws.data_ptr(),
        ws.numel() * ws.element_size(), _stream(stream)))
    return grad, scales, clipped


class StoredGradients:
    """The workspace of a norms_direct_store call: it holds the per-sample
    gradients that stored_clipped_noisy_grad reads.  Keep it alive (and
    unchanged) until that call has been enqueued."""

    def __init__(self, ws, B: int, d: int, p: int):
        self.ws, self.B, self.d, self.p = ws, B, d, p


def norms_direct_store(A, G, sqnorms=None, accumulate: bool = False, ws=None, stream=None):
    """Exact per-sample squared norms (direct method), keeping every A_i^T G_i.

    Returns (sqnorms, StoredGradients).  With accumulate=True the norms are
    added to `sqnorms` (summing the layers of a model)."""
    B, T, d, p, dt = _check_pair(A, G)
    nb = workspace_bytes(L.OP_STORED_DIRECT, B, T, d, p, dt, 0)
    ws = _workspace(nb, A.device, ws)
    if sqnorms is None:
        if accumulate:
            raise ValueError("accumulate needs the sqnorms tensor to add to")
        sqnorms = torch.empty(B, dtype=torch.float32, device=A.device)
    L.check("dpclip_norms_direct_store", L.lib.dpclip_norms_direct_store(
        A.data_ptr(), G.data_ptr(), B, T, d, p, dt, int(bool(accumulate)), sqnorms.data_ptr(),
        ws.data_ptr(), ws.numel() * ws.element_size(), _stream(stream)))
    return sqnorms, StoredGradients(ws, B, d, p)


def stored_clipped_noisy_grad(stored: StoredGradients, sqnorms, C: float, sigma: float, seed: int,
                              offset: int = 0, grad=None, scales=None, clipped=None, stream=None,
                              want_scales: bool = True, update: SGDUpdate = None,
                              fiber: FiberAdamW = None, store_grad: bool = True):
    """clipped_noisy_grad from the per-sample gradients kept by norms_direct_store.

    Returns (grad [d, p] fp32, scales [B] fp32, clipped [B] uint8)."""
    B, d, p, ws = stored.B, stored.d, stored.p, stored.ws
    if sqnorms.dtype != torch.float32 or sqnorms.numel() != B or not sqnorms.is_cuda:
        raise ValueError("sqnorms must be a CUDA float32 tensor of B entries")
    wants = update.store_grad if update is not None else (store_grad if fiber is not None else True)
    if grad is None and wants:
        grad = torch.empty(d, p, dtype=torch.float32, device=ws.device)
    if want_scales:
        scales = torch.empty(B, dtype=torch.float32, device=ws.device) if scales is None else scales
        clipped = torch.empty(B, dtype=torch.uint8, device=ws.device) if clipped is None else clipped
    if fiber is not None:
        L.check("dpclip_stored_clipped_noisy_grad_fiber",
                L.lib.dpclip_stored_clipped_noisy_grad_fiber(
                    B, d, p, sqnorms.data_ptr(), float(C), float(sigma), seed, offset,
                    grad.data_ptr() if grad is not None else None,
                    scales.data_ptr() if scales is not None else None,
                    clipped.data_ptr() if clipped is not None else None,
                    ctypes.pointer(fiber._c()), ws.data_ptr(), ws.numel() * ws.element_size(),
                    _stream(stream)))
        return grad, scales, clipped
    L.check("dpclip_stored_clipped_noisy_grad_ex", L.lib.dpclip_stored_clipped_noisy_grad_ex(
        B, d, p, sqnorms.data_ptr(), float(C), float(sigma), seed, offset,
        grad.data_ptr() if grad is not None else None,
        scales.data_ptr() if scales is not None else None,
        clipped.data_ptr() if clipped is not None else None, _upd(update), ws.data_ptr(),
        ws.numel() * ws.element_size(), _stream(stream)))
    return grad, scales, clipped


def bias_grads(G, sqnorms=None, accumulate: bool = False, want_grads: bool = True, ws=None,
               stream=None):
    """Per-sample bias gradients b_i = sum_t G_i[t, :] and their squared norms.

    Returns (sqnorms [B], bias_grads [B, p] or None).  accumulate=True adds
    ||b_i||^2 to the given sqnorms (e.g. the weights' norms of the layer)."""
    if not G.is_cuda or G.dim() != 3 or G.dtype not in _DT or not G.is_contiguous():
        raise ValueError("G must be a contiguous CUDA [B, T, p] float32 or bfloat16 tensor")
    B, T, p = G.shape
    nb = workspace_bytes(L.OP_BIAS, B, T, 0, p, _DT[G.dtype], 0)
    ws = _workspace(nb, G.device, ws)
    if sqnorms is None:
        if accumulate:
            raise ValueError("accumulate needs the sqnorms tensor to add to")
        sqnorms = torch.empty(B, dtype=torch.float32, device=G.device)
    bg = torch.empty(B, p, dtype=torch.float32, device=G.device) if want_grads else None
    L.check("dpclip_bias_grads", L.lib.dpclip_bias_grads(
        G.data_ptr(), B, T, p, _DT[G.dtype], int(bool(accumulate)), sqnorms.data_ptr(),
        bg.data_ptr() if bg is not None else None, ws.data_ptr(), ws.numel() * ws.element_size(),
        _stream(stream)))
    return sqnorms, bg


def clipped_noisy_bias_grad(bias_grads, sqnorms, C: float, sigma: float, seed: int, offset: int = 0,
                            out=None, stream=None, update: SGDUpdate = None,
                            fiber: FiberAdamW = None, store_grad: bool = True):
    """sum_i s_i b_i + sigma C z (z: Philox stream 4), fp32 [p]; with
    `update` or `fiber`, also applies it.  bias_grads of shape [0, p]: the
    noise alone."""
    B, p = bias_grads.shape
    wants = update.store_grad if update is not None else (store_grad if fiber is not None else True)
    if out is None and wants:
        out = torch.empty(p, dtype=torch.float32, device=bias_grads.device)
    if fiber is not None:
        L.check("dpclip_clipped_noisy_bias_grad_fiber", L.lib.dpclip_clipped_noisy_bias_grad_fiber(
            bias_grads.data_ptr() if B else None, B, p, sqnorms.data_ptr() if B else None,
            float(C), float(sigma), seed, offset, out.data_ptr() if out is not None else None,
            ctypes.pointer(fiber._c()), _stream(stream)))
        return out
    L.check("dpclip_clipped_noisy_bias_grad_ex", L.lib.dpclip_clipped_noisy_bias_grad_ex(
        bias_grads.data_ptr() if B else None, B, p, sqnorms.data_ptr() if B else None, float(C),
        float(sigma), seed, offset, out.data_ptr() if out is not None else None, _upd(update),
        _stream(stream)))
    return out


def clip_scales(sqnorms, C: float, stream=None):
    B = sqnorms.numel()
    scales = torch.empty(B, dtype=torch.float32, device=sqnorms.device)
    clipped = torch.empty(B, dtype=torch.uint8, device=sqnorms.device)
    L.check("dpclip_clip_scales", L.lib.dpclip_clip_scales(
        sqnorms.data_ptr(), B, float(C), scales.data_ptr(), clipped.data_ptr(), _stream(stream)))
    return scales, clipped


def philox_normal(n: int, seed: int, stream_id: int, offset: int = 0, dtype=torch.float32,
                  device="cuda", stream=None):
    out = torch.empty(n, dtype=dtype, device=device)
    L.check("dpclip_philox_normal", L.lib.dpclip_philox_normal(
        out.data_ptr(), n, _DT[dtype], seed, stream_id, offset, _stream(stream)))
    return out


def philox_rademacher(n: int, seed: int, stream_id: int, offset: int = 0, dtype=torch.float32,
                      device="cuda", stream=None):
    out = torch.empty(n, dtype=dtype, device=device)
    L.check("dpclip_philox_rademacher", L.lib.dpclip_philox_rademacher(
        out.data_ptr(), n, _DT[dtype], seed, stream_id, offset, _stream(stream)))
    return out


def workspace_status(ws, stream=None) -> int:
    return L.lib.dpclip_workspace_status(ws.data_ptr(), _stream(stream))


def selftest_wait_timeout(ws, timeout_us: int, stream=None) -> None:
    L.check("dpclip_selftest_wait_timeout", L.lib.dpclip_selftest_wait_timeout(
        ws.data_ptr(), ws.numel() * ws.element_size(), timeout_us, _stream(stream)))
