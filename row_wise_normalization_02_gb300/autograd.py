"""PyTorch training functions over the C ABI.

Forward and backward both run in this library's kernels; PyTorch allocates
the outputs, the tensors saved for the backward and the backward's
workspace, and supplies the current stream.

    y = rms_norm(x, gamma, eps)
    y, h = fused_add_rms_norm(x, residual, gamma, eps)     # h = residual + x
    y = layer_norm(x, gamma, beta, eps)                    # beta may be None

Rows are the last dimension of x (contiguous, on a CUDA device); x and the
weights are bf16 or float32, and bf16 activations may take float32 weights.
The weight gradients come out of the kernels in float32 (the fused add
returns dgamma in the weight dtype, rounded once by its kernel); autograd
casts a float32 gradient to a bf16 weight's dtype.

fused_add_rms_norm is out of place: h is a new tensor (the residual is
copied into it and the kernel adds x over the copy), so that the h saved for
the backward is never modified by the next layer.  The C ABI's
rmsnorm_fused_add_fwd, which writes h over the residual itself, avoids that
copy where no backward is needed.
"""
from __future__ import annotations

import torch

from . import (layernorm_bwd, layernorm_bwd_workspace_size, layernorm_fwd, rmsnorm_bwd,
               rmsnorm_bwd_workspace_size, rmsnorm_fused_add_bwd, rmsnorm_fused_add_fwd,
               rmsnorm_fwd)

__all__ = ["rms_norm", "fused_add_rms_norm", "layer_norm"]

_DT = {torch.bfloat16: "bf16", torch.float32: "f32"}


def _dt(t: torch.Tensor) -> str:
    try:
        return _DT[t.dtype]
    except KeyError:
        raise TypeError(f"unsupported dtype {t.dtype}: bf16 or float32") from None


def _rows(x: torch.Tensor, *weights):
    if not x.is_cuda or not x.is_contiguous() or x.dim() < 1:
        raise ValueError("x must be a contiguous CUDA tensor with rows in its last dimension")
    N = x.shape[-1]
    for w in weights:
        if w is not None and (w.shape != (N,) or not w.is_contiguous() or w.device != x.device):
            raise ValueError(f"weights must be contiguous vectors of {N} on {x.device}")
    return (x.numel() // N if N else 0), N


def _stream(device) -> int:
    """The current stream of x's device: the C ABI launches on the current
    device, so every call below also makes x's device current."""
    return torch.cuda.current_stream(device).cuda_stream


def _workspace(nbytes: int, device) -> torch.Tensor:
    return torch.empty(max(nbytes, 16), dtype=torch.uint8, device=device)


class _RMSNorm(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, gamma, eps):
        M, N = _rows(x, gamma)
        y = torch.empty_like(x)
        rstd = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
        with torch.cuda.device(x.device):
            rmsnorm_fwd(x, gamma, y, rstd, M, N, eps, _dt(x), _dt(gamma), _stream(x.device))
        ctx.save_for_backward(x, gamma, rstd)
        ctx.eps = eps
        return y

    @staticmethod
    def backward(ctx, dy):
        x, gamma, rstd = ctx.saved_tensors
        M, N = _rows(x)
        dy = dy.contiguous()
        dx = torch.empty_like(x)
        dgamma, ws, nbytes = None, None, 0
        if ctx.needs_input_grad[1]:
            dgamma = torch.empty(N, dtype=torch.float32, device=x.device)
            nbytes = rmsnorm_bwd_workspace_size(M, N, _dt(x), _dt(gamma), x.device.index)
            ws = _workspace(nbytes, x.device)
        with torch.cuda.device(x.device):
            rmsnorm_bwd(dy, x, rstd, gamma, dx, dgamma, ws, nbytes, M, N, ctx.eps, _dt(x),
                        _dt(gamma), _stream(x.device))
        return dx, dgamma, None


class _FusedAddRMSNorm(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, residual, gamma, eps):
        M, N = _rows(x, gamma)
        if residual.shape != x.shape or residual.dtype != x.dtype:
            raise ValueError("residual must have the shape and dtype of x")
        if not residual.is_cuda or residual.device != x.device:
            raise ValueError(f"residual must be on x's device ({x.device})")
        h = residual.contiguous().clone()
        y = torch.empty_like(x)
        rstd = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
        with torch.cuda.device(x.device):
            rmsnorm_fused_add_fwd(x, h, gamma, y, rstd, M, N, eps, _dt(x), _dt(gamma),
                                  _stream(x.device))
        ctx.save_for_backward(h, gamma, rstd)
        ctx.eps = eps
        return y, h

    @staticmethod
    def backward(ctx, dy, dh):
        h, gamma, rstd = ctx.saved_tensors
        M, N = _rows(h)
        dy = dy.contiguous()
        # the gradient reaching h along the residual path; the kernel writes
        # dh_total = dx_norm + dh over it (the gradient of both x and residual)
        dres = dh.contiguous().clone()
        dgamma, ws, nbytes = None, None, 0
        if ctx.needs_input_grad[2]:
            dgamma = torch.empty(N, dtype=gamma.dtype, device=h.device)
            nbytes = rmsnorm_bwd_workspace_size(M, N, _dt(h), _dt(gamma), h.device.index)
            ws = _workspace(nbytes, h.device)
        with torch.cuda.device(h.device):
            rmsnorm_fused_add_bwd(dy, h, rstd, gamma, dres, dgamma, _dt(gamma), ws, nbytes, M,
                                  N, ctx.eps, _dt(h), _dt(gamma), _stream(h.device))
        return dres, dres, dgamma, None


class _LayerNorm(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, gamma, beta, eps):
        M, N = _rows(x, gamma, beta)
        y = torch.empty_like(x)
        mean = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
        rstd = torch.empty_like(mean)
        with torch.cuda.device(x.device):
            layernorm_fwd(x, gamma, beta, y, mean, rstd, M, N, eps, _dt(x), _dt(gamma),
                          _stream(x.device))
        ctx.save_for_backward(x, gamma, mean, rstd)
        ctx.eps = eps
        ctx.has_beta = beta is not None
        return y

    @staticmethod
    def backward(ctx, dy):
        x, gamma, mean, rstd = ctx.saved_tensors
        M, N = _rows(x)
        dy = dy.contiguous()
        dx = torch.empty_like(x)
        want_g = ctx.needs_input_grad[1]
        want_b = ctx.has_beta and ctx.needs_input_grad[2]
        dgamma = torch.empty(N, dtype=torch.float32, device=x.device) if want_g else None
        dbeta = torch.empty(N, dtype=torch.float32, device=x.device) if want_b else None
        ws, nbytes = None, 0
        if want_g or want_b:
            nbytes = layernorm_bwd_workspace_size(M, N, _dt(x), _dt(gamma), x.device.index)
            ws = _workspace(nbytes, x.device)
        with torch.cuda.device(x.device):
            layernorm_bwd(dy, x, mean, rstd, gamma, dx, dgamma, dbeta, ws, nbytes, M, N,
                          ctx.eps, _dt(x), _dt(gamma), _stream(x.device))
        return dx, dgamma, dbeta, None


def rms_norm(x: torch.Tensor, gamma: torch.Tensor, eps: float = 1e-6) -> torch.Tensor:
    """y = x / sqrt(mean(x^2) + eps) * gamma over the last dimension."""
    return _RMSNorm.apply(x, gamma, float(eps))


def fused_add_rms_norm(x: torch.Tensor, residual: torch.Tensor, gamma: torch.Tensor,
                       eps: float = 1e-6):
    """h = residual + x (rounded to x's dtype) and y = rms_norm(h, gamma, eps);
    returns (y, h), h a new tensor."""
    return _FusedAddRMSNorm.apply(x, residual, gamma, float(eps))


def layer_norm(x: torch.Tensor, gamma: torch.Tensor, beta: torch.Tensor | None = None,
               eps: float = 1e-5) -> torch.Tensor:
    """y = (x - mean) / sqrt(var + eps) * gamma + beta over the last dimension."""
    return _LayerNorm.apply(x, gamma, beta, float(eps))
