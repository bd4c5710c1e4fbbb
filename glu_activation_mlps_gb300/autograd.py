"""PyTorch autograd functions and modules over the C ABI.

The pattern follows "Kernel Profile: SwiGLU (Tier 1 - Element-wise)" (Forward
Pass, Backward Pass, Key Patterns): the forward saves the gate and up
projections a and b and nothing else; the backward recomputes the activation
from a in the kernel, and may write da over a and db over b (the saved tensors)
instead of allocating.  Every computation runs in the library's CUDA kernels;
these classes only marshal tensors.  "Skill: Write a Triton SiLU-Mul (SwiGLU)
Kernel" (Purpose) gives the surrounding MLP, down(act(gate(x)) * up(x)).
"""
from __future__ import annotations

import torch
from torch import nn

from . import add_rmsnorm as _add_rmsnorm
from . import add_rmsnorm_bwd as _add_rmsnorm_bwd
from . import bwd as _bwd
from . import fwd as _fwd
from . import gemm_fwd as _gemm_fwd

ACTS = ("silu", "gelu_erf", "gelu_tanh", "relu")


def _check_act(act: str) -> str:
    if act not in ACTS:
        raise ValueError(f"unknown activation {act!r}; expected one of {ACTS}")
    return act


class GLUFunction(torch.autograd.Function):
    """y = act(a) * b for separate gate and up tensors of one shape.

    With ``inplace_backward`` the backward writes da into a's storage and db
    into b's: a and b must not be used elsewhere after the backward (in an MLP
    they are the gate/up projections' outputs, used only here)."""

    @staticmethod
    def forward(ctx, a, b, act: str = "silu", inplace_backward: bool = False):
        y = _fwd(a, b, act=act)
        ctx.save_for_backward(a, b)
        ctx.act = act
        ctx.inplace_backward = inplace_backward
        return y

    @staticmethod
    def backward(ctx, dy):
        a, b = ctx.saved_tensors
        if dy.stride(-1) != 1:
            dy = dy.contiguous()
        da, db = _bwd(dy, a, b, act=ctx.act, inplace=ctx.inplace_backward)
        return da, db, None, None


class GLUConcatFunction(torch.autograd.Function):
    """y = act(x[..., :I]) * x[..., I:] for one tensor holding [gate | up] per
    row (the output of a fused gate/up projection); the gradient is dx = [da | db]."""

    @staticmethod
    def forward(ctx, x, act: str = "silu", inplace_backward: bool = False):
        y = _fwd(x, layout="concat", act=act)
        ctx.save_for_backward(x)
        ctx.act = act
        ctx.inplace_backward = inplace_backward
        return y

    @staticmethod
    def backward(ctx, dy):
        (x,) = ctx.saved_tensors
        if dy.stride(-1) != 1:
            dy = dy.contiguous()
        dx = _bwd(dy, x, layout="concat", act=ctx.act, inplace=ctx.inplace_backward)
        return dx, None, None


def glu(a, b=None, act: str = "silu", inplace_backward: bool = False):
    """Functional form: glu(a, b) for separate tensors, glu(x) for [gate | up]."""
    _check_act(act)
    if b is None:
        return GLUConcatFunction.apply(a, act, inplace_backward)
    return GLUFunction.apply(a, b, act, inplace_backward)


class GLU(nn.Module):
    """The gated activation as a module: forward(a, b) or forward(x) with x = [gate | up]."""

    def __init__(self, act: str = "silu", inplace_backward: bool = False):
        super().__init__()
        self.act = _check_act(act)
        self.inplace_backward = inplace_backward

    def forward(self, a, b=None):
        return glu(a, b, self.act, self.inplace_backward)

    def extra_repr(self):
        return f"act={self.act}, inplace_backward={self.inplace_backward}"


def _gemm_ready(x, w) -> bool:
    """Inputs the tensor-core GEMM with the activation in its epilogue takes:
    f16/bf16 CUDA tensors of one dtype, rows contiguous, 16-byte aligned bases
    and row strides (the tensor-memory accelerator's rule)."""
    if not (x.is_cuda and x.dtype in (torch.float16, torch.bfloat16) and w.dtype == x.dtype):
        return False
    if x.stride(-1) != 1 or w.stride(-1) != 1 or x.data_ptr() % 16 or w.data_ptr() % 16:
        return False
    if (w.stride(0) * w.element_size()) % 16:
        return False
    if x.dim() > 1 and (x.stride(-2) * x.element_size()) % 16:
        return False
    return True


class GatedMLP(nn.Module):
    """down(act(x W_gate^T) * (x W_up^T)) with the projections as torch Linear
    layers (no bias) and the gated activation from the library.  With
    ``fused_gate_up`` the gate and up projections are one Linear of 2 * I
    outputs whose result feeds the [gate | up] layout directly, so no split or
    copy is needed between the projection and the activation.

    Without autograd (inference: torch.no_grad(), or no input or weight that
    requires a gradient) the gate and up projections and the activation run
    as one tensor-core GEMM with the activation in its epilogue (glu_gemm_fwd),
    so the gate and up matrices never reach HBM ("Skill: Write a Triton
    SiLU-Mul (SwiGLU) Kernel", Performance requirements, "Versus epilogue
    fusion").  Training keeps the projections, because the backward needs
    them."""

    def __init__(self, hidden: int, intermediate: int, act: str = "silu", fused_gate_up: bool = True,
                 device=None, dtype=None):
        super().__init__()
        kw = {"device": device, "dtype": dtype, "bias": False}
        self.act = _check_act(act)
        self.fused_gate_up = fused_gate_up
        if fused_gate_up:
            self.gate_up_proj = nn.Linear(hidden, 2 * intermediate, **kw)
        else:
            self.gate_proj = nn.Linear(hidden, intermediate, **kw)
            self.up_proj = nn.Linear(hidden, intermediate, **kw)
        self.down_proj = nn.Linear(intermediate, hidden, **kw)

    def _gate_up_weights(self):
        if self.fused_gate_up:
            w = self.gate_up_proj.weight
            n = w.shape[0] // 2
            return w[:n], w[n:]
        return self.gate_proj.weight, self.up_proj.weight

    def forward(self, x):
        wg, wu = self._gate_up_weights()
        grad = torch.is_grad_enabled() and (x.requires_grad or wg.requires_grad or wu.requires_grad)
        if not grad and _gemm_ready(x, wg) and _gemm_ready(x, wu) and wg.stride(0) == wu.stride(0):
            return self.down_proj(_gemm_fwd(x, wg, wu, act=self.act))
        if self.fused_gate_up:
            h = glu(self.gate_up_proj(x), act=self.act, inplace_backward=True)
        else:
            h = glu(self.gate_proj(x), self.up_proj(x), act=self.act, inplace_backward=True)
        return self.down_proj(h)


class AddRMSNormFunction(torch.autograd.Function):
    """(h, y) = (x + residual, rmsnorm(x + residual) * gamma) in one pass
    ("Skill: Write a Triton Fused Add+RMSNorm Kernel", Purpose; steps 9-10 for
    the backward).  The forward saves h and rstd; the backward sends the same
    gradient to x and to the residual (the norm's gradient plus the gradient
    arriving at h from the residual stream) and accumulates gamma's."""

    @staticmethod
    def forward(ctx, x, residual, gamma, eps: float = 1e-5):
        h, y, rstd = _add_rmsnorm(x, residual, gamma, eps, rstd=True)
        ctx.save_for_backward(h, rstd, gamma)
        return h, y

    @staticmethod
    def backward(ctx, dh, dy):
        h, rstd, gamma = ctx.saved_tensors
        if dy is None:
            dy = torch.zeros_like(h)
        dy = dy if dy.stride(-1) == 1 else dy.contiguous()
        if dh is not None and dh.stride(-1) != 1:
            dh = dh.contiguous()
        want_g = ctx.needs_input_grad[2]
        out = _add_rmsnorm_bwd(dy, h, rstd, gamma, dh=dh, dgamma=True if want_g else None)
        dx, dg = out if want_g else (out, None)
        return dx, dx, (dg.to(gamma.dtype) if dg is not None else None), None


class FusedAddRMSNorm(nn.Module):
    """The residual add + RMSNorm at the end of a decoder sub-block:
    forward(x, residual) -> (h, y), h the next block's residual stream."""

    def __init__(self, hidden: int, eps: float = 1e-5, device=None, dtype=None):
        super().__init__()
        self.eps = eps
        self.weight = nn.Parameter(torch.ones(hidden, device=device, dtype=dtype))

    def forward(self, x, residual):
        return AddRMSNormFunction.apply(x, residual, self.weight, self.eps)

    def extra_repr(self):
        return f"{self.weight.shape[0]}, eps={self.eps}"
