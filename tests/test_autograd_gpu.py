"""The autograd layer: GLUFunction / GLUConcatFunction gradients against the
oracle (bit patterns under the 1-ulp bar), with and without the in-place
backward, a torch fp64 autograd cross-check in f32, and the GatedMLP module
against a plain PyTorch composition with the same weights."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import glu_activation_mlps_gb300 as glu
from glu_activation_mlps_gb300 import autograd as ga
import glu_synth
from helpers import compare, to_bits, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    glu.build()
    glu.lib()
    glu.glu_set_tuning(0, 0, 0, 0, 0)


@pytest.mark.parametrize("inplace", [False, True])
@pytest.mark.parametrize("act", ["silu", "gelu_erf", "gelu_tanh", "relu"])
def test_split_function_gradients_match_oracle(orc, act, inplace):
    dt, shape = "bf16", (3, 37, 1000)
    rng = np.random.default_rng(31)
    a = glu_synth.normal_bits(rng, shape, 2.0, dt)
    b = glu_synth.normal_bits(rng, shape, 1.0, dt)
    dy = glu_synth.normal_bits(rng, shape, 1.0, dt)
    A = to_dev(a, dt).requires_grad_(True)
    B = to_dev(b, dt).requires_grad_(True)
    # a non-leaf copy so that the in-place backward may overwrite it
    A2, B2 = A * 1, B * 1
    y = ga.glu(A2, B2, act=act, inplace_backward=inplace)
    compare(to_bits(y.detach(), dt), orc.fwd(act, dt, a, b), dt, what=f"{act} autograd y")
    y.backward(to_dev(dy, dt))
    da_o, db_o = orc.bwd(act, dt, dy, a, b)
    compare(to_bits(A.grad, dt), da_o, dt, what=f"{act} autograd da")
    compare(to_bits(B.grad, dt), db_o, dt, what=f"{act} autograd db")


def test_concat_function_gradient_matches_oracle(orc):
    dt, rows, cols = "bf16", 50, 1111
    rng = np.random.default_rng(32)
    x = glu_synth.normal_bits(rng, (rows, 2 * cols), 1.5, dt)
    dy = glu_synth.normal_bits(rng, (rows, cols), 1.0, dt)
    for inplace in (False, True):
        X = to_dev(x, dt).requires_grad_(True)
        y = ga.glu(X * 1, act="gelu_tanh", inplace_backward=inplace)
        compare(to_bits(y.detach(), dt), orc.fwd_concat("gelu_tanh", dt, x, cols), dt, what="concat y")
        y.backward(to_dev(dy, dt))
        dx_o = orc.bwd_concat("gelu_tanh", dt, dy, x, cols)
        compare(to_bits(X.grad, dt)[:, :cols], dx_o[:, :cols], dt, what="concat da")
        compare(to_bits(X.grad, dt)[:, cols:], dx_o[:, cols:], dt, what="concat db")


@pytest.mark.parametrize("act", ["silu", "gelu_erf", "gelu_tanh"])
def test_f32_gradients_against_torch_fp64_autograd(act):
    g = torch.Generator(device="cuda").manual_seed(3)
    a = torch.randn(64, 513, device="cuda", generator=g) * 2
    b = torch.randn(64, 513, device="cuda", generator=g)
    dy = torch.randn(64, 513, device="cuda", generator=g)
    A, B = a.clone().requires_grad_(True), b.clone().requires_grad_(True)
    ga.glu(A, B, act=act).backward(dy)
    fn = {"silu": F.silu, "gelu_erf": lambda t: F.gelu(t, approximate="none"),
          "gelu_tanh": lambda t: F.gelu(t, approximate="tanh")}[act]
    A64, B64 = a.double().requires_grad_(True), b.double().requires_grad_(True)
    (fn(A64) * B64).backward(dy.double())
    scale = (dy.double().abs() * (B64.detach().abs() + 1)).max()
    assert (A.grad.double() - A64.grad).abs().max() / scale < 1e-5
    assert (B.grad.double() - B64.grad).abs().max() / scale < 1e-5


@pytest.mark.parametrize("fused", [True, False])
def test_gated_mlp_matches_plain_torch(fused):
    torch.manual_seed(0)
    hidden, inter = 256, 704
    mlp = ga.GatedMLP(hidden, inter, act="silu", fused_gate_up=fused, device="cuda", dtype=torch.bfloat16)
    x = torch.randn(8, 33, hidden, device="cuda", dtype=torch.bfloat16, requires_grad=True)
    y = mlp(x)
    # the same weights through plain PyTorch ops
    if fused:
        wg, wu = mlp.gate_up_proj.weight[:inter], mlp.gate_up_proj.weight[inter:]
    else:
        wg, wu = mlp.gate_proj.weight, mlp.up_proj.weight
    xr = x.detach().clone().requires_grad_(True)
    h = F.silu((xr @ wg.t()).float()) * (xr @ wu.t()).float()
    yr = h.to(torch.bfloat16) @ mlp.down_proj.weight.t()
    assert torch.allclose(y.float(), yr.float(), atol=2e-2, rtol=2e-2)
    gy = torch.randn_like(y)
    y.backward(gy)
    yr.backward(gy)
    assert torch.allclose(x.grad.float(), xr.grad.float(), atol=3e-2, rtol=3e-2)
    assert mlp.down_proj.weight.grad is not None


@pytest.mark.parametrize("act", ["silu", "gelu_tanh"])
@pytest.mark.parametrize("fused", [True, False])
def test_gated_mlp_inference_uses_the_fused_gemm(fused, act):
    """Under torch.no_grad() the module runs glu_gemm_fwd (the last launch is the
    GEMM's) and agrees with its training path on the same weights."""
    torch.manual_seed(1)
    hidden, inter = 512, 1408
    mlp = ga.GatedMLP(hidden, inter, act=act, fused_gate_up=fused, device="cuda", dtype=torch.bfloat16)
    x = torch.randn(3, 70, hidden, device="cuda", dtype=torch.bfloat16)
    y_train = mlp(x.clone().requires_grad_(True)).detach()
    wg, wu = mlp._gate_up_weights()
    with torch.no_grad():
        h = glu.gemm_fwd(x, wg, wu, act=act)
        assert glu.glu_last_launch()["path"] == 3
        y = mlp(x)
    assert torch.equal(y, mlp.down_proj(h).detach())
    assert torch.allclose(y.float(), y_train.float(), atol=2e-2, rtol=2e-2)


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
def test_fused_add_rmsnorm_module_matches_torch_autograd(dt):
    """FusedAddRMSNorm against torch autograd through x + residual and F.rms_norm,
    with gradients arriving at both outputs (y, and h through the residual stream)."""
    if not hasattr(F, "rms_norm"):
        pytest.skip("torch without rms_norm")
    torch.manual_seed(3)
    H = 1536
    mod = ga.FusedAddRMSNorm(H, eps=1e-5, device="cuda", dtype=dt)
    with torch.no_grad():
        mod.weight.copy_(1 + 0.1 * torch.randn(H, device="cuda"))
    x = torch.randn(4, 50, H, device="cuda", dtype=dt, requires_grad=True)
    r = (4 * torch.randn(4, 50, H, device="cuda")).to(dt).requires_grad_(True)
    h, y = mod(x, r)
    gh, gy = torch.randn_like(h), torch.randn_like(y)
    (h * gh).sum().backward(retain_graph=True)
    (y * gy).sum().backward()
    xr = x.detach().double().requires_grad_(True)
    rr = r.detach().double().requires_grad_(True)
    wr = mod.weight.detach().double().requires_grad_(True)
    hr = xr + rr
    yr = F.rms_norm(hr, (H,), wr, 1e-5)
    ((hr * gh.double()).sum() + (yr * gy.double()).sum()).backward()
    tol = 2e-2 if dt == torch.bfloat16 else 1e-4
    assert torch.allclose(y.double(), yr, atol=tol, rtol=tol)
    assert torch.allclose(x.grad.double(), xr.grad, atol=tol, rtol=tol)
    assert torch.allclose(r.grad.double(), rr.grad, atol=tol, rtol=tol)
    assert torch.allclose(mod.weight.grad.double(), wr.grad, atol=tol * 50, rtol=tol)
