"""A decoder block's MLP half as one chain of launches on one stream, with no
synchronisation between them: residual add + RMSNorm, the gate/up projections
with SwiGLU in the GEMM epilogue, the down projection (torch), the next
residual add + RMSNorm; then the training direction's element-wise pieces.
Every library kernel lets the next launch start early and waits for its
predecessor before reading, so each step must see the previous step's full
output: checked against a plain PyTorch fp32 composition of the same math,
and against the same chain with a synchronisation after every step (identical
bits: every step is deterministic)."""
import pytest
import torch
import torch.nn.functional as F

import glu_activation_mlps_gb300 as glu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    glu.build()
    glu.lib()


def chain(x, res, g1, wg, wu, wd, g2, sync):
    step = torch.cuda.synchronize if sync else (lambda: None)
    h1, y1 = glu.add_rmsnorm(x, res, g1, 1e-5)
    step()
    act = glu.gemm_fwd(y1, wg, wu, act="silu")
    step()
    out = act @ wd.t()
    step()
    h2, y2 = glu.add_rmsnorm(out, h1, g2, 1e-5)
    step()
    # backward pieces of the activation on the gate/up outputs, in place
    a, b = y1 @ wg.t(), y1 @ wu.t()
    dy = torch.ones_like(a) * 0.01
    da, db = glu.bwd(dy, a, b, act="silu", inplace=True)
    step()
    torch.cuda.synchronize()
    return h1, y1, act, h2, y2, da, db


@pytest.mark.parametrize("tokens", [48, 1000])
def test_decoder_mlp_chain(tokens):
    torch.manual_seed(5)
    H, I = 1024, 2816
    dev, dt = "cuda", torch.bfloat16
    x = torch.randn(tokens, H, device=dev).to(dt)
    res = (4 * torch.randn(tokens, H, device=dev)).to(dt)
    g1 = (1 + 0.1 * torch.randn(H, device=dev)).to(dt)
    g2 = (1 + 0.1 * torch.randn(H, device=dev)).to(dt)
    wg = (torch.randn(I, H, device=dev) / H ** 0.5).to(dt)
    wu = (torch.randn(I, H, device=dev) / H ** 0.5).to(dt)
    wd = (torch.randn(H, I, device=dev) / I ** 0.5).to(dt)

    fast = chain(x, res, g1, wg, wu, wd, g2, sync=False)
    slow = chain(x, res, g1, wg, wu, wd, g2, sync=True)
    for f, s_ in zip(fast, slow):
        assert torch.equal(f, s_)

    h1, y1, act, h2, y2, da, db = fast
    # plain PyTorch in fp32 on the same bf16 inputs
    r_h1 = x.float() + res.float()
    r_y1 = F.rms_norm(r_h1, (H,), g1.float(), 1e-5)
    assert torch.equal(h1, r_h1.to(dt))
    assert torch.allclose(y1.float(), r_y1, atol=2e-2, rtol=2e-2)
    gu = y1.float() @ wg.float().t(), y1.float() @ wu.float().t()
    r_act = F.silu(gu[0]) * gu[1]
    assert torch.allclose(act.float(), r_act, atol=2e-2, rtol=2e-2)
    out = act @ wd.t()
    r_h2 = out.float() + h1.float()
    assert torch.equal(h2, r_h2.to(dt))
    assert torch.allclose(y2.float(), F.rms_norm(r_h2, (H,), g2.float(), 1e-5), atol=2e-2, rtol=2e-2)
    a, b = (y1 @ wg.t()).float(), (y1 @ wu.t()).float()
    sg = torch.sigmoid(a)
    assert torch.allclose(da.float(), 0.01 * (a * sg * (1 - sg) + sg) * b, atol=1e-3, rtol=2e-2)
    assert torch.allclose(db.float(), 0.01 * a * sg, atol=1e-3, rtol=2e-2)
    assert glu.glu_wait_timeouts() == 0
