"""A third opinion next to the oracle: the same op composed from plain
PyTorch ops on the GPU (its own silu, fp32 throughout, IEEE division, its own
float8_e4m3fn cast), compared with the fused kernel's output.

The two sides compute y = silu(g) * u * w with different silu formulas, so y
may differ in its last bits; everything after y is the same arithmetic (group
absmax, s = amax / 448 with one rounding, RN(y / s), round-to-nearest-even
E4M3). So the fp32 scales agree to a few ulps, almost every code is
identical, and no code is more than one E4M3 step away."""
import pytest
import torch
import torch.nn.functional as F

import activation_fp8_quantization_gb300 as tk
from activation_fp8_quantization_gb300 import workloads as wls

pytestmark = pytest.mark.gpu


def _torch_quant(x, w, H, g):
    T = x.shape[0]
    y = F.silu(x[:, :H].float()) * x[:, H:].float() * w[:, None]
    yg = y.view(T, H // g, g)
    amax = yg.abs().amax(-1)
    s = torch.where(amax == 0, torch.ones_like(amax), amax / 448.0)
    q = (yg / s[..., None]).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
    return q.view(torch.uint8).view(T, H), s


@pytest.mark.parametrize("name", ["moe_T8192_H2048_g128", "ragged_T100003_H3072_g128"])
@pytest.mark.parametrize("kernel", ["rows", "block"])
def test_fused_kernel_agrees_with_a_torch_composition(name, kernel, monkeypatch):
    monkeypatch.setenv("TK_KERNEL", kernel)
    wl = wls.WORKLOADS[name].with_rows(4099)
    x, w = wls.make_inputs(wl, "cuda")
    op = tk.SwigluQuant(wl.H, wl.group, "fp32", "e4m3", True)
    q, s = op(x, w)
    q_t, s_t = _torch_quant(x, w, wl.H, wl.group)
    torch.cuda.synchronize()
    rel = ((s - s_t).abs() / s_t).max().item()
    assert rel < 2.0 ** -20, "scales differ by %g relative" % rel
    same = (q == q_t).float().mean().item()
    assert same > 0.999, "only %.5f of the codes identical" % same
    a = q.view(torch.float8_e4m3fn).float()
    b = q_t.view(torch.float8_e4m3fn).float()
    step = torch.exp2(torch.floor(torch.log2(torch.maximum(a.abs(), b.abs()).clamp_min(2.0 ** -6))) - 3)
    assert ((a - b).abs() <= step).all()
    print(name, kernel, "codes identical %.6f, scales within %.2g relative" % (same, rel))
