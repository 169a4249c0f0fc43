"""The fused op on page-locked host buffers read and written in place by the
kernel (tk_swiglu_quant_run_mapped), through the C ABI: the same codes,
scales and clamp counters as the device call, bit for bit; device pointers
and pageable host memory are refused before anything is launched."""
import numpy as np
import pytest
import torch

import activation_fp8_quantization_gb300 as tk
from activation_fp8_quantization_gb300 import workloads as wls

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("layout", ["row", "col"])
@pytest.mark.parametrize("name,rows", [("moe_T8192_H2048_g128", 3001), ("moe_T32768_H2048_g128_ue8m0_clamp7", 4099),
                                       ("fp4_T65536_H2048_g32_ue8m0_clamp7", 517), ("ragged_T100003_H3072_g128", 1023),
                                       ("per_token_T256_H512", 256)])
def test_mapped_equals_device(name, rows, layout):
    wl = wls.WORKLOADS[name].with_rows(rows)
    count = wl.clamp is not None
    op = tk.SwigluQuant(wl.H, wl.group, wl.scale_fmt, wl.out_fmt, wl.w_dist is not None, wl.clamp, count,
                        scale_layout=layout)
    x, w = wls.make_inputs(wl, "cpu")
    c_dev = torch.zeros(2, dtype=torch.int64, device="cuda") if count else None
    q0, s0 = op(x.cuda(), None if w is None else w.cuda(), clamped_count=c_dev)
    x_h = x.pin_memory()
    w_h = None if w is None else w.pin_memory()
    c_h = torch.zeros(2, dtype=torch.int64).pin_memory() if count else None
    s = torch.cuda.Stream()
    q1, s1 = op.mapped(x_h, w_h, clamped_count=c_h, stream=s)
    s.synchronize()
    torch.cuda.synchronize()
    assert torch.equal(q1, q0.cpu())
    if layout == "row":
        assert torch.equal(s1, s0.cpu())
    else:   # compare the written entries: the column layout's padding rows are not written
        T = wl.T
        G = wl.groups_per_row
        a, b = s1.numpy().reshape(G, -1)[:, :T], s0.cpu().numpy().reshape(G, -1)[:, :T]
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))
    if count:
        assert c_h.tolist() == c_dev.cpu().tolist()


def test_mapped_refuses_device_and_pageable_memory():
    H, T = 512, 64
    op = tk.SwigluQuant(H, 128, "fp32", "e4m3", True)
    x_d = torch.zeros((T, 2 * H), dtype=torch.bfloat16, device="cuda")
    w_h = torch.ones(T).pin_memory()
    q_h = torch.empty((T, H), dtype=torch.uint8).pin_memory()
    s_h = torch.empty((T, H // 128), dtype=torch.float32).pin_memory()
    with pytest.raises(tk.TkError) as e:   # device memory is not host memory
        tk.tk_swiglu_quant_run_mapped(op.plan, T, x_d, w_h, q_h, s_h, None, None)
    assert e.value.status == 1
    raw = np.zeros(T * 2 * H * 2 + 256, np.uint8)   # pageable, with a 256-byte-aligned start inside
    start = raw.ctypes.data + (-raw.ctypes.data) % 256
    with pytest.raises(tk.TkError) as e:   # pageable host memory is refused
        tk.tk_swiglu_quant_run_mapped(op.plan, T, start, w_h, q_h, s_h, None, None)
    assert e.value.status == 1
    # zero rows: nothing is checked or launched
    tk.tk_swiglu_quant_run_mapped(op.plan, 0, None, None, None, None, None, None)
