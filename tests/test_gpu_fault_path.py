"""The failure path of the kernels' bounded waits, exercised on the GPU
without a fault: tk_diag_unanswered_wait runs one thread that waits on an
mbarrier nothing arrives at, with the same wait helper as the library's
kernels. It must give up after the given number of tries, set bit 0 of the
fault word and return, and the context must stay usable."""
import time

import pytest
import torch

import oracle
from parity import compare

import activation_fp8_quantization_gb300 as tk
from activation_fp8_quantization_gb300 import workloads as wls

pytestmark = pytest.mark.gpu


def test_unanswered_wait_gives_up_and_flags():
    dev = torch.cuda.current_device()
    tk.tk_fault_word(dev, clear=True)
    stream = torch.cuda.current_stream()
    times = {}
    for tries in (1, 256):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        tk.tk_diag_unanswered_wait(dev, tries, stream.cuda_stream)
        torch.cuda.synchronize()
        times[tries] = time.perf_counter() - t0
        assert tk.tk_fault_word(dev, clear=True) == 1
    assert tk.tk_fault_word(dev) == 0
    per_try = (times[256] - times[1]) / 255
    print("unanswered try_wait: %.3f us per try; the kernels' limit of 2^19 tries: %.2f s"
          % (per_try * 1e6, per_try * (1 << 19)))
    # the give-up comes well after any legitimate copy, and within seconds
    assert 0.1 < per_try * (1 << 19) < 10.0
    # the context stays usable: an ordinary run afterwards matches the oracle
    wl = wls.WORKLOADS["moe_T8192_H2048_g128"].with_rows(300)
    x, w = wls.make_inputs(wl, "cpu")
    op = tk.SwigluQuant(wl.H, wl.group, wl.scale_fmt, wl.out_fmt, True)
    q, s = op(x.cuda(), w.cuda())
    torch.cuda.synchronize()
    ref = oracle.swiglu_quant(wls.bf16_bits(x), w.numpy(), wl.group, wl.scale_fmt, wl.out_fmt, want_y=True)
    compare(q.cpu().numpy(), s.cpu().numpy(), ref, wl.group, wl.scale_fmt, wl.out_fmt).check("after the wait")
    assert tk.tk_fault_word(dev) == 0
