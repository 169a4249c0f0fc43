"""The host-buffer call that allocates nothing (tk_swiglu_quant_run_host_static).

It serves callers that may not allocate device memory at all, such as a
plug-in whose host application owns every byte of HBM through its own pool,
or a process with a fixed memory budget. Instead of a caller workspace it
stages rows in a fixed array built into the library. This file checks,
through the C ABI, that two calls in a row give the same codes, scales and
clamp counts as the workspace-based call (bit for bit, which is inside the
parity tolerance), and that a pipe too large for the array is refused
without any work being enqueued.

This file is collected last, and it passes both on its own in a fresh
process and after the rest of the suite.
"""
import pytest
import torch

import activation_fp8_quantization_gb300 as tk
from activation_fp8_quantization_gb300 import _abi
from activation_fp8_quantization_gb300 import workloads as wls

pytestmark = pytest.mark.gpu


def test_static_workspace_matches_caller_workspace_twice():
    wl = wls.WORKLOADS["moe_T32768_H2048_g128_ue8m0_clamp7"].with_rows(3001)
    x, w = wls.make_inputs(wl, "cpu")
    op = tk.SwigluQuant(wl.H, wl.group, wl.scale_fmt, wl.out_fmt, True, wl.clamp, True)
    pipe = tk.HostPipe(op, 1000)
    assert pipe.ws_bytes <= _abi.STATIC_SCRATCH_BYTES
    xh, wh = x.pin_memory(), w.pin_memory()

    # the existing entry point, with a workspace the caller allocated
    c_ref = torch.zeros(2, dtype=torch.int64).pin_memory()
    q_ref, s_ref = pipe(xh, wh, clamped_count=c_ref)
    torch.cuda.synchronize()
    q_shape, s_shape, s_dtype = op.output_shapes(wl.T)

    c = torch.zeros(2, dtype=torch.int64).pin_memory()
    stream = torch.cuda.current_stream()
    for call in range(1, 3):
        q = torch.full(q_shape, 0x5A, dtype=torch.uint8).pin_memory()
        s = torch.full(s_shape, 3, dtype=s_dtype).pin_memory()
        tk.tk_swiglu_quant_run_host_static(pipe.pipe, wl.T, xh, wh, q, s, c, stream.cuda_stream)
        torch.cuda.synchronize()
        assert torch.equal(q, q_ref), "codes differ on call %d" % call
        assert torch.equal(s, s_ref), "scales differ on call %d" % call
        # the counter is added to, like the workspace call's
        assert c.tolist() == [call * int(c_ref[0]), call * int(c_ref[1])]
    assert tk.tk_fault_word(torch.cuda.current_device()) == 0


def test_static_workspace_refuses_a_pipe_that_does_not_fit():
    op = tk.SwigluQuant(2048, 128, "fp32", "e4m3", True)
    pipe = tk.HostPipe(op, 8192)   # three slots of 8192 rows: far beyond 32 MiB
    assert pipe.ws_bytes > _abi.STATIC_SCRATCH_BYTES
    x = torch.zeros(16, 4096, dtype=torch.bfloat16).pin_memory()
    w = torch.ones(16).pin_memory()
    q = torch.empty(16, 2048, dtype=torch.uint8).pin_memory()
    s = torch.empty(16, 16).pin_memory()
    with pytest.raises(tk.TkError) as e:
        tk.tk_swiglu_quant_run_host_static(pipe.pipe, 16, x, w, q, s, None, None)
    assert e.value.status == 2
    assert "chunk_rows" in str(e.value)


def test_static_workspace_row_count_statuses_match_the_workspace_call():
    """T < 0 and T == 0 answer as tk_swiglu_quant_run_host does, before the
    size check: INVALID_ARG, and OK with nothing enqueued, even on a pipe too
    large for the built-in array."""
    op = tk.SwigluQuant(2048, 128, "fp32", "e4m3", True)
    big = tk.HostPipe(op, 8192)
    assert big.ws_bytes > _abi.STATIC_SCRATCH_BYTES
    x = torch.zeros(16, 4096, dtype=torch.bfloat16).pin_memory()
    w = torch.ones(16).pin_memory()
    q = torch.full((16, 2048), 0x33, dtype=torch.uint8).pin_memory()
    s = torch.full((16, 16), 5.0).pin_memory()
    with pytest.raises(tk.TkError) as e:
        tk.tk_swiglu_quant_run_host_static(big.pipe, -1, x, w, q, s, None, None)
    assert e.value.status == 1
    tk.tk_swiglu_quant_run_host_static(big.pipe, 0, x, w, q, s, None, None)
    torch.cuda.synchronize()
    assert bool((q == 0x33).all()) and bool((s == 5.0).all())
