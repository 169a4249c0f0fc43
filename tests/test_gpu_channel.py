"""Per-channel cast on the GPU against the oracle, through the C ABI.

One scale per column from the column's absolute maximum over every row; the
input is the activation itself, so scales and codes must equal the oracle's
bit for bit. Cases: every format combination on hand-shaped inputs (zero,
subnormal, saturating and tiny columns), the batch sizes 1, 257, 8192 and
100003, and the benchmark workloads at full size (the whole output compared).
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import parallel
from parity import unpack

import activation_fp8_quantization_gb300 as tk
from activation_fp8_quantization_gb300 import workloads as wls

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, params=["chunk", "split"])
def channel_kernel(request, monkeypatch):
    """Every test runs on both forms of the cast (read when a plan is made):
    the chunk quantize pass, which reduces its scales itself, and the scale
    kernel followed by the row quantize pass."""
    monkeypatch.setenv("TK_CHANNEL_KERNEL", request.param)
    return request.param


def _shaped_input(T, H, in_dtype, seed):
    rng = np.random.default_rng(seed)
    v = rng.standard_normal((T, H)) * np.exp2(rng.integers(-40, 40, (1, H)))
    v[:, 3 % H] = 0.0                                     # an all-zero column
    if H > 5:
        v[:, 4] = 2.0 ** -140 * np.sign(rng.standard_normal(T))   # subnormal column (fp32)
        v[:, 5] = np.where(np.arange(T) % 3 == 0, 448.0, -0.0)    # exact Qmax and -0
    if H > 6:
        v[:, 6] = rng.standard_normal(T) * 1e-30
    y = torch.from_numpy(v.astype(np.float32))
    return y.to(torch.bfloat16) if in_dtype == "bf16" else y


def _check(x_cpu, q, s, scale_fmt, out_fmt, procs=None):
    y = x_cpu.float().numpy()
    if y.size > 4_000_000:
        rq, rs = parallel.quant_cols_f32(y, scale_fmt, out_fmt, procs=procs)
    else:
        rq, rs = oracle.quant_cols_f32(y, scale_fmt, out_fmt)
    gq, gs = q.cpu().numpy(), s.cpu().numpy()
    if scale_fmt == "fp32":
        bad_s = np.nonzero(gs.view(np.uint32) != rs.view(np.uint32))[0]
    else:
        bad_s = np.nonzero(gs != rs)[0]
    assert bad_s.size == 0, "scales differ at columns %s: %s vs %s" % (bad_s[:5], gs[bad_s[:5]], rs[bad_s[:5]])
    bad = np.argwhere(unpack(gq, out_fmt) != unpack(rq, out_fmt))
    assert bad.size == 0, "codes differ at %s" % (bad[:5].tolist(),)


def _run(op, x, workspace=None):
    q, s = op(x, workspace=workspace)
    torch.cuda.synchronize()
    assert tk.tk_fault_word(torch.cuda.current_device()) == 0
    return q, s


@pytest.mark.parametrize("T", [1, 2, 33, 257, 4099])
@pytest.mark.parametrize("in_dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("H", [16, 48, 512, 1040, 4096, 7168, 9216])
@pytest.mark.parametrize("scale_fmt,out_fmt", [("fp32", "e4m3"), ("ue8m0", "e4m3"),
                                               ("ue8m0", "e2m1"), ("fp32", "e2m1")])
def test_channel_bit_exact(T, in_dtype, H, scale_fmt, out_fmt):
    if T * H > 2_500_000 and (in_dtype, scale_fmt, out_fmt) != ("bf16", "fp32", "e4m3"):
        pytest.skip("the largest shapes run in one format combination")
    x = _shaped_input(T, H, in_dtype, seed=T * 7 + H)
    op = tk.QuantCast(H, 0, scale_fmt, out_fmt, in_dtype, granularity="channel")
    q, s = _run(op, x.cuda())
    assert tuple(s.shape) == (H,)
    _check(x, q, s, scale_fmt, out_fmt)


@pytest.mark.parametrize("T,H", [(1, 4096), (257, 4096), (8192, 4096), (100003, 2048)])
def test_channel_batch_sizes(T, H):
    """The batch sizes of the workloads' ladder on the per-channel inputs
    (every column its own LogNormal magnitude); the whole output compared."""
    wl = wls.CAST_WORKLOADS["cast_T8192_H4096_channel_bf16"]
    wl = wls.Workload(**{**wl.__dict__, "T": T, "H": H})
    x, _ = wls.make_inputs(wl, "cpu")
    op = tk.QuantCast(H, 0, wl.scale_fmt, wl.out_fmt, wl.in_dtype, granularity="channel")
    q, s = _run(op, x.cuda())
    _check(x, q, s, wl.scale_fmt, wl.out_fmt)


@pytest.mark.parametrize("name", [n for n, w in wls.CAST_WORKLOADS.items() if w.channel])
def test_channel_workload_full_size(name):
    """Each per-channel benchmark workload at full size, in the benchmark's
    launch configuration, every code and scale compared."""
    wl = wls.CAST_WORKLOADS[name]
    x, _ = wls.make_inputs(wl, "cpu")
    op = tk.QuantCast(wl.H, 0, wl.scale_fmt, wl.out_fmt, wl.in_dtype, granularity="channel")
    q, s = _run(op, x.cuda())
    _check(x, q, s, wl.scale_fmt, wl.out_fmt)


def test_channel_workspace_needs_no_initialisation():
    """Workspace filled with 0xFF (NaN partial maxima) before the run, and
    the same workspace reused by a second run of other data: both exact."""
    H, T = 3072, 5000
    op = tk.QuantCast(H, 0, "fp32", "e4m3", "bf16", granularity="channel")
    ws = torch.full((op.workspace_bytes(T),), 0xFF, dtype=torch.uint8, device="cuda")
    for seed in (1, 2):
        x = _shaped_input(T, H, "bf16", seed)
        q, s = _run(op, x.cuda(), workspace=ws)
        _check(x, q, s, "fp32", "e4m3")


def test_channel_runs_repeat_bit_for_bit():
    H, T = 4096, 20000
    x = _shaped_input(T, H, "bf16", 5).cuda()
    op = tk.QuantCast(H, 0, "ue8m0", "e2m1", "bf16", granularity="channel")
    q1, s1 = _run(op, x)
    q2, s2 = _run(op, x)
    assert torch.equal(q1, q2) and torch.equal(s1, s2)


def test_channel_argument_errors():
    H, T = 1024, 100
    op = tk.QuantCast(H, 0, "fp32", "e4m3", "bf16", granularity="channel")
    x = torch.zeros((T, H), dtype=torch.bfloat16, device="cuda")
    q = torch.empty((T, H), dtype=torch.uint8, device="cuda")
    s = torch.full((H + 4,), 7.0, dtype=torch.float32, device="cuda")
    need = tk.tk_quant_cast_workspace_size(op.plan, T)
    assert need > 0 and tk.tk_quant_cast_workspace_size(op.plan, 0) == 0
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    # the workspace-free call refuses a per-channel plan
    with pytest.raises(tk.TkError) as e:
        tk.tk_quant_cast_run(op.plan, T, x, q, s, stream)
    assert e.value.status == 1
    # too little workspace, or none
    with pytest.raises(tk.TkError) as e:
        tk.tk_quant_cast_run_ws(op.plan, T, x, q, s, ws, need - 4, stream)
    assert e.value.status == 1
    with pytest.raises(tk.TkError) as e:
        tk.tk_quant_cast_run_ws(op.plan, T, x, q, s, None, 0, stream)
    assert e.value.status == 1
    # scales must be 16-byte aligned
    with pytest.raises(tk.TkError) as e:
        tk.tk_quant_cast_run_ws(op.plan, T, x, q, s.data_ptr() + 4, ws, need, stream)
    assert e.value.status == 3
    # zero rows: nothing runs, the scales stay as they were
    tk.tk_quant_cast_run_ws(op.plan, 0, x, q, s, None, 0, stream)
    torch.cuda.synchronize()
    assert bool((s == 7.0).all())
    # a per-token plan needs no workspace and runs through the same call
    op2 = tk.QuantCast(H, 0, "fp32", "e4m3", "bf16")
    assert tk.tk_quant_cast_workspace_size(op2.plan, T) == 0
    q2, s2 = op2(x)
    torch.cuda.synchronize()
    assert bool((s2 == 1.0).all()) and not bool(q2.any())


def test_channel_launch_info(channel_kernel, monkeypatch):
    """The plan picks the form by the size of the codes (96 MiB), unless
    TK_CHANNEL_KERNEL forces one; launch_info reports the choice."""
    monkeypatch.delenv("TK_CHANNEL_KERNEL")
    op = tk.QuantCast(7168, 0, "ue8m0", "e4m3", "bf16", granularity="channel")
    assert op.launch_info(0)["launches"] == 0
    small = op.launch_info(8192)               # 56 MiB of codes
    big = op.launch_info(16384)                # 112 MiB
    assert (small["form"], small["launches"]) == (1, 2)
    assert (big["form"], big["launches"]) == (2, 3)
    monkeypatch.setenv("TK_CHANNEL_KERNEL", channel_kernel)
    forced = tk.QuantCast(7168, 0, "ue8m0", "e4m3", "bf16", granularity="channel")
    want = 1 if channel_kernel == "chunk" else 2
    assert forced.launch_info(8192)["form"] == want and forced.launch_info(16384)["form"] == want
    per_block = tk.QuantCast(7168, 128, "ue8m0", "e4m3", "bf16")
    assert per_block.launch_info(100)["launches"] == 1 and per_block.launch_info(100)["form"] == 0
