"""The fused op with the codes written transposed (tk_swiglu_quant_run_transposed),
through the C ABI.

The transposed kernel runs the same arithmetic as the row-major kernels, so
its codes, scales and clamp counters must equal theirs bit for bit (the codes
after transposing back), and its codes meet the oracle under the tolerance of
the other parity tests (the oracle's own transpose, pinned on CPU, gives the
expected layout). Rows T <= t < ld of every code row are zero; nothing past
ld * H bytes is written.
"""
import numpy as np
import pytest
import torch

import oracle
from parity import compare

import activation_fp8_quantization_gb300 as tk
from activation_fp8_quantization_gb300 import _abi
from activation_fp8_quantization_gb300 import workloads as wls

pytestmark = pytest.mark.gpu


def _inputs(T, H, seed, dist="row_lognormal", clamp=None):
    wl = wls.Workload("t", T, H, 128, "fp32", "e4m3", dist, seed=seed, w_dist="topk8_norm",
                      clamp=clamp)
    return wls.make_inputs(wl, "cpu")


def _both(op, x, w):
    """(row-major codes, scales, counts) and (qt, scales, counts) of one input."""
    counts0 = torch.zeros(2, dtype=torch.int64, device="cuda") if op.count_clamped else None
    counts1 = torch.zeros(2, dtype=torch.int64, device="cuda") if op.count_clamped else None
    q, s = op(x, w, clamped_count=counts0)
    qt, st = op.transposed(x, w, clamped_count=counts1)
    torch.cuda.synchronize()
    return (q, s, counts0), (qt, st, counts1)


@pytest.mark.parametrize("scale_fmt", ["fp32", "ue8m0"])
@pytest.mark.parametrize("group", [32, 64, 128])
@pytest.mark.parametrize("H,T", [(128, 1), (256, 15), (256, 16), (512, 17), (2048, 63), (2048, 64),
                                 (2048, 65), (1024, 1000), (7168, 129), (16384, 33)])
def test_transposed_matches_row_major_and_oracle(H, T, group, scale_fmt):
    x, w = _inputs(T, H, seed=H + 7 * T + group)
    op = tk.SwigluQuant(H, group, scale_fmt, "e4m3", True)
    (q, s, _), (qt, st, _) = _both(op, x.cuda(), w.cuda())
    _, ld = tk.tk_swiglu_quant_transposed_size(op.plan, T)
    assert ld == (T + 31) // 32 * 32 and qt.shape == (H, ld)
    qt_h = qt.cpu().numpy()
    assert np.array_equal(qt_h[:, :T].T, q.cpu().numpy())
    assert not qt_h[:, T:].any()
    assert torch.equal(st.view(torch.uint8), s.view(torch.uint8))
    ref = oracle.swiglu_quant(wls.bf16_bits(x), w.numpy(), group, scale_fmt, "e4m3", want_y=True)
    # the transposed codes against the oracle's transposed codes (padding included)
    want_t = oracle.codes_transposed(ref["q"], ld)
    rep = compare(qt_h[:, :T].T.copy(), st.cpu().numpy(), ref, group, scale_fmt, "e4m3")
    rep.check("H=%d T=%d g=%d %s" % (H, T, group, scale_fmt))
    assert np.array_equal(qt_h[:, T:], want_t[:, T:])


@pytest.mark.parametrize("layout", ["col", "col_packed"])
def test_transposed_scale_layouts(layout):
    H, T, group = 2048, 300, 128
    x, w = _inputs(T, H, seed=5)
    op = tk.SwigluQuant(H, group, "ue8m0", "e4m3", True, scale_layout=layout)
    (q, s, _), (qt, st, _) = _both(op, x.cuda(), w.cuda())
    assert np.array_equal(qt.cpu().numpy()[:, :T].T, q.cpu().numpy())
    # compare the written entries only (padding rows of the column layouts are not written)
    ref = oracle.swiglu_quant(wls.bf16_bits(x), w.numpy(), group, "ue8m0", "e4m3")
    want = oracle.scales_to_layout(ref["scales"], "ue8m0", layout, fill=0)
    got = st.cpu().numpy().view(np.uint8).reshape(-1)
    mask = oracle.scales_to_layout(np.ones_like(ref["scales"]), "ue8m0", layout, fill=0) != 0
    assert got.size == want.size
    assert (got[mask] == want[mask]).mean() > 0.999
    assert np.array_equal(got[mask], s.cpu().numpy().view(np.uint8).reshape(-1)[mask])


def test_transposed_clamp_counters():
    H, T, group, L = 2048, 777, 128, 7.0
    wl = wls.WORKLOADS["moe_T32768_H2048_g128_ue8m0_clamp7"].with_rows(T)
    x, w = wls.make_inputs(wl, "cpu")
    op = tk.SwigluQuant(H, group, "ue8m0", "e4m3", True, clamp_limit=L, count_clamped=True)
    (q, s, c0), (qt, st, c1) = _both(op, x.cuda(), w.cuda())
    assert np.array_equal(qt.cpu().numpy()[:, :T].T, q.cpu().numpy())
    assert torch.equal(st, s)
    ref = oracle.swiglu_quant(wls.bf16_bits(x), w.numpy(), group, "ue8m0", "e4m3", clamp=L)
    assert c1.cpu().tolist() == ref["counts"].tolist() == c0.cpu().tolist()


@pytest.mark.parametrize("name", ["moe_T8192_H2048_g128", "moe_T32768_H2048_g128_ue8m0_clamp7",
                                  "ragged_T100003_H3072_g128"])
def test_transposed_full_bench_workload(name):
    """The workloads `bench.py --transposed` times, at full size and in its
    launch configuration (the plan's prefetch form and grid): every code and
    scale equal to the row-major kernel's output (itself compared with the
    oracle at full size), the clamp counters too, the padding zero."""
    wl = wls.WORKLOADS[name]
    x, w = wls.make_inputs(wl, "cuda")
    op = tk.SwigluQuant(wl.H, wl.group, wl.scale_fmt, wl.out_fmt, True, wl.clamp, wl.clamp is not None)
    (q, s, c0), (qt, st, c1) = _both(op, x, w)
    assert torch.equal(qt[:, :wl.T].t(), q)
    assert not bool(qt[:, wl.T:].any())
    assert torch.equal(st, s)
    if wl.clamp is not None:
        assert c0.cpu().tolist() == c1.cpu().tolist()
    assert tk.tk_fault_word(torch.cuda.current_device()) == 0


def test_transposed_writes_nothing_past_ld():
    H, T = 256, 40
    x, w = _inputs(T, H, seed=11)
    op = tk.SwigluQuant(H, 128, "fp32", "e4m3", True)
    n, ld = tk.tk_swiglu_quant_transposed_size(op.plan, T)
    assert n == H * ld
    guard = 4096
    buf = torch.full((n + 2 * guard,), 0x5A, dtype=torch.uint8, device="cuda")
    s = torch.empty((T, H // 128), dtype=torch.float32, device="cuda")
    xc, wc = x.cuda(), w.cuda()
    tk.tk_swiglu_quant_run_transposed(op.plan, T, xc, wc, buf.data_ptr() + guard, s, None,
                                      torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    b = buf.cpu().numpy()
    assert (b[:guard] == 0x5A).all() and (b[guard + n:] == 0x5A).all()
    q, _ = op(xc, wc)
    torch.cuda.synchronize()
    assert np.array_equal(b[guard:guard + n].reshape(H, ld)[:, :T].T, q.cpu().numpy())


def test_transposed_refused_where_unsupported():
    for args in ((256, 128, "ue8m0", "e2m1"), (256, 0, "fp32", "e4m3"), (144, 16, "fp32", "e4m3")):
        op = tk.SwigluQuant(*args, True)
        with pytest.raises(tk.TkError) as e:
            tk.tk_swiglu_quant_transposed_size(op.plan, 10)
        assert e.value.status == 2
        x = torch.zeros((10, 2 * args[0]), dtype=torch.bfloat16, device="cuda")
        with pytest.raises(tk.TkError) as e:
            op.transposed(x, torch.ones(10, device="cuda"))
        assert e.value.status == 2
    op = tk.SwigluQuant(256, 128, "fp32", "e4m3", True)
    x = torch.zeros((10, 512), dtype=torch.bfloat16, device="cuda")
    qt = torch.empty((256 * 16 + 16,), dtype=torch.uint8, device="cuda")
    s = torch.empty((10, 2), dtype=torch.float32, device="cuda")
    with pytest.raises(tk.TkError) as e:   # qt must be 16-byte aligned
        _abi.tk_swiglu_quant_run_transposed(op.plan, 10, x, torch.ones(10, device="cuda"), qt.data_ptr() + 8, s,
                                            None, None)
    assert e.value.status == 3


def test_transposed_zero_rows_is_a_noop():
    op = tk.SwigluQuant(256, 128, "fp32", "e4m3", True)
    n, ld = tk.tk_swiglu_quant_transposed_size(op.plan, 0)
    assert n == 0 and ld == 0
    tk.tk_swiglu_quant_run_transposed(op.plan, 0, None, None, None, None, None, None)
    torch.cuda.synchronize()
