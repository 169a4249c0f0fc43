"""The multi-process oracle runner gives the same bytes as one
single-threaded call (rows, or columns for the per-channel cast, split over
spawned processes)."""
import numpy as np

import oracle
from oracle import parallel
from activation_fp8_quantization_gb300 import workloads as wls


def test_rows_split_equals_one_call():
    wl = wls.WORKLOADS["moe_T32768_H2048_g128_ue8m0_clamp7"].with_rows(101)
    x, w = wls.make_inputs(wl, "cpu")
    xb, wn = wls.bf16_bits(x), w.numpy()
    one = oracle.swiglu_quant(xb, wn, wl.group, wl.scale_fmt, wl.out_fmt, clamp=wl.clamp, want_y=True)
    many = parallel.swiglu_quant(xb, wn, wl.group, wl.scale_fmt, wl.out_fmt, clamp=wl.clamp, want_y=True,
                                 procs=3)
    for k in ("q", "scales", "counts", "y"):
        assert np.array_equal(one[k], many[k]), k


def test_columns_split_equals_one_call():
    rng = np.random.default_rng(3)
    y = (rng.standard_normal((37, 50)) * np.exp(rng.standard_normal((1, 50)))).astype(np.float32)
    for scale_fmt, out_fmt in (("fp32", "e4m3"), ("ue8m0", "e2m1")):
        q1, s1 = oracle.quant_cols_f32(y, scale_fmt, out_fmt)
        q2, s2 = parallel.quant_cols_f32(y, scale_fmt, out_fmt, procs=4)
        assert np.array_equal(q1, q2) and np.array_equal(s1, s2), (scale_fmt, out_fmt)
