"""The GPU parity checker (tests/parity.py) on CPU: a stand-in for the
kernel's output is made from the oracle's, with one planted difference, and
the checker must accept or reject it as the acceptance rules say."""
import numpy as np

import oracle
from parity import compare


def _boundary_case():
    # One row, two groups of 32. Group 0's amax is exactly 448 * 2^-3, so an
    # activation a few ulp larger would take the exponent -2 instead of -3.
    y = np.linspace(-0.03, 0.03, 64, dtype=np.float32).reshape(1, 64)
    y[0, 5] = np.float32(448.0 * 2.0 ** -3)
    q, s = oracle.quant_rows_f32(y, 32, "ue8m0", "e4m3")
    return y, q, s


def test_identical_output_passes():
    y, q, s = _boundary_case()
    rep = compare(q.copy(), s.copy(), {"y": y, "q": q, "scales": s}, 32, "ue8m0", "e4m3")
    rep.check("identical")
    assert rep.n_boundary_flips == 0


def test_boundary_flip_with_recomputed_codes_passes():
    y, q, s = _boundary_case()
    gq, gs = q.copy(), s.copy()
    gs[0, 0] += 1                     # the neighbouring exponent, 2^-2
    scale = np.float32(2.0 ** (int(gs[0, 0]) - 127))
    gq[0, :32] = [oracle.load().tko_e4m3_encode(float(v / scale)) for v in y[0, :32]]
    rep = compare(gq, gs, {"y": y, "q": q, "scales": s}, 32, "ue8m0", "e4m3")
    rep.check("flip")
    assert rep.n_boundary_flips == 1 and rep.n_flip_code_mismatch == 0


def test_boundary_flip_with_stale_codes_fails():
    y, q, s = _boundary_case()
    gq, gs = q.copy(), s.copy()
    gs[0, 0] += 1                     # exponent flipped but codes left at the old scale
    rep = compare(gq, gs, {"y": y, "q": q, "scales": s}, 32, "ue8m0", "e4m3")
    assert rep.n_flip_code_mismatch > 0
    try:
        rep.check("stale")
    except AssertionError:
        return
    raise AssertionError("the checker accepted codes that do not follow the kernel's scale")


def test_flip_away_from_a_boundary_fails():
    y, q, s = _boundary_case()
    gs = s.copy()
    gs[0, 1] += 1                     # group 1 is nowhere near a boundary
    rep = compare(q.copy(), gs, {"y": y, "q": q, "scales": s}, 32, "ue8m0", "e4m3")
    assert rep.notes


def test_chunked_comparison_merges_like_one_comparison():
    from parity import compare_chunked
    rng = np.random.default_rng(8)
    y = (rng.standard_normal((300, 256)) * np.exp(rng.standard_normal((300, 1)))).astype(np.float32)
    q, s = oracle.quant_rows_f32(y, 128, "fp32", "e4m3")
    ref = {"y": y, "q": q, "scales": s}
    gq = q.copy()
    gq[5, 7] ^= 1                      # one code a step away
    gq[250, 3] ^= 1
    one = compare(gq, s, ref, 128, "fp32", "e4m3")
    many = compare_chunked(gq, s, ref, 128, "fp32", "e4m3", chunk_rows=64)
    for k in ("n_codes", "n_code_mismatch", "max_step", "n_groups", "max_scale_rel"):
        assert getattr(one, k) == getattr(many, k), k
    assert many.n_code_mismatch == 2
