"""Pins for the CPU oracle: checks against what the pages and the mathematics
fix, never against the oracle itself.

Each pin takes a loaded oracle library and raises AssertionError on a
mismatch. ``test_oracle_pins.py`` runs them on the real oracle;
``test_oracle_mutants.py`` runs them on copies of the oracle with one planted
mistake each and requires that some pin fails.

Sources of truth used here:
  * torch's CPU ``float8_e4m3fn`` cast and decode (a library routine; RNE,
    non-saturating, so it is used below 464 only) and its ``float8_e8m0fnu``
    cast (rounds a positive value up to a power of two) on quotients that are
    exact;
  * the OCP E2M1 grid {0, 0.5, 1, 1.5, 2, 3, 4, 6} and an independent
    brute-force nearest-even search written here in numpy;
  * textbook SwiGLU ``g * expit(g) * u * w`` with scipy's logistic function;
  * the hand-worked rows in tests/golden/hand_rows.json;
  * closed forms and invariants of absmax scaling.
"""
from __future__ import annotations

import json
import os

import numpy as np
import torch
from scipy.special import expit

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "hand_rows.json")

E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _bf16_bits(values) -> np.ndarray:
    t = torch.tensor(np.asarray(values, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _e4m3_grid_f64(lib) -> np.ndarray:
    return np.array([lib.tko_e4m3_decode(c) for c in range(0x7F)], np.float64)


# ------------------------------------------------------------------ formats

def pin_e4m3_decode_vs_torch(lib):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).float().double().numpy()
    got = np.array([lib.tko_e4m3_decode(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got)), "NaN codes differ"
    assert np.array_equal(ref[~nan], got[~nan]), "E4M3 decode differs from torch"
    # signed zero: code 0x80 is -0
    assert np.signbit(got[0x80]) and not np.signbit(got[0x00])


def _e4m3_sweep() -> np.ndarray:
    """fp32 values: every finite grid point, every midpoint and its fp32
    neighbours, random log-uniform magnitudes, tiny and zero values."""
    grid = np.array([float(torch.tensor([c], dtype=torch.uint8).view(torch.float8_e4m3fn).float())
                     for c in range(0x7F)])
    mids = (grid[:-1] + grid[1:]) / 2
    pts = np.concatenate([grid, mids]).astype(np.float32)
    up = np.nextafter(pts, np.float32(np.inf))
    dn = np.nextafter(pts, np.float32(-np.inf))
    rng = np.random.default_rng(7)
    rnd = np.exp2(rng.uniform(-14.0, np.log2(463.9), 6000)).astype(np.float32)
    tiny = np.array([1e-30, 2.0 ** -126, 2.0 ** -149, 2.0 ** -11, 2.0 ** -10], np.float32)
    v = np.concatenate([pts, up, dn, rnd, tiny, np.float32([0.0])])
    v = v[np.abs(v) < 464.0]
    return np.concatenate([v, -v]).astype(np.float32)


def pin_e4m3_encode_vs_torch(lib):
    v = _e4m3_sweep()
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([lib.tko_e4m3_encode(float(a)) for a in v], np.uint8)
    bad = np.nonzero(ref != got)[0]
    assert bad.size == 0, "E4M3 encode differs from torch at %r" % (v[bad[:5]],)


def pin_e4m3_saturation_and_roundtrip(lib):
    for a in [448.0, 449.0, 464.0, 480.0, 1e4, 3.0e38]:
        assert lib.tko_e4m3_encode(a) == 0x7E, a
        assert lib.tko_e4m3_encode(-a) == 0xFE, a
    for c in range(256):
        if c & 0x7F == 0x7F:
            continue
        assert lib.tko_e4m3_encode(lib.tko_e4m3_decode(c)) == c, hex(c)


def pin_e2m1_decode_table(lib):
    got = np.array([lib.tko_e2m1_decode(c) for c in range(16)])
    assert np.array_equal(got[:8], E2M1_GRID)
    assert np.array_equal(got[8:], -E2M1_GRID)
    assert np.signbit(got[8])


def pin_e2m1_ties(lib):
    # Ties go to the even code (even mantissa bit).
    table = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0,
             7.0: 6.0, 100.0: 6.0, 0.2: 0.0, 0.3: 0.5, 5.01: 6.0, 4.99: 4.0}
    for a, want in table.items():
        for sgn in (1.0, -1.0):
            code = lib.tko_e2m1_encode(sgn * a)
            got = lib.tko_e2m1_decode(code)
            assert got == sgn * want, (sgn * a, got, want)


def pin_e2m1_encode_bruteforce(lib):
    rng = np.random.default_rng(11)
    mids = (E2M1_GRID[:-1] + E2M1_GRID[1:]) / 2
    v = np.concatenate([E2M1_GRID, mids, rng.uniform(0, 8, 4000)]).astype(np.float32)
    v = np.concatenate([v, np.nextafter(v, np.float32(9)), np.nextafter(v, np.float32(-1))])
    v = v[v >= 0]
    dist = np.abs(v[:, None].astype(np.float64) - E2M1_GRID[None, :])
    # nearest; on a tie prefer the even code: sort key (distance, code parity)
    key = dist * 4.0 + (np.arange(8) % 2)[None, :] * 1e-9
    want = np.argmin(key, axis=1)
    want[v >= 6.0] = 7
    got = np.array([lib.tko_e2m1_encode(float(a)) for a in v])
    assert np.array_equal(got, want), v[got != want][:5]
    gotn = np.array([lib.tko_e2m1_encode(-float(a)) for a in v])
    assert np.array_equal(gotn, want | 8)


def pin_ue8m0(lib):
    # amax = qmax * 2^k exactly -> exponent k; one ulp above -> k + 1.
    for qmax in (448.0, 6.0):
        for k in range(-120, 118, 7):
            a = np.float32(qmax * 2.0 ** k)
            assert lib.tko_ue8m0_byte(float(a), qmax) == k + 127, (qmax, k)
            a_up = np.nextafter(a, np.float32(np.inf))
            assert lib.tko_ue8m0_byte(float(a_up), qmax) == k + 128, (qmax, k)
    assert lib.tko_ue8m0_byte(0.0, 448.0) == 127
    # torch's e8m0 cast rounds a positive value to the nearest power of two
    # (mantissa >= 1.5 goes up). The scale rule takes the smallest power of
    # two not below the quotient, so on exact quotients amax / 448 = m * 2^e
    # (1 <= m < 2) the two agree when m == 1 or m >= 1.5, and the scale rule
    # is one above torch when 1 < m < 1.5.
    for n in [1, 3, 5, 7, 9, 11, 13, 15, 17, 100, 127, 1000]:
        m = n / 2.0 ** np.floor(np.log2(n))
        for j in range(-30, 30, 3):
            amax = np.float32(7.0 * n * 2.0 ** j)          # 448 = 7 * 64
            quot = np.float32(n * 2.0 ** (j - 6))          # exact amax / 448
            ref = torch.tensor([float(quot)]).to(torch.float8_e8m0fnu).view(torch.uint8).item()
            want = ref + (1 if 1.0 < m < 1.5 else 0)
            assert lib.tko_ue8m0_byte(float(amax), 448.0) == want, (n, j)
    for b in [0, 1, 100, 127, 200, 254]:
        assert lib.tko_ue8m0_value(b) == np.float32(2.0 ** (b - 127))


def pin_ue8m0_lower_clamp(lib):
    # UE8M0's smallest finite scale is 2^-127 (byte 0). An amax that a
    # smaller power of two would cover still gets byte 0; the first amax above
    # Qmax * 2^-127 needs 2^-126 (byte 1). Subnormal amax included.
    for qmax in (448.0, 6.0):
        edge = np.float32(qmax * 2.0 ** -127)          # exact: 7 * 2^-121, 3 * 2^-126
        assert float(edge) == qmax * 2.0 ** -127
        assert lib.tko_ue8m0_byte(float(edge), qmax) == 0, qmax
        above = np.nextafter(edge, np.float32(np.inf))
        assert lib.tko_ue8m0_byte(float(above), qmax) == 1, qmax
        tiny = [np.nextafter(edge, np.float32(0)), edge / np.float32(2), np.float32(qmax * 2.0 ** -130),
                np.float32(2.0 ** -126), np.float32(2.0 ** -130), np.float32(2.0 ** -140),
                np.float32(3 * 2.0 ** -149), np.float32(2.0 ** -149)]
        for a in tiny:
            assert a > 0 and lib.tko_ue8m0_byte(float(a), qmax) == 0, (qmax, float(a))
    # through a whole row: a group whose amax is 2^-130 gets byte 0, so the
    # codes are the E4M3 encoding (torch's cast) of y * 2^127, exact in fp32
    y = np.array([[2.0 ** -130, -2.0 ** -131, 3 * 2.0 ** -133, 0.0]], np.float32)
    q, s = oracle.quant_rows_f32(y, 0, "ue8m0", "e4m3", lib=lib)
    assert int(s[0, 0]) == 0
    want = torch.from_numpy(y * np.float32(2.0 ** 127)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(q, want), (q, want)


def _random_positive_f32(rng, n):
    """Positive fp32 values spread over every binade, subnormals included."""
    bits = rng.integers(1, 0x7F7FFFFF, n, dtype=np.int64).astype(np.uint32)
    sub = rng.integers(1, 0x007FFFFF, n // 8, dtype=np.int64).astype(np.uint32)
    return np.concatenate([bits, sub]).view(np.float32)


def pin_fp32_scale_ieee(lib):
    # The fp32 scale is the IEEE single-precision quotient amax / Qmax,
    # correctly rounded (numpy's float32 division), replaced by 1 only when
    # it is zero. Non-power-of-two amax, normal and subnormal, and quotients
    # that come out subnormal.
    rng = np.random.default_rng(17)
    a = _random_positive_f32(rng, 4000)
    for qmax in (448.0, 6.0):
        want = a / np.float32(qmax)
        want = np.where(want == 0, np.float32(1.0), want)
        got = np.array([lib.tko_fp32_scale(float(v), qmax) for v in a], np.float32)
        bad = np.nonzero(got.view(np.uint32) != want.view(np.uint32))[0]
        assert bad.size == 0, (qmax, a[bad[:3]], got[bad[:3]], want[bad[:3]])
    # through whole rows: every group's scale is fl32(max|y| / Qmax) bit for bit
    y = (rng.standard_normal((6, 256)) * np.exp2(rng.uniform(-140, 100, (6, 1)))).astype(np.float32)
    for out_fmt, qmax in (("e4m3", 448.0), ("e2m1", 6.0)):
        _, sc = oracle.quant_rows_f32(y, 32, "fp32", out_fmt, lib=lib)
        amax = np.abs(y).reshape(6, 8, 32).max(axis=2)
        want = amax / np.float32(qmax)
        want = np.where(want == 0, np.float32(1.0), want)
        assert np.array_equal(sc.view(np.uint32), want.view(np.uint32)), out_fmt


# ---------------------------------------------------------------- full rows

def _fmt_codes(q: np.ndarray):
    return ["%02X" % int(c) for c in q.reshape(-1)]


def pin_hand_rows(lib):
    rows = json.load(open(GOLDEN))["rows"]
    for r in rows:
        x = _bf16_bits(np.concatenate([r["gate"], r["up"]]))[None, :]
        w = None if r["w"] is None else np.array([r["w"]], np.float32)
        out = oracle.swiglu_quant(x, w, r["group"], r["scale_fmt"], r["out_fmt"],
                                  clamp=r["clamp"], lib=lib)
        assert _fmt_codes(out["q"]) == r["q"], (r["name"], _fmt_codes(out["q"]))
        if r["scale_fmt"] == "fp32":
            s = float(out["scales"].reshape(-1)[0])
            assert abs(s - r["scale_approx"]) <= 1e-6 * r["scale_approx"], (r["name"], s)
        else:
            assert int(out["scales"].reshape(-1)[0]) == r["scale_byte"], r["name"]
        assert out["counts"].tolist() == r["counts"], (r["name"], out["counts"])


def pin_clamp_limit_strict(lib):
    # The guard fires on values strictly past the limit ("val > clamp value").
    x = _bf16_bits([7.0, 8.0, -7.0, 7.0, -8.0, 7.0])[None, :]
    out = oracle.swiglu_quant(x, None, 0, "fp32", "e4m3", clamp=7.0, lib=lib)
    assert out["counts"].tolist() == [1, 1]
    # counts accumulate into the caller's counter across calls
    acc = np.zeros(2, np.int64)
    q = np.zeros(3, np.uint8)
    s = np.zeros(1, np.float32)
    for _ in range(3):
        lib.tko_swiglu_quant(x.ctypes.data, 1, 3, None, 0, 0, 0, 1, 7.0,
                             q.ctypes.data, s.ctypes.data, acc.ctypes.data, None)
    assert acc.tolist() == [3, 3]


def _random_rows(rng, rows, H, spread=True):
    v = rng.standard_normal((rows, 2 * H)).astype(np.float32)
    if spread:
        v *= np.exp(rng.standard_normal((rows, 1))).astype(np.float32)
    return _bf16_bits(v)


def pin_swiglu_textbook(lib):
    rng = np.random.default_rng(3)
    H = 256
    x = _random_rows(rng, 24, H)
    w = rng.uniform(0.01, 1.0, 24).astype(np.float32)
    for clamp in (None, 3.0):
        out = oracle.swiglu_quant(x, w, 128, "fp32", "e4m3", clamp=clamp, want_y=True, lib=lib)
        g = _bits_to_f64(x[:, :H])
        u = _bits_to_f64(x[:, H:])
        cnt = [0, 0]
        if clamp is not None:
            cnt = [int((g > clamp).sum()), int((np.abs(u) > clamp).sum())]
            g = np.minimum(g, clamp)
            u = np.clip(u, -clamp, clamp)
        ref = (g * expit(g) * u * w.astype(np.float64)[:, None]).astype(np.float32)
        got = out["y"]
        ulp = np.abs(got.view(np.int32).astype(np.int64) - ref.view(np.int32).astype(np.int64))
        assert ulp.max() <= 1, "activation differs from textbook SwiGLU by %d ulp" % ulp.max()
        assert out["counts"].tolist() == cnt


def _spacing(a: np.ndarray, out_fmt: str) -> np.ndarray:
    """Grid spacing of the format at magnitude a (within a's binade)."""
    a = np.abs(a).astype(np.float64)
    if out_fmt == "e4m3":
        e = np.floor(np.log2(np.maximum(a, 2.0 ** -6)))
        return 2.0 ** (e - 3)
    return np.where(a < 2.0, 0.5, np.where(a < 4.0, 1.0, 2.0))


def pin_invariants(lib):
    rng = np.random.default_rng(5)
    H = 512
    x = _random_rows(rng, 16, H)
    w = rng.uniform(0.05, 1.0, 16).astype(np.float32)
    for out_fmt, qmax in (("e4m3", 448.0), ("e2m1", 6.0)):
        dec = (oracle.e4m3_decode_table(lib) if out_fmt == "e4m3"
               else oracle.e2m1_decode_table(lib))
        for scale_fmt in ("fp32", "ue8m0"):
            for group in (32, 128, 0):
                out = oracle.swiglu_quant(x, w, group, scale_fmt, out_fmt, want_y=True, lib=lib)
                y = out["y"].astype(np.float64)
                g = H if group == 0 else group
                q = out["q"] if out_fmt == "e4m3" else oracle.unpack_e2m1(out["q"])
                vals = dec[q]
                sc = out["scales"].astype(np.float64)
                if scale_fmt == "ue8m0":
                    sc = 2.0 ** (sc - 127.0)
                s_full = np.repeat(sc, g, axis=1)
                assert np.all(np.abs(vals) <= qmax)
                yq = y / s_full
                err = np.abs(vals - yq)
                bound = 0.5 * _spacing(yq, out_fmt) + 2.0 ** -23 * np.abs(yq)
                assert np.all(err <= bound), (out_fmt, scale_fmt, group, err.max())
                yg = y.reshape(y.shape[0], -1, g)
                amax = np.abs(yg).max(axis=2)
                ratio = amax / sc
                if scale_fmt == "fp32":
                    arg = np.abs(yg).argmax(axis=2)
                    top = np.take_along_axis(vals.reshape(yg.shape), arg[..., None], axis=2)
                    assert np.all(np.abs(top) == qmax), (out_fmt, group)
                    assert np.allclose(ratio, qmax, rtol=2.0 ** -22)
                else:
                    assert np.all((ratio > qmax / 2) & (ratio <= qmax)), (out_fmt, group)


def pin_group_indexing(lib):
    # Each group j of each row r gets a different planted peak, so a mixed-up
    # group or row index shows in the scales and in which code reaches max.
    H, g, rows = 512, 128, 3
    gate = np.full((rows, H), 4.0, np.float32)
    up = np.full((rows, H), 0.01, np.float32)
    peaks = {}
    for r in range(rows):
        for j in range(H // g):
            col = j * g + (17 * j + 5 * r) % g
            up[r, col] = float(2 ** (j + r + 1))
            peaks[(r, j)] = col
    x = _bf16_bits(np.concatenate([gate, up], axis=1))
    out = oracle.swiglu_quant(x, None, g, "ue8m0", "e4m3", want_y=True, lib=lib)
    silu4 = 4.0 * expit(4.0)
    for (r, j), col in peaks.items():
        amax = np.float32(silu4 * 2 ** (j + r + 1))
        k = int(np.ceil(np.log2(float(amax) / 448.0)))
        assert int(out["scales"][r, j]) == k + 127, (r, j)
        big = [c for c in range(j * g, (j + 1) * g) if out["q"][r, c] & 0x7F >= 0x70]
        assert big == [col], (r, j, big, col)


def pin_zero_and_signed_zero(lib):
    H = 64
    for out_fmt in ("e4m3", "e2m1"):
        for scale_fmt in ("fp32", "ue8m0"):
            gate = np.zeros((1, H), np.float32)
            up = np.where(np.arange(H) % 2 == 0, 1.0, -1.0).astype(np.float32)[None, :]
            x = _bf16_bits(np.concatenate([gate, up], axis=1))
            out = oracle.swiglu_quant(x, None, 32, scale_fmt, out_fmt, lib=lib)
            sc = out["scales"].reshape(-1)
            if scale_fmt == "fp32":
                assert np.all(sc == 1.0)
            else:
                assert np.all(sc == 127)
            q = out["q"] if out_fmt == "e4m3" else oracle.unpack_e2m1(out["q"])
            sign = 0x80 if out_fmt == "e4m3" else 0x8
            # 0 * (+1) = +0 and 0 * (-1) = -0: codes are signed zeros
            want = np.where(np.arange(H) % 2 == 0, 0, sign)
            assert np.array_equal(q.reshape(-1), want), (out_fmt, q)


def pin_e2m1_packing(lib):
    # One group of 4 values whose codes are all different: 6*[1, 0.5, -1/3, 1/6]
    y = np.array([[6.0, 3.0, -2.0, 1.0]], np.float32)
    q, s = oracle.quant_rows_f32(y, 0, "fp32", "e2m1", lib=lib)
    assert float(s[0, 0]) == 1.0
    # codes: 6 -> 0x7, 3 -> 0x5, -2 -> 0xC, 1 -> 0x2; value 2k in the low nibble
    assert q.tolist() == [[0x57, 0x2C]], q


def pin_quant_rows_indexing(lib):
    # Multi-row, multi-group fp32 input: group j of row r holds one peak
    # 2^(j + 4r) among values 0.5, so its scale is peak / 448 and the only
    # maximal code sits at the peak's column.
    rows, H, g = 3, 256, 64
    y = np.full((rows, H), 0.5, np.float32)
    cols = {}
    for r in range(rows):
        for j in range(H // g):
            c = j * g + (11 * j + 7 * r) % g
            y[r, c] = np.float32(2.0 ** (j + 4 * r))
            cols[(r, j)] = c
    for out_fmt, qmax, top in (("e4m3", 448.0, 0x7E), ("e2m1", 6.0, 0x7)):
        q, sc = oracle.quant_rows_f32(y, g, "fp32", out_fmt, lib=lib)
        q = q if out_fmt == "e4m3" else oracle.unpack_e2m1(q)
        for (r, j), c in cols.items():
            assert sc[r, j] == np.float32(y[r, c]) / np.float32(qmax), (out_fmt, r, j)
            tops = [k for k in range(j * g, (j + 1) * g) if q[r, k] == top]
            assert tops == [c], (out_fmt, r, j, tops)


GOLDEN_COLS = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "hand_cols.json")


def pin_quant_cols_hand(lib):
    # tests/golden/hand_cols.json: a 3 x 4 input worked by hand in three modes
    d = json.load(open(GOLDEN_COLS))
    x = np.array(d["x"], np.float32)
    for c in d["cases"]:
        q, s = oracle.quant_cols_f32(x, c["scale_fmt"], c["out_fmt"], lib=lib)
        assert [["%02X" % int(v) for v in r] for r in q] == c["q"], (c["name"], q)
        if c["scale_fmt"] == "ue8m0":
            assert s.tolist() == c["scales"], (c["name"], s)
        else:
            assert np.allclose(s, c["scales_approx"], rtol=1e-6), (c["name"], s)


def pin_quant_cols_is_rows_of_transpose(lib):
    # Per-channel quantization of y is per-token quantization of y's
    # transpose (one group per row of y.T = one column of y), transposed back.
    rng = np.random.default_rng(23)
    rows, H = 10, 12
    y = (rng.standard_normal((rows, H)) * np.exp2(rng.uniform(-8, 8, (1, H)))).astype(np.float32)
    y[:, 5] = 0.0                           # an all-zero column
    y[3, 7] = -np.abs(y[:, 7]).max() * 1.5     # a negative column peak
    for scale_fmt in ("fp32", "ue8m0"):
        for out_fmt in ("e4m3", "e2m1"):
            q, s = oracle.quant_cols_f32(y, scale_fmt, out_fmt, lib=lib)
            qt, st = oracle.quant_rows_f32(np.ascontiguousarray(y.T), 0, scale_fmt, out_fmt, lib=lib)
            if out_fmt == "e2m1":
                q, qt = oracle.unpack_e2m1(q), oracle.unpack_e2m1(qt)
            assert np.array_equal(q, qt.T), (scale_fmt, out_fmt)
            assert np.array_equal(s, st.reshape(-1)), (scale_fmt, out_fmt)


def pin_quant_cols_planted_peaks(lib):
    # Column j holds one peak among small values; its scale is exactly
    # fl32(peak / Qmax) and the only saturated code of the column is the
    # peak's row.
    rows, H = 9, 16
    y = np.full((rows, H), 0.01, np.float32)
    peaks = {}
    for j in range(H):
        r = (5 * j + 2) % rows
        y[r, j] = np.float32((-1.0) ** j * 1.3 * 2.0 ** (j % 7 - 3))
        peaks[j] = r
    for out_fmt, qmax, top in (("e4m3", 448.0, 0x7E), ("e2m1", 6.0, 0x7)):
        q, s = oracle.quant_cols_f32(y, "fp32", out_fmt, lib=lib)
        q = q if out_fmt == "e4m3" else oracle.unpack_e2m1(q)
        mag = q & (0x7F if out_fmt == "e4m3" else 0x7)
        for j, r in peaks.items():
            assert s[j] == np.float32(abs(y[r, j])) / np.float32(qmax), (out_fmt, j)
            assert np.nonzero(mag[:, j] == top)[0].tolist() == [r], (out_fmt, j, mag[:, j])


def pin_scale_layouts(lib):
    # column-major = numpy's transpose into a padded [G, ld] array; packed =
    # little-endian words of four consecutive group exponents (hand example)
    rng = np.random.default_rng(9)
    for rows in (1, 3, 17):
        f = rng.standard_normal((rows, 8)).astype(np.float32)
        got = oracle.scales_to_layout(f, "fp32", "col", lib=lib).view(np.float32)
        ld = -(-rows // 4) * 4
        want = np.zeros((8, ld), np.float32)
        want[:, :rows] = f.T
        assert np.array_equal(got.reshape(8, ld), want), rows
        b = rng.integers(0, 255, (rows, 8)).astype(np.uint8)
        got = oracle.scales_to_layout(b, "ue8m0", "col", lib=lib)
        ld = -(-rows // 16) * 16
        want = np.zeros((8, ld), np.uint8)
        want[:, :rows] = b.T
        assert np.array_equal(got.reshape(8, ld), want), rows
    b = np.array([[1, 2, 3, 4, 5, 6, 7, 8], [9, 10, 11, 12, 13, 14, 15, 16]], np.uint8)
    words = oracle.scales_to_layout(b, "ue8m0", "col_packed", lib=lib).view("<u4").reshape(2, 4)
    assert words[0, 0] == 0x04030201 and words[0, 1] == 0x0C0B0A09
    assert words[1, 0] == 0x08070605 and words[1, 1] == 0x100F0E0D
    assert words[0, 2] == 0 and words[1, 3] == 0     # padding rows 2, 3 not written


def pin_codes_transposed(lib):
    # hand example: 2 rows x 3 columns, ld 4 -> column i holds rows 0, 1 then zeros
    q = np.array([[1, 2, 3], [4, 5, 6]], np.uint8)
    got = oracle.codes_transposed(q, 4, lib=lib)
    assert got.tolist() == [[1, 4, 0, 0], [2, 5, 0, 0], [3, 6, 0, 0]]
    # numpy's transpose into a zero-padded array
    rng = np.random.default_rng(21)
    for rows, ld in ((1, 16), (17, 32), (64, 64)):
        q = rng.integers(0, 256, (rows, 48)).astype(np.uint8)
        want = np.zeros((48, ld), np.uint8)
        want[:, :rows] = q.T
        assert np.array_equal(oracle.codes_transposed(q, ld, lib=lib), want), (rows, ld)


def _ulp(v, mant_bits):
    v = np.maximum(np.abs(v), 2.0 ** -126)
    return np.exp2(np.floor(np.log2(v)) - mant_bits)


def pin_swiglu_backward(lib):
    from scipy.special import expit
    # hand-worked, L = 7, w = 0.5: column 0 has g = 0, u = 2, dy = 1:
    # sigmoid(0) = 1/2, silu = 0, silu' = 1/2 -> dgate = 1 * 0.5 * 2 * 0.5 = 0.5
    # (bf16 0x3F00), dup = 0; column 1 has g = 8 > L (clamped, so dgate = 0),
    # u = 1, dy = 2 -> dup = 2 * 0.5 * silu(7), silu(7) = 7 * expit(7) = 6.99362,
    # nearest bf16 7.0 (0x40E0); dw = 2 * silu(7) * 1 = 13.98724.
    x = np.array([[0x0000, 0x4100, 0x4000, 0x3F80]], np.uint16)     # g = (0, 8), u = (2, 1)
    dy = np.array([[0x3F80, 0x4000]], np.uint16)                     # (1, 2)
    dx, dw = oracle.swiglu_backward(x, dy, np.array([0.5], np.float32), clamp=7.0, lib=lib)
    assert dx.tolist() == [[0x3F00, 0x0000, 0x0000, 0x40E0]], [hex(v) for v in dx[0]]
    assert abs(float(dw[0]) - 2 * 7 * expit(7.0)) <= 2e-6
    # central differences of an independent forward (scipy's expit), in float64,
    # for the gate, the up half and the weight, with and without clamping
    rng = np.random.default_rng(31)
    rows, H = 3, 64
    for L in (None, 1.5):
        g = rng.normal(0, 2, (rows, H))
        u = rng.normal(0, 1.5, (rows, H))
        if L is not None:   # keep every value away from the clamp's kink
            g = np.where(np.abs(g - L) < 0.05, g + 0.2, g)
            u = np.where(np.abs(np.abs(u) - L) < 0.05, u * 1.1, u)
        xb = _bf16_bits(np.concatenate([g, u], axis=1))
        db = _bf16_bits(rng.normal(0, 1, (rows, H)))
        wv = rng.uniform(0.1, 1.0, rows).astype(np.float32)
        dx, dw = oracle.swiglu_backward(xb, db, wv, clamp=L, lib=lib)
        xv, dv = _bf16_to_f64(xb), _bf16_to_f64(db)
        gv, uv, w64 = xv[:, :H], xv[:, H:], wv.astype(np.float64)[:, None]

        def F(gg, uu, ww):   # the loss sum(dy * y) of the forward, per element
            if L is not None:
                gg = np.minimum(gg, L)
                uu = np.clip(uu, -L, L)
            return dv * gg * expit(gg) * uu * ww

        hg = 1e-6 * np.maximum(1.0, np.abs(gv))
        hu = 1e-6 * np.maximum(1.0, np.abs(uv))
        fd_g = (F(gv + hg, uv, w64) - F(gv - hg, uv, w64)) / (2 * hg)
        fd_u = (F(gv, uv + hu, w64) - F(gv, uv - hu, w64)) / (2 * hu)
        fd_w = (F(gv, uv, w64 + 1e-3) - F(gv, uv, w64 - 1e-3)).sum(axis=1) / 2e-3
        got = _bf16_to_f64(dx)
        for name, want, have in (("gate", fd_g, got[:, :H]), ("up", fd_u, got[:, H:])):
            tol = 0.5 * _ulp(want, 7) * (1 + 1e-6) + 1e-9 * np.abs(want) + 1e-30
            assert (np.abs(have - want) <= tol).all(), (name, L, np.abs(have - want).max())
        scale = np.abs(F(gv, uv, 1.0)).sum(axis=1)
        tol = 0.5 * _ulp(fd_w, 23) * (1 + 1e-6) + 1e-9 * scale
        assert (np.abs(dw.astype(np.float64) - fd_w) <= tol).all(), (L, np.abs(dw - fd_w).max())
    # no weights: w = 1
    dx1, dw1 = oracle.swiglu_backward(xb, db, None, clamp=L, lib=lib)
    dxw, dww = oracle.swiglu_backward(xb, db, np.ones(rows, np.float32), clamp=L, lib=lib)
    assert np.array_equal(dx1, dxw) and np.array_equal(dw1, dww)


def _bf16_to_f64(bits):
    return (np.asarray(bits, np.uint32) << 16).view(np.float32).astype(np.float64)


def pin_moe_reduce(lib):
    # hand-worked: y rows [1, 2] and [3, -1]; token 0 takes both with weights
    # 0.5 and 0.25 -> [1.25, 0.75]; token 1 takes row 1 with weight 2 and an
    # empty slot -> [6, -2] (bf16 0x3FA0 0x3F40 0x40C0 0xC000)
    y = np.array([[0x3F80, 0x4000], [0x4040, 0xBF80]], np.uint16)
    pos = np.array([[0, 1], [1, -1]], np.int32)
    w = np.array([[0.5, 0.25], [2.0, 9.0]], np.float32)
    assert oracle.moe_reduce(y, pos, w, 1.0, lib=lib).reshape(-1).tolist() == [0x3FA0, 0x3F40, 0x40C0, 0xC000]
    # global scale multiplies the sum
    assert oracle.moe_reduce(y, pos, w, 2.0, lib=lib).reshape(-1).tolist() == [0x4020, 0x3FC0, 0x4140, 0xC080]
    # exact bf16 midpoints round to the even mantissa: 1 + 2^-8 lies between
    # 1.0 (0x3F80) and 1 + 2^-7 (0x3F81) -> 0x3F80; 1 + 3 * 2^-8 lies between
    # 0x3F81 and 0x3F82 -> 0x3F82
    one = np.array([[0x3F80]], np.uint16)
    for wt, want in ((1 + 2.0 ** -8, 0x3F80), (1 + 3 * 2.0 ** -8, 0x3F82)):
        got = oracle.moe_reduce(one, np.array([[0]], np.int32), np.array([[wt]], np.float32), 1.0, lib=lib)
        assert int(got[0, 0]) == want, (wt, hex(int(got[0, 0])))
    rng = np.random.default_rng(13)
    R, H, T, K = 40, 256, 9, 4
    yb = _bf16_bits(rng.standard_normal((R, H)))
    # identity: one slot, weight 1, scale 1 gives the gathered rows back exactly
    perm = rng.permutation(R)[:T].astype(np.int32)
    got = oracle.moe_reduce(yb, perm[:, None], np.ones((T, 1), np.float32), 1.0, lib=lib)
    assert np.array_equal(got, yb[perm])
    # all slots empty: zeros
    got = oracle.moe_reduce(yb, np.full((T, K), -1, np.int32), np.ones((T, K), np.float32), 1.0, lib=lib)
    assert not got.any()
    # against a float64 einsum rounded to bf16 by torch (<= 1 bf16 ulp: torch may
    # round through fp32)
    pos = rng.integers(-1, R, (T, K)).astype(np.int32)
    w = rng.uniform(0, 1, (T, K)).astype(np.float32)
    yv = _bf16_to_f64(yb)
    ref = np.zeros((T, H))
    for t in range(T):
        for k in range(K):
            if pos[t, k] >= 0:
                ref[t] += float(w[t, k]) * yv[pos[t, k]]
    ref_b = torch.tensor(0.75 * ref).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.moe_reduce(yb, pos, w, 0.75, lib=lib)
    diff = np.abs(got.astype(np.int32) - ref_b.astype(np.int32))
    assert diff.max() <= 1 and (diff == 0).mean() > 0.99, diff.max()
    # E4M3 rows with 1x128 scales: codes decode through torch's float8 view
    codes = rng.integers(0, 256, (R, H)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0   # no NaN codes
    sc = rng.uniform(0.5, 2.0, (R, H // 128)).astype(np.float32)
    dec = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy() * np.repeat(sc, 128, axis=1)
    ref = np.zeros((T, H))
    for t in range(T):
        for k in range(K):
            if pos[t, k] >= 0:
                ref[t] += float(w[t, k]) * dec[pos[t, k]]
    ref_b = torch.tensor(ref).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.moe_reduce(codes, pos, w, 1.0, y_scale=sc, lib=lib)
    diff = np.abs(got.astype(np.int32) - ref_b.astype(np.int32))
    assert diff.max() <= 1 and (diff == 0).mean() > 0.99, diff.max()


ALL_PINS = [
    pin_e4m3_decode_vs_torch,
    pin_e4m3_encode_vs_torch,
    pin_e4m3_saturation_and_roundtrip,
    pin_e2m1_decode_table,
    pin_e2m1_ties,
    pin_e2m1_encode_bruteforce,
    pin_ue8m0,
    pin_ue8m0_lower_clamp,
    pin_fp32_scale_ieee,
    pin_hand_rows,
    pin_clamp_limit_strict,
    pin_swiglu_textbook,
    pin_invariants,
    pin_group_indexing,
    pin_zero_and_signed_zero,
    pin_e2m1_packing,
    pin_quant_rows_indexing,
    pin_quant_cols_hand,
    pin_quant_cols_is_rows_of_transpose,
    pin_quant_cols_planted_peaks,
    pin_scale_layouts,
    pin_codes_transposed,
    pin_swiglu_backward,
    pin_moe_reduce,
]
