"""The C-ABI library on a machine without a GPU: it loads, exports every
entry point the header declares, and its host-side checks answer without
touching a device."""
import ctypes
import os
import re

import pytest

import activation_fp8_quantization_gb300 as tk
from activation_fp8_quantization_gb300 import _abi

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "tk_swiglu_quant.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tk_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_binding():
    names = declared_functions()
    assert len(names) >= 12
    assert set(names) == set(_abi.SIGNATURES), set(names) ^ set(_abi.SIGNATURES)


def test_library_exports_every_declared_symbol():
    lib = _abi.lib()
    for name in declared_functions():
        assert hasattr(lib, name), name
    raw = ctypes.CDLL(_abi.LIB_PATH)
    for name in declared_functions():
        assert ctypes.cast(getattr(raw, name), ctypes.c_void_p).value


def D(**kw):
    base = dict(hidden=2048, group_size=128, scale_fmt=0, out_fmt=0, has_topk_weights=1,
                use_clamp=0, clamp_limit=0.0, count_clamped=0, scale_layout=0)
    base.update(kw)
    return tk.SwigluQuantDesc(**base)


@pytest.mark.parametrize("kw,status", [
    ({}, 0),
    (dict(group_size=0), 0),
    (dict(group_size=32, out_fmt=1, scale_fmt=1), 0),
    (dict(hidden=16384, group_size=512), 0),
    (dict(hidden=0), 1),
    (dict(hidden=-16), 1),
    (dict(hidden=2040), 2),
    (dict(hidden=16400), 2),
    (dict(group_size=-1), 1),
    (dict(group_size=96), 2),
    (dict(group_size=1024), 2),
    (dict(hidden=2064, group_size=128), 2),
    (dict(scale_fmt=2), 1),
    (dict(out_fmt=5), 1),
    (dict(has_topk_weights=2), 1),
    (dict(use_clamp=1, clamp_limit=float("nan")), 1),
    (dict(use_clamp=1, clamp_limit=float("inf")), 1),
    (dict(use_clamp=1, clamp_limit=-1.0), 1),
    (dict(use_clamp=1, clamp_limit=7.0, count_clamped=1), 0),
    (dict(count_clamped=1), 1),
    (dict(scale_layout=3), 1),
    (dict(scale_layout=1), 0),
    (dict(scale_layout=2, scale_fmt=1), 0),
    (dict(scale_layout=2, scale_fmt=0), 2),
    (dict(scale_layout=2, scale_fmt=1, group_size=512), 0),
    (dict(scale_layout=2, scale_fmt=1, group_size=0), 2),
])
def test_validate(kw, status):
    assert tk.tk_swiglu_quant_validate(D(**kw)) == status
    if status:
        assert tk.tk_last_error_message()


def test_cast_validate():
    C = tk.QuantCastDesc
    assert tk.tk_quant_cast_validate(C(4096, 128, 0, 0, 0, 0)) == 0
    assert tk.tk_quant_cast_validate(C(4096, 0, 1, 1, 1, 0)) == 0
    assert tk.tk_quant_cast_validate(C(4096, 128, 0, 0, 2, 0)) == 1
    assert tk.tk_quant_cast_validate(C(100, 0, 0, 0, 0, 0)) == 2
    assert tk.tk_quant_cast_validate(C(4096, 128, 1, 0, 0, 2)) == 0
    assert tk.tk_quant_cast_validate(C(4096, 128, 0, 0, 0, 2)) == 2
    # per channel: group_size 0, scales one row [H] (row-major), any formats
    for sf in (0, 1):
        for of in (0, 1):
            for dt in (0, 1):
                assert tk.tk_quant_cast_validate(C(4096, 0, sf, of, dt, 0, 1)) == 0
    assert tk.tk_quant_cast_validate(C(4096, 128, 0, 0, 0, 0, 1)) == 1   # group_size must be 0
    assert tk.tk_quant_cast_validate(C(4096, 0, 0, 0, 0, 1, 1)) == 2     # no column-major [H]
    assert tk.tk_quant_cast_validate(C(4096, 0, 0, 0, 0, 7, 1)) == 1     # unknown layout
    assert tk.tk_quant_cast_validate(C(4096, 0, 0, 0, 0, 0, 2)) == 1     # unknown granularity
    assert tk.tk_quant_cast_validate(C(4112, 0, 0, 0, 0, 0, 1)) == 0     # any multiple of 16


def test_output_sizes_of_scale_layouts():
    # column-major: columns padded to 16 bytes of scale elements
    assert tk.tk_swiglu_quant_output_sizes(D(scale_layout=1), 1001) == (1001 * 2048, 16 * 1004 * 4)
    assert tk.tk_swiglu_quant_output_sizes(D(scale_layout=1, scale_fmt=1), 1001) == (
        1001 * 2048, 16 * 1008)
    # packed UE8M0: 4 exponents per int32 word, rows padded to 4
    assert tk.tk_swiglu_quant_output_sizes(D(scale_layout=2, scale_fmt=1), 1001) == (
        1001 * 2048, 4 * 1004 * 4)
    C = tk.QuantCastDesc
    assert tk.tk_quant_cast_output_sizes(C(4096, 32, 1, 1, 0, 2), 7) == (7 * 2048, 32 * 8 * 4)
    assert tk.tk_quant_cast_output_sizes(C(4096, 0, 0, 0, 1, 0), 7) == (7 * 4096, 7 * 4)
    # per channel: one scale per column, whatever the number of rows
    assert tk.tk_quant_cast_output_sizes(C(4096, 0, 0, 0, 0, 0, 1), 7) == (7 * 4096, 4096 * 4)
    assert tk.tk_quant_cast_output_sizes(C(4096, 0, 1, 1, 0, 0, 1), 100003) == (100003 * 2048, 4096)


def test_output_sizes():
    assert tk.tk_swiglu_quant_output_sizes(D(), 8192) == (8192 * 2048, 8192 * 16 * 4)
    assert tk.tk_swiglu_quant_output_sizes(D(group_size=32, scale_fmt=1, out_fmt=1), 65536) == (
        65536 * 1024, 65536 * 64)
    assert tk.tk_swiglu_quant_output_sizes(D(group_size=0), 256) == (256 * 2048, 256 * 4)
    assert tk.tk_swiglu_quant_output_sizes(D(), 0) == (0, 0)
    with pytest.raises(tk.TkError):
        tk.tk_swiglu_quant_output_sizes(D(), -1)


def test_null_handling_and_status_strings():
    lib = _abi.lib()
    assert lib.tk_swiglu_quant_run(None, 4, None, None, None, None, None, None) == 1
    assert lib.tk_quant_cast_run(None, 4, None, None, None, None) == 1
    assert lib.tk_swiglu_quant_validate(None) == 1
    assert lib.tk_swiglu_quant_plan_destroy(None) == 0
    assert lib.tk_swiglu_quant_plan(ctypes.byref(D()), 0, None) == 1
    for s, n in _abi.STATUS_NAMES.items():
        assert tk.tk_status_string(s) == n


def test_plan_without_gpu_reports_cuda_error():
    try:
        import torch
        if torch.cuda.is_available():
            pytest.skip("a GPU is present")
    except ImportError:
        pass
    with pytest.raises(tk.TkError) as e:
        tk.tk_swiglu_quant_plan(D(), 0)
    assert e.value.status in (1, 4)


def test_reduce_validate():
    R = tk.MoeReduceDesc
    assert tk.tk_moe_reduce_validate(R(2048, 8, 0)) == 0
    assert tk.tk_moe_reduce_validate(R(7168, 8, 1)) == 0
    assert tk.tk_moe_reduce_validate(R(8192, 64, 0)) == 0
    assert tk.tk_moe_reduce_validate(R(0, 8, 0)) == 1
    assert tk.tk_moe_reduce_validate(R(2048, 0, 0)) == 1
    assert tk.tk_moe_reduce_validate(R(2048, 8, 2)) == 1
    assert tk.tk_moe_reduce_validate(R(2040, 8, 0)) == 2
    assert tk.tk_moe_reduce_validate(R(8208, 8, 0)) == 2
    assert tk.tk_moe_reduce_validate(R(2048, 65, 0)) == 2
    assert tk.tk_moe_reduce_validate(R(2064, 8, 1)) == 2


def test_backward_validate():
    B = tk.SwigluBackwardDesc
    v = tk.tk_swiglu_backward_validate
    # hidden, has_w, use_clamp, L, recompute, group, scale_fmt, out_fmt, layout
    assert v(B(2048, 1, 0, 0.0, 0, 0, 0, 0, 0)) == 0
    assert v(B(7168, 1, 1, 7.0, 0, 0, 0, 0, 0)) == 0
    assert v(B(128, 0, 0, 0.0, 0, 0, 0, 0, 0)) == 0
    assert v(B(2048, 1, 1, 7.0, 1, 128, 1, 0, 2)) == 0     # recompute, UE8M0, packed scales
    assert v(B(2048, 1, 0, 0.0, 1, 32, 1, 1, 0)) == 0      # recompute into E2M1
    assert v(B(0, 1, 0, 0.0, 0, 0, 0, 0, 0)) == 1
    assert v(B(2048, 2, 0, 0.0, 0, 0, 0, 0, 0)) == 1
    assert v(B(2048, 1, 1, -1.0, 0, 0, 0, 0, 0)) == 1      # clamp limit must be > 0
    assert v(B(2048, 1, 1, float("inf"), 0, 0, 0, 0, 0)) == 1
    assert v(B(96, 1, 0, 0.0, 0, 0, 0, 0, 0)) == 2         # neither a small power of two nor % 512
    assert v(B(3000, 1, 0, 0.0, 0, 0, 0, 0, 0)) == 2
    assert v(B(16384, 1, 0, 0.0, 0, 0, 0, 0, 0)) == 2      # above 8192
    assert v(B(2048, 1, 0, 0.0, 1, 0, 0, 0, 0)) == 2       # recompute needs a group size
    assert v(B(2048, 1, 0, 0.0, 1, 128, 0, 0, 2)) == 2     # packed layout needs UE8M0


def test_unanswered_wait_rejects_tries_out_of_range():
    # checked on the host before any device is touched
    for tries in (0, (1 << 22) + 1):
        with pytest.raises(tk.TkError) as e:
            tk.tk_diag_unanswered_wait(0, tries, None)
        assert e.value.status == 1


def _enum_values(name):
    """{constant: value} of `typedef enum <name> {...}` in the header."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    body = re.search(r"typedef enum %s \{(.*?)\}" % name, text, flags=re.S).group(1)
    return {k: int(v) for k, v in re.findall(r"\b(TK_[A-Z0-9_]+)\s*=\s*(\d+)", body)}


def test_binding_tables_match_the_header_enums():
    """The Python binding's name tables carry the header's enum values, so a
    value added or renumbered on one side only fails here."""
    assert {v: k for k, v in _abi.STATUS_NAMES.items()} == _enum_values("tk_status")
    assert _enum_values("tk_scale_fmt") == {"TK_SCALE_" + k.upper(): v for k, v in _abi.SCALE_FMTS.items()}
    assert _enum_values("tk_out_fmt") == {"TK_OUT_" + k.upper(): v for k, v in _abi.OUT_FMTS.items()}
    assert _enum_values("tk_in_dtype") == {"TK_IN_" + k.upper(): v for k, v in _abi.IN_DTYPES.items()}
    assert sorted(_enum_values("tk_scale_layout").values()) == sorted(_abi.SCALE_LAYOUTS.values())
    assert sorted(_enum_values("tk_granularity").values()) == sorted(_abi.GRANULARITIES.values())
    assert sorted(_enum_values("tk_reduce_in_fmt").values()) == sorted(_abi.REDUCE_IN_FMTS.values())
    kinds = _enum_values("tk_kernel_kind")
    assert sorted(kinds.values()) == sorted(_abi.KERNEL_NAMES)
    assert kinds["TK_KERNEL_BLOCK_RING"] == 2 and _abi.KERNEL_NAMES[2] == "block_stream_kernel"
    forms = _enum_values("tk_cast_form")
    assert sorted(forms.values()) == sorted(_abi.CAST_FORMS)
    assert _abi.CAST_FORMS[forms["TK_CAST_ROWS"]] == "row_quant_kernel"
    assert _abi.CAST_FORMS[forms["TK_CAST_BLOCK_RING"]] == "block_stream_kernel"
    assert _abi.CAST_FORMS[forms["TK_CAST_WARP_STREAM"]] == "warp_stream_kernel"
    assert "col_chunk_quant_kernel" in _abi.CAST_FORMS[forms["TK_CAST_CHANNEL_CHUNK"]]
    assert "col_scale_kernel" in _abi.CAST_FORMS[forms["TK_CAST_CHANNEL_SPLIT"]]
