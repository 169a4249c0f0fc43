"""Host-side helpers of bench.py that need no GPU: the device-code hash that
decides whether a committed ncu summary still describes the running kernels."""
import bench


def test_code_only_drops_comments_and_layout_but_keeps_literals():
    src = 'int a = 1;   // note\n/* block\n comment */  asm("x // y"); char c = \'/\';\nint  b;'
    assert bench._code_only(src) == 'int a = 1; asm("x // y"); char c = \'/\'; int b;'
    # an escaped quote does not end a string literal
    assert bench._code_only('s = "a\\" // b"; // c') == 's = "a\\" // b";'


def test_hash_is_stable_under_comment_edits(tmp_path, monkeypatch):
    csrc = tmp_path / "activation_fp8_quantization_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text("__global__ void k() { int a = 1; }\n")
    (csrc / "tk_api.cu").write_text("int host_side = 0;\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_hash()
    (csrc / "k.cu").write_text("// a kernel\n__global__ void k() {\n    int a = 1;   /* one */\n}\n")
    assert bench.kernel_source_hash() == h0
    (csrc / "tk_api.cu").write_text("int host_side = 1;\n")        # host code is not hashed
    assert bench.kernel_source_hash() == h0
    (csrc / "k.cu").write_text("__global__ void k() { int a = 2; }\n")
    assert bench.kernel_source_hash() != h0


def test_family_hash_covers_only_its_sources(tmp_path, monkeypatch):
    csrc = tmp_path / "activation_fp8_quantization_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for name in ("tk_kernels.cuh", "tk_internal.h", "tk_swiglu_kernels.cu", "tk_channel_kernels.cu"):
        (csrc / name).write_text("int %s = 0;\n" % name.split(".")[0])
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench.kernel_source_hash("swiglu_quant")
    (csrc / "tk_channel_kernels.cu").write_text("int changed = 1;\n")   # another family's file
    assert bench.kernel_source_hash("swiglu_quant") == h
    (csrc / "tk_kernels.cuh").write_text("int changed = 2;\n")          # a shared header
    assert bench.kernel_source_hash("swiglu_quant") != h


def test_family_sources_exist_and_cover_every_kernel_file():
    """Every kernel file belongs to some profile family, and every family's
    files exist, so a committed profile's hash always names real sources."""
    import os
    csrc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                        "activation_fp8_quantization_gb300", "csrc")
    listed = set()
    for fam, files in bench.FAMILY_SOURCES.items():
        for f in files:
            assert os.path.exists(os.path.join(csrc, f)), (fam, f)
            listed.add(f)
    kernels = {n for n in os.listdir(csrc) if n.endswith("_kernels.cu") and n != "tk_diag_kernels.cu"}
    assert kernels <= listed, kernels - listed
    assert set(bench.PROFILE_FAMILY.values()) == set(bench.FAMILY_SOURCES)
