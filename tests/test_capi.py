"""The C-ABI library builds, loads, exports every symbol include/minite.h
declares, and rejects bad arguments on the host. No GPU needed (no kernel is
launched: every call here fails validation before reaching the device)."""
import ctypes
import os
import re

import pytest

from nvfp4_w4a4_moe_permute_gb300 import build as B
from nvfp4_w4a4_moe_permute_gb300 import minite as M

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "minite.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return M.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(minite_\w+)\s*\(", src)))


def test_header_declares_the_path_entry_points():
    names = declared_functions()
    for n in ["minite_quantize_nvfp4", "minite_moe_permute_quant", "minite_grouped_gemm_nvfp4",
              "minite_swiglu_weighted_quant", "minite_swiglu_backward_quant",
              "minite_moe_combine"]:
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n
    assert set(declared_functions()) == set(M.EXPORTS)


def test_status_strings_and_version(lib):
    assert M.minite_status_string(0) == "ok"
    assert M.minite_status_string(4).startswith("device pipeline wait")
    assert M.minite_status_string(99) == "unknown status"
    assert re.match(r"^\d+\.\d+\.\d+$", M.minite_version())


def test_workspace_sizes(lib):
    assert M.minite_workspace_bytes(M.OP_QUANTIZE, 128) == 512
    a = M.minite_workspace_bytes(M.OP_PERMUTE_QUANT, 4096, 2048, 128, 8)
    b = M.minite_workspace_bytes(M.OP_PERMUTE_QUANT, 8192, 2048, 128, 8)
    assert 0 < a < b
    # the token-order scale staging grows with H
    assert M.minite_workspace_bytes(M.OP_PERMUTE_QUANT, 4096, 4096, 128, 8) > a
    assert M.minite_workspace_bytes(99, 1) == 0
    # token-order scales (T x H/16 bytes) and global scales (T floats)
    assert M.minite_workspace_bytes(M.OP_COMBINE_BACKWARD_QUANT, 4096, 2048) == 4096 * 128 + 4096 * 4
    assert M.minite_workspace_bytes(M.OP_COMBINE_BACKWARD_QUANT, 0, 2048) == 0
    assert M.minite_workspace_bytes(M.OP_QUANTIZE_TOKENS, 128) == 512
    # plus one float per source row when rows are gathered
    assert M.minite_workspace_bytes(M.OP_QUANTIZE_TOKENS, 128, 1000) == 512 + 4000
    assert M.minite_workspace_bytes(M.OP_QUANTIZE_TOKENS, 2000) == 0


def _c(lib, name):
    return getattr(lib, name)


def test_host_validation_rejects_bad_arguments(lib):
    vp = ctypes.c_void_p
    fake = vp(4096)  # never dereferenced: validation fails first
    # null input
    assert lib.minite_quantize_nvfp4(None, 1, 16, 64, 0, 0, None, fake, fake, fake, None, 0, None, None) == 1
    # bad scale mode
    assert lib.minite_quantize_nvfp4(fake, 1, 16, 64, 7, 0, None, fake, fake, fake, None, 0, None, None) == 1
    # cols not a multiple of 16
    assert lib.minite_quantize_nvfp4(fake, 1, 16, 40, 0, 0, None, fake, fake, fake, None, 0, None, None) == 2
    # per-row scales with the transposed layout are not supported
    assert lib.minite_quantize_nvfp4(fake, 1, 16, 64, 0, 1, None, fake, fake, fake, None, 0, None, None) == 2
    # per-group without gscale_in needs a workspace
    assert lib.minite_quantize_nvfp4(fake, 1, 16, 64, 1, 0, None, fake, fake, fake, None, 0, None, None) == 1
    # two-orientation weight quantization: rows not a multiple of 16, no workspace
    assert lib.minite_quantize_nvfp4_dual(fake, 1, 24, 64, fake, fake, fake, fake, fake, fake, 512,
                                          None, None) == 2
    assert lib.minite_quantize_nvfp4_dual(fake, 1, 32, 64, fake, fake, fake, fake, fake, None, 0,
                                          None, None) == 1
    # permute: H not a multiple of 64, too many experts, misaligned x
    args = [fake, fake, None, 16, 96, 4, 2] + [fake] * 7 + [None, fake, 1 << 20, None, None]
    assert lib.minite_moe_permute_quant(*args) == 2
    args = [fake, fake, None, 16, 128, 2000, 2] + [fake] * 7 + [None, fake, 1 << 20, None, None]
    assert lib.minite_moe_permute_quant(*args) == 2
    args = [vp(4098), fake, None, 16, 128, 4, 2] + [fake] * 7 + [None, fake, 1 << 20, None, None]
    assert lib.minite_moe_permute_quant(*args) == 1
    # permute: workspace too small
    args = [fake, fake, None, 16, 128, 4, 2] + [fake] * 7 + [None, fake, 8, None, None]
    assert lib.minite_moe_permute_quant(*args) == 1
    # gemm: K not a multiple of 64, N not a multiple of 32, bad out dtype
    g = [fake] * 8
    assert lib.minite_grouped_gemm_nvfp4(*g, 128, 128, 96, 1, fake, 0, None, None) == 2
    assert lib.minite_grouped_gemm_nvfp4(*g, 128, 100, 128, 1, fake, 0, None, None) == 2
    assert lib.minite_grouped_gemm_nvfp4(*g, 128, 128, 128, 1, fake, 5, None, None) == 1
    assert lib.minite_grouped_gemm_nvfp4(*g, 128, 128, 128, 1, None, 0, None, None) == 1
    # swiglu: I not a multiple of 64
    assert lib.minite_swiglu_weighted_quant(fake, None, 16, 96, 1, fake, fake, fake, fake, fake, None, None) == 2
    # swiglu backward: I too large, dh missing, misaligned dh
    assert lib.minite_swiglu_backward_quant(fake, fake, None, 16, 4096, 1, fake, fake, fake, fake,
                                            fake, None, None) == 2
    assert lib.minite_swiglu_backward_quant(fake, None, None, 16, 128, 1, fake, fake, fake, fake,
                                            fake, None, None) == 1
    assert lib.minite_swiglu_backward_quant(fake, vp(4112), None, 16, 128, 1, fake, fake, fake,
                                            fake, fake, None, None) == 1
    # combine backward: H not a multiple of 64, no workspace, workspace too small
    cb = lambda T, H, E, k, ws, n: lib.minite_moe_combine_backward_quant(  # noqa: E731
        fake, T, H, E, k, fake, fake, fake, fake, fake, fake, fake, ws, n, None, None)
    assert cb(16, 96, 2, 2, fake, 1 << 20) == 2
    assert cb(16, 128, 2, 2, None, 1 << 20) == 1
    assert cb(16, 128, 2, 2, fake, 8) == 1
    # token-axis quantizer: C not a multiple of 16, k_cap not a multiple of 256, misaligned
    # codes, misaligned row maxima
    qt = lambda C, kcap, codes, ra=None: lib.minite_quantize_tokens_nvfp4(  # noqa: E731
        fake, 64, None, ra, 64, C, 2, fake, kcap, codes, fake, fake, fake, fake, 1024, None, None)
    assert qt(40, 1024, fake) == 2
    assert qt(64, 1000, fake) == 2
    assert qt(64, 1024, vp(4112)) == 1
    assert qt(64, 1024, fake, vp(4098)) == 1
    # weight-gradient GEMM: N not a multiple of 32, bad out dtype
    wg = lambda N, dt: lib.minite_grouped_gemm_wgrad_nvfp4(  # noqa: E731
        fake, fake, fake, fake, fake, fake, fake, 2, 128, N, 1024, fake, dt, None, None)
    assert wg(100, 0) == 2
    assert wg(128, 7) == 1
    # SwiGLU keeping h: h_out missing; misaligned row maxima
    assert lib.minite_swiglu_weighted_quant_keep_h(fake, None, 16, 128, 1, fake, fake, fake, fake,
                                                   fake, None, None, None, None) == 1
    assert lib.minite_swiglu_weighted_quant_keep_h(fake, None, 16, 128, 1, fake, fake, fake, fake,
                                                   fake, fake, vp(4098), None, None) == 1
    # SwiGLU backward keeping [dg | du]: dgu_out missing; misaligned row maxima
    assert lib.minite_swiglu_backward_quant_keep(fake, fake, None, 16, 128, 1, fake, fake, fake,
                                                 fake, fake, None, None, None, None) == 1
    assert lib.minite_swiglu_backward_quant_keep(fake, fake, None, 16, 128, 1, fake, fake, fake,
                                                 fake, fake, fake, vp(4098), None, None) == 1
    # combine: N not a multiple of 8, k too large
    assert lib.minite_moe_combine(fake, fake, 4, 8, 12, 2, fake, None, None) == 2
    assert lib.minite_moe_combine(fake, fake, 4, 8, 16, 64, fake, None, None) == 2
    assert lib.minite_test_convert(None, 4, None, None, None, None) == 1


def test_python_binding_fails_loudly_without_library(tmp_path):
    import importlib
    saved = M._LIB
    try:
        M._LIB = None
        with pytest.raises(M.MiniteError):
            M.load(str(tmp_path / "missing.so"))
    finally:
        M._LIB = saved
