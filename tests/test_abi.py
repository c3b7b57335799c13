"""Host-side checks of the C ABI: the library builds, loads and exports every declared entry
point; argument validation; the tile order against the oracle's.  No kernel is launched."""
import os
import random
import re

import pytest

from conftest import ROOT, read_golden

fg = pytest.importorskip("gemm_epilogue_gb300.binding")


@pytest.fixture(scope="module")
def lib():
    from gemm_epilogue_gb300 import build
    build.build()
    return fg.lib()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "fgemm.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\**\s+\**(fgemm_[a-z0-9_]+)\s*\(",
                                 text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for want in ("fgemm_bias_relu", "fgemm_addmm_gate", "fgemm_unfused_bias_relu",
                 "fgemm_unfused_addmm_gate", "fgemm_device_status"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(declared_functions()) <= set(fg._SIGS)


def test_library_has_sm103a_code_only_build_flags():
    from gemm_epilogue_gb300 import build
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_status_strings(lib):
    assert fg.fgemm_status_string(0) == "FGEMM_OK"
    assert fg.fgemm_status_string(6) == "FGEMM_ERR_TIMEOUT"
    assert fg.fgemm_status_string(99) == "FGEMM_ERR_UNKNOWN"


def test_tile_order_matches_oracle_and_golden(lib):
    from oracle import schedule
    g = read_golden("grouped_order_3x2_g2.txt")
    assert [fg.fgemm_tile_of(p, 3, 2, 2) for p in range(6)] == \
        [tuple(int(v) for v in g[str(p)].split(",")) for p in range(6)]
    rnd = random.Random(1)
    for _ in range(100):
        tm, tn, grp = rnd.randint(1, 40), rnd.randint(1, 40), rnd.randint(1, 10)
        assert [fg.fgemm_tile_of(p, tm, tn, grp) for p in range(tm * tn)] == schedule.order(tm, tn, grp)
    # the shapes of the measured workloads (128 x 256 tiles)
    for tm, tn in [(32, 16), (8, 85), (64, 56), (2, 1)]:
        for grp in (1, 4, 8):
            assert [fg.fgemm_tile_of(p, tm, tn, grp) for p in range(tm * tn)] == schedule.order(tm, tn, grp)


def test_tile_of_rejects_out_of_range(lib):
    assert fg.call_status("fgemm_tile_of", 6, 3, 2, 2, None, None) == fg.ERR_INVALID_VALUE
    import ctypes
    m, n = ctypes.c_int64(), ctypes.c_int64()
    assert fg.call_status("fgemm_tile_of", 6, 3, 2, 2, ctypes.byref(m), ctypes.byref(n)) == fg.ERR_INVALID_VALUE
    assert fg.call_status("fgemm_tile_of", 0, 3, 2, 0, ctypes.byref(m), ctypes.byref(n)) == fg.ERR_INVALID_VALUE


# Validation: every case below returns before any device is touched, so no pointer is used.
# Real-looking pointers would be dereferenced only after validation passes, so the cases that
# pass validation are left to the GPU tests.

def test_empty_problems_return_ok_without_launch(lib):
    import ctypes
    taken = ctypes.c_int(-1)
    assert fg.call_status("fgemm_bias_relu_ex", None, None, None, None, 0, 16, 8, fg.BF16, None,
                          None, ctypes.byref(taken)) == fg.OK
    assert taken.value == fg.PATH_NONE
    assert fg.call_status("fgemm_addmm_gate", None, None, None, None, None, 5, 0, 8, fg.F16, None) == fg.OK


def test_negative_or_huge_sizes(lib):
    assert fg.call_status("fgemm_bias_relu", None, None, None, None, -1, 4, 4, fg.F16, None) == fg.ERR_INVALID_VALUE
    assert fg.call_status("fgemm_bias_relu", None, None, None, None, 4, 4, -2, fg.F16, None) == fg.ERR_INVALID_VALUE
    assert fg.call_status("fgemm_bias_relu", None, None, None, None, 1 << 31, 4, 4, fg.F16, None) == fg.ERR_INVALID_VALUE


def test_unknown_dtypes(lib):
    for d in (0, 0x3, 0x20, 0x200, 0x1000, -1, fg.F16 | 0x30):
        assert fg.call_status("fgemm_bias_relu", None, None, None, None, 4, 4, 4, d, None) == fg.ERR_UNSUPPORTED_DTYPE


def test_null_pointers(lib):
    # out missing, bias missing, Y missing (gate), A/B missing with K > 0
    assert fg.call_status("fgemm_bias_relu", 4096, 4096, 4096, None, 4, 4, 4, fg.F16, None) == fg.ERR_INVALID_VALUE
    assert fg.call_status("fgemm_bias_relu", 4096, 4096, None, 4096, 4, 4, 4, fg.F16, None) == fg.ERR_INVALID_VALUE
    assert fg.call_status("fgemm_addmm_gate", 4096, 4096, 4096, None, 4096, 4, 4, 4, fg.F16, None) == fg.ERR_INVALID_VALUE
    assert fg.call_status("fgemm_bias_relu", None, 4096, 4096, 4096, 4, 4, 4, fg.F16, None) == fg.ERR_INVALID_VALUE


def test_misaligned_pointers(lib):
    # odd byte addresses for 16-bit data, 2-byte-aligned for fp32 bias / out
    assert fg.call_status("fgemm_bias_relu", 4097, 4096, 4096, 4096, 4, 4, 4, fg.F16, None) == fg.ERR_MISALIGNED
    assert fg.call_status("fgemm_bias_relu", 4096, 4096, 4098, 4096, 4, 4, 4, fg.BF16 | fg.BIAS_F32, None) == fg.ERR_MISALIGNED
    assert fg.call_status("fgemm_bias_relu", 4096, 4096, 4096, 4098, 4, 4, 4, fg.BF16 | fg.OUT_F32, None) == fg.ERR_MISALIGNED
    assert fg.call_status("fgemm_addmm_gate", 4096, 4096, 4096, 4097, 4096, 4, 4, 4, fg.F16, None) == fg.ERR_MISALIGNED


def test_bad_options(lib):
    import ctypes
    for field, val in (("group_m", -1), ("path", 9), ("split_k", 9), ("max_ctas", -3), ("timeout_ms", -1),
                       ("cta_pair", 3), ("tail_split", 2), ("skinny_tiles", 3), ("stages", 9),
                       ("inject_stall", 2), ("bias_init", 3), ("full_last_n", -1), ("y_blocks", 4),
                       ("k_rows", 3), ("bias_mma", 3), ("bias_mma", -1), ("pdl", 3), ("raster", 2), ("epi_warps", 12)):
        o = fg.Opts()
        setattr(o, field, val)
        st = fg.call_status("fgemm_bias_relu_ex", 4096, 4096, 4096, 4096, 4, 4, 4, fg.F16, None,
                            ctypes.byref(o), None)
        assert st == fg.ERR_INVALID_VALUE, field


def test_unfused_workspace_size(lib):
    assert fg.fgemm_unfused_workspace_bytes(4096, 4096, fg.BF16, 0) == 4096 * 4096 * 2
    assert fg.fgemm_unfused_workspace_bytes(4096, 4096, fg.BF16, 1) == 4096 * 4096 * 4
    assert fg.fgemm_unfused_workspace_bytes(3, 5, fg.F16, 0) == 256
    assert fg.fgemm_unfused_workspace_bytes(3, 5, 0x7, 0) == 0
    assert fg.call_status("fgemm_unfused_bias_relu", 4096, 4096, 4096, 4096, 4, 4, 4, fg.F16, None,
                          0, 0, None) == fg.ERR_WORKSPACE


@pytest.mark.skipif(__import__("torch").cuda.is_available(), reason="checks the no-GPU answer")
def test_no_device_is_reported_without_a_gpu(lib):
    # all arguments valid; the call reaches the device check and stops there
    st = fg.call_status("fgemm_bias_relu", 4096, 4096, 4096, 4096, 4, 4, 4, fg.F16, None)
    assert st == fg.ERR_NO_DEVICE


def test_second_operand_type_rules(lib):
    # the gate / residual's Y type: 16-bit, and a 16-bit output has Y's type; other entries refuse
    # the Y bits.  Refused before any device is touched.
    bad = [("fgemm_addmm_gate", fg.E4M3 | fg.BIAS_F32 | fg.OUT_F16),                 # Y would be fp8
           ("fgemm_addmm_gate", fg.E4M3 | fg.BIAS_F32 | fg.OUT_BF16 | fg.Y_F16),     # out != Y
           ("fgemm_addmm_gate", fg.F16 | fg.OUT_BF16),                               # out != Y (f16)
           ("fgemm_bias_residual_relu", fg.BF16 | fg.Y_F16),                          # out bf16, R f16
           ("fgemm_addmm_gate", fg.F16 | 0x3000)]                                    # unknown Y code
    for name, word in bad:
        assert fg.call_status(name, None, None, None, None, None, 4, 4, 4, word, None) == \
            fg.ERR_UNSUPPORTED_DTYPE, (name, hex(word))
    assert fg.call_status("fgemm_bias_relu", None, None, None, None, 4, 4, 4,
                          fg.F16 | fg.Y_BF16, None) == fg.ERR_UNSUPPORTED_DTYPE
    # accepted words (the call then fails on the NULL buffers, not on the type)
    for word in (fg.E4M3 | fg.BIAS_F32 | fg.OUT_F16 | fg.Y_F16,
                 fg.E4M3 | fg.BIAS_BF16 | fg.OUT_F32 | fg.Y_BF16, fg.F16 | fg.Y_BF16 | fg.OUT_BF16):
        assert fg.call_status("fgemm_addmm_gate", None, None, None, None, None, 4, 4, 4, word,
                              None) == fg.ERR_INVALID_VALUE, hex(word)
