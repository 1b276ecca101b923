"""The C-ABI library: it loads without a GPU, exports every entry point that include/moe4.h
declares, and rejects bad arguments on the host before any CUDA call (sizes, flags, alignment,
missing workspace).  No compute call is made here."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe4.h")


@pytest.fixture(scope="module")
def lib():
    from precision_moe_numerics_03_b300 import build, moe4
    build.build()
    return moe4.load()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?(?:int|size_t|char)\s*\*?\s*(\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = _declared()
    for required in ["nvfp4_quantize", "mxfp8_requant_transpose_sr", "grouped_expert_gemm_nvfp4",
                     "grouped_gemm_mxfp8", "hadamard_quant", "hadamard_dequant"]:
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    from precision_moe_numerics_03_b300 import moe4
    names = _declared()
    assert len(names) >= 20
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(moe4.exported_symbols()) == names


def test_host_side_queries(lib):
    assert lib.moe4_version() >= 100
    assert lib.moe4_status_string(0) == b"ok"
    assert b"argument" in lib.moe4_status_string(-1)
    assert lib.moe4_workspace_size(1, 384, 0, 0) == 384 * 4
    assert lib.moe4_workspace_size(2, 0, 0, 0) == 4
    assert lib.moe4_workspace_size(3, 16384, 8, 384) == (128 * 384 + 384) * 4
    assert lib.moe4_workspace_size_gemm(0, 256, 1, 256, 512) == 256 * 32 * 2


FAKE = 1 << 20          # a 16-byte aligned address that is never dereferenced
MISALIGNED = FAKE + 4


@pytest.mark.parametrize("case", [
    # (entry point, arguments) -- each must fail its host-side checks
    ("nvfp4_quantize", (FAKE, 1, 16, 15, 16, FAKE, FAKE, FAKE, None, 1, FAKE, 64, None)),   # cols % 16
    ("nvfp4_quantize", (FAKE, 1, 16, 16, 8, FAKE, FAKE, FAKE, None, 1, FAKE, 64, None)),    # ld < cols
    ("nvfp4_quantize", (MISALIGNED, 1, 16, 16, 16, FAKE, FAKE, FAKE, None, 1, FAKE, 64, None)),
    ("nvfp4_quantize", (FAKE, 1, 16, 16, 16, FAKE, FAKE, FAKE, None, 1 << 30, FAKE, 64, None)),  # bad flag
    ("nvfp4_quantize", (FAKE, 1, 16, 16, 16, FAKE, FAKE, FAKE, None, 2, FAKE, 64, None)),   # AMAX_GIVEN, no amax
    ("nvfp4_quantize", (FAKE, 65536, 16, 16, 16, FAKE, FAKE, FAKE, None, 1, FAKE, 1 << 20, None)),  # amax pass grid
    ("nvfp4_quantize_f32", (FAKE, 65536, 16, 16, 16, FAKE, FAKE, FAKE, None, 1, FAKE, 1 << 20, None)),
    ("nvfp4_dequantize", (FAKE, FAKE, FAKE, 1, 16, 16, FAKE, 0x200 | 0x10000, None)),          # canonical sf only
    ("nvfp4_dequantize", (FAKE, FAKE, FAKE, 1, 16, 16, FAKE, 0x300, None)),                    # two outputs
    ("mxfp8_requant_transpose_sr", (FAKE, FAKE, FAKE, 1, 48, 64, FAKE, FAKE, 0, 0, 4, None)),  # rows % 32
    ("mxfp8_quantize", (FAKE, 32, 64, FAKE, FAKE, 0, 0, 0x30, None)),                        # both layouts
    ("mxfp8_quantize_rowcol", (FAKE, 48, 64, FAKE, FAKE, FAKE, FAKE, 0, None)),                # rows % 32
    ("mxfp8_quantize_rowcol", (FAKE, 32, 64, FAKE, FAKE, FAKE, FAKE, 0x4, None)),              # no SR
    ("mxfp8_quantize_rowcol", (FAKE, 32, 64, MISALIGNED, FAKE, FAKE, FAKE, 0, None)),          # q_row align
    ("moe4_swiglu_backward_mxfp8", (FAKE, FAKE, 48, 64, FAKE, FAKE, FAKE, FAKE, 0, None)),        # rows % 32
    ("moe4_swiglu_backward_mxfp8", (FAKE, FAKE, 32, 48, FAKE, FAKE, FAKE, FAKE, 0, None)),        # f % 32
    ("moe4_swiglu_backward_mxfp8", (FAKE, MISALIGNED, 32, 64, FAKE, FAKE, FAKE, FAKE, 0, None)),  # dh alignment
    ("moe4_combine_backward_mxfp8", (FAKE, FAKE, FAKE, FAKE, 4, 8, 48, 128, FAKE, FAKE, FAKE, FAKE, 0, None)),  # d % 32
    ("moe4_combine_backward_mxfp8", (FAKE, FAKE, FAKE, FAKE, 4, 40, 64, 128, FAKE, FAKE, FAKE, FAKE, 0, None)),  # k > 32
    ("moe4_combine_backward_mxfp8", (FAKE, FAKE, FAKE, FAKE, 4, 8, 64, 100, FAKE, FAKE, FAKE, FAKE, 0, None)),  # rows % 32
    ("hadamard_quant", (FAKE, 4, 64, FAKE, FAKE, FAKE, 1, FAKE, 4, None)),                   # cols % 128
    ("hadamard_quant", (FAKE, 4, 128, FAKE, FAKE, FAKE, 1 | 0x10000, FAKE, 4, None)),         # bad flag
    ("grouped_expert_gemm_nvfp4_hadamard_amax", (FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 128, 256, 256, FAKE,
                                                 None, 0, None, 0, None)),                    # no amax_out
    ("grouped_expert_gemm_nvfp4_hadamard_amax", (FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 128, 256, 256, FAKE,
                                                 FAKE, 0x200, None, 0, None)),                # output flag
    ("grouped_gemm_mxfp8_swiglu_backward", (FAKE, FAKE, FAKE, FAKE, FAKE, 1, 128, 128, 256, FAKE, FAKE, 0, None, 0,
                                            None)),                                           # f % 256
    ("grouped_gemm_mxfp8_swiglu_backward", (FAKE, FAKE, FAKE, FAKE, FAKE, 1, 128, 256, 256, None, FAKE, 0, None, 0,
                                            None)),                                           # no gu
    ("grouped_gemm_mxfp8_swiglu_backward", (FAKE, FAKE, FAKE, FAKE, FAKE, 1, 128, 256, 256, FAKE, MISALIGNED, 0,
                                            None, 0, None)),                                  # dgu alignment
    ("grouped_gemm_mxfp8_swiglu_backward", (FAKE, FAKE, FAKE, FAKE, FAKE, 1, 128, 256, 256, FAKE, FAKE, 0x1000,
                                            None, 0, None)),                                  # bad flag
    ("grouped_expert_gemm_nvfp4_swiglu", (FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 128, 192, 256, FAKE, FAKE,
                                          FAKE, 0, None, 0, None)),                           # f % 128
    ("grouped_expert_gemm_nvfp4_swiglu", (FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 128, 128, 256, FAKE, None,
                                          FAKE, 0, None, 0, None)),                           # no h
    ("grouped_expert_gemm_nvfp4_swiglu", (FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 128, 128, 256, FAKE,
                                          MISALIGNED, FAKE, 0, None, 0, None)),               # h alignment
    ("grouped_expert_gemm_nvfp4_swiglu", (FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 128, 128, 256, FAKE, FAKE,
                                          FAKE, 0x100, None, 0, None)),                       # output flag
    ("grouped_expert_gemm_nvfp4_hadamard_mx", (FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 128, 200, 256, FAKE,
                                               FAKE, 0, None, 0, None)),                      # N % 256
    ("grouped_expert_gemm_nvfp4_hadamard_mx", (FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 128, 256, 256,
                                               MISALIGNED, FAKE, 0, None, 0, None)),          # q alignment
    ("grouped_expert_gemm_nvfp4_hadamard_mx", (FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 128, 256, 256, FAKE,
                                               FAKE, 0x100, None, 0, None)),                  # output flag
    ("grouped_expert_gemm_nvfp4", (FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 100, 256, 256, FAKE, 0x100,
                                   None, 0, None)),                                          # rows % 128
    ("grouped_expert_gemm_nvfp4", (FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 128, 256, 256, FAKE, 0x300,
                                   None, 0, None)),                                          # two outputs
    ("grouped_gemm_mxfp8", (FAKE, FAKE, FAKE, FAKE, FAKE, 1, 128, 256, 128, FAKE, 0x100 | 0x1000 | 0x2000,
                            None, 0, None)),                                                 # both groupings
    ("grouped_gemm_mxfp8", (FAKE, FAKE, FAKE, FAKE, FAKE, 1, 128, 256, 128, FAKE, 0x200 | 0x2000 | 0x4000,
                            None, 0, None)),                                                 # bf16 accumulate
    ("grouped_gemm_mxfp8", (FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 14, 1 << 17, 256, 128, FAKE, 0x100 | 0x2000,
                            None, 0, None)),                                                 # E*M past int32
    ("moe4_route_topk", (FAKE, 4, 8, 40, FAKE, FAKE, None)),                                 # k > 32
    ("moe4_permute_plan", (FAKE, 4, 2, 8, FAKE, FAKE, FAKE, 10, FAKE, 1 << 20, None)),       # rows_cap too small
    ("moe4_permute_plan", (FAKE, 1 << 28, 8, 8, FAKE, FAKE, FAKE, 1 << 32, FAKE, 1 << 40, None)),  # rows past int32
    ("moe4_combine", (FAKE, FAKE, FAKE, 4, 40, 16, FAKE, None)),                             # k > 32
    ("moe4_swiglu", (FAKE, 4, 6, FAKE, None)),                                               # f % 4
    ("moe4_swiglu_amax", (FAKE, 4, 8, FAKE, None, None)),                                    # no amax_out
    ("moe4_swiglu_amax", (FAKE, 4, 8, FAKE, FAKE + 2, None)),                                # amax alignment
    ("moe4_combine", (FAKE, FAKE, FAKE, 4, 2, 12, FAKE, None)),                              # d % 8
    ("moe4_dispatch_backward", (FAKE, FAKE, 4, 40, 16, FAKE, None)),                         # k > 32
    ("moe4_combine_hadamard", (FAKE, FAKE, FAKE, FAKE, FAKE, 4, 8, 64, FAKE, None)),          # d % 128
    ("moe4_combine_hadamard", (FAKE, FAKE, FAKE, FAKE, FAKE, 4, 33, 128, FAKE, None)),        # k > 32
    ("moe4_dispatch_backward", (FAKE, FAKE, 4, 2, 16, MISALIGNED, None)),                    # dx alignment
    ("moe4_sgd_update", (FAKE, FAKE, 6, 0.1, FAKE, None)),                                   # n % 4
    ("moe4_sf_to_mma_layout", (FAKE, 1, 100, 4, FAKE, None)),                                # rows % 128
    ("moe4_convert", (7, FAKE, 4, FAKE, None)),                                              # bad kind
    ("moe4_convert", (2, FAKE, 4, MISALIGNED, None)),                                        # bf16 out align 8
    # output scales in the tile layout need whole 128-row tiles and groups of four blocks
    ("mxfp8_requant_transpose_sr", (FAKE, FAKE, FAKE, 1, 96, 128, FAKE, FAKE, 0, 0, 0x40000, None)),  # rows % 128
    ("mxfp8_requant_transpose_sr", (FAKE, FAKE, FAKE, 1, 128, 64, FAKE, FAKE, 0, 0, 0x40000, None)),  # cols % 128
    ("mxfp8_quantize_rowcol", (FAKE, 96, 128, FAKE, FAKE, FAKE, FAKE, 0x40000, None)),          # rows % 128
    ("moe4_swiglu_backward_mxfp8", (FAKE, FAKE, 128, 32, FAKE, FAKE, FAKE, FAKE, 0x40000, None)),  # f % 64
    ("moe4_combine_backward_mxfp8", (FAKE, FAKE, FAKE, FAKE, 4, 8, 64, 128, FAKE, FAKE, FAKE, FAKE, 0x40000,
                                     None)),                                                  # d % 128
    ("mxfp8_quantize", (FAKE, 128, 128, FAKE, FAKE, 0, 0, 0x10 | 0x40000, None)),             # not offered
    # the fused weight path: cols % 64, rows % 32, no amax, tile layouts on 128-row tiles
    ("nvfp4_quantize_f32_requant", (FAKE, 1, 128, 96, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, 0, 0, None, 5, None)),
    ("nvfp4_quantize_f32_requant", (FAKE, 1, 48, 128, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, 0, 0, None, 5, None)),
    ("nvfp4_quantize_f32_requant", (FAKE, 1, 128, 128, None, FAKE, FAKE, FAKE, FAKE, FAKE, 0, 0, 0, None, 5, None)),
    ("nvfp4_quantize_f32_requant", (FAKE, 1, 96, 128, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, 0, 0, None, 0x10005,
                                    None)),
    ("nvfp4_quantize_f32_requant", (FAKE, 1, 128, 64, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, 0, 0, None, 0x40005,
                                    None)),
    ("nvfp4_quantize_f32_requant", (FAKE, 1, 128, 128, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, 0, 0, None, 0x100,
                                    None)),                                                   # bad flag
    ("nvfp4_quantize_f32_requant", (FAKE, 1, 128, 128, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, 0, 0, None,
                                    0x300005, None)),                                         # both passes alone
    ("nvfp4_quantize_f32_requant", (FAKE, 1, 128, 128, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, 0, -1, None, 5,
                                    None)),                                                   # mat_base < 0
])
def test_argument_checks_fail_on_host(lib, case):
    name, args = case
    assert getattr(lib, name)(*args) == -1


def test_missing_workspace_is_reported(lib):
    # nvfp4_quantize without AMAX_GIVEN and without ws -> MOE4_ERR_WORKSPACE, before any launch
    assert lib.nvfp4_quantize(FAKE, 1, 16, 16, 16, FAKE, FAKE, FAKE, None, 1, None, 0, None) == -5
    assert lib.hadamard_quant(FAKE, 4, 128, FAKE, FAKE, FAKE, 1, None, 0, None) == -5
    # the GEMMs with canonical scales need room for their tensor-core copies
    assert lib.grouped_expert_gemm_nvfp4(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 128, 256, 256, FAKE, 0x200,
                                         None, 0, None) == -5
    assert lib.grouped_gemm_mxfp8(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 128, 256, 128, FAKE, 0x100 | 0x1000,
                                  None, 0, None) == -5
    # the fused SGD reports it before clearing amax_out (nothing is enqueued on an error return)
    assert lib.grouped_gemm_mxfp8_wgrad_sgd(FAKE, FAKE, FAKE, FAKE, FAKE, 2, 128, 256, 256, FAKE, None, 0.1, FAKE,
                                            0, FAKE, 64, None) == -5


def test_python_flags_match_the_header():
    from precision_moe_numerics_03_b300 import moe4
    defs = dict(re.findall(r"^#define MOE4_(\w+)\s+(0x[0-9A-Fa-f]+)u", open(HEADER).read(), flags=re.M))
    assert len(defs) >= 12
    for name, value in defs.items():
        assert getattr(moe4, name) == int(value, 16), name


def test_plain_c_caller(lib, tmp_path):
    """include/moe4.h compiles as strict C99 and a C program linked against libmoe4.so runs the
    host-side calls (queries and argument checks) without Python or a GPU."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    pkg = os.path.join(ROOT, "precision_moe_numerics_03_b300")
    exe = str(tmp_path / "c_abi_check")
    subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "c_abi_check.c"), "-L", pkg, "-lmoe4", "-Wl,-rpath," + pkg,
                    "-o", exe], check=True, capture_output=True, text=True)
    out = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stderr
    assert out.stdout.strip() == "ok"


def test_group_offsets_check_on_host(lib):
    """moe4_check_group_offsets: the rules the grouped GEMMs assume of their offsets, checked on a
    host copy (a group offset over the total, a decreasing entry, a ragged one, a non-zero start)."""
    import numpy as np
    from precision_moe_numerics_03_b300 import moe4

    def check(offs, total, align=128):
        a = np.ascontiguousarray(offs, dtype=np.int32)
        return lib.moe4_check_group_offsets(a.ctypes.data, a.size - 1, total, align)

    assert check([0, 128, 128, 512], 512) == 0            # an empty group is fine
    assert check([0, 0], 0) == 0
    assert check([0, 128, 640], 512) == -1                 # last offset over the total
    assert check([0, 256, 128, 512], 512) == -1            # decreasing
    assert check([0, 100, 512], 512) == -1                 # not a multiple of 128
    assert check([0, 100, 200], 200, align=1) == 0
    assert check([128, 256], 256) == -1                    # does not start at 0
    assert lib.moe4_check_group_offsets(None, 2, 0, 128) == -1
    moe4.moe4_check_group_offsets(np.array([0, 128, 256], np.int32), 256)
    with pytest.raises(moe4.Moe4Error):
        moe4.moe4_check_group_offsets(np.array([0, 384, 256], np.int32), 256)


def test_library_exports_nothing_undeclared(lib):
    """Every C-named function the library exports is declared in include/moe4.h (the reverse of
    test_every_declared_symbol_is_exported): no undocumented entry point."""
    import shutil
    import subprocess
    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("no nm")
    from precision_moe_numerics_03_b300 import moe4
    out = subprocess.run([nm, "-D", "--defined-only", moe4.LIB_PATH], check=True, capture_output=True,
                         text=True).stdout
    exported = sorted({f[2] for f in (ln.split() for ln in out.splitlines())
                       if len(f) == 3 and f[1] == "T" and not f[2].startswith("_")})
    assert exported == _declared()
