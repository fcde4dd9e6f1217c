"""C ABI checks that need no GPU: the library builds, loads, exports every
function include/ozemu.h declares, and its host-side queries and argument
checks behave as documented (checks run before any CUDA call)."""

import ctypes
import os
import re

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def oz():
    import ozaki_ii_fp64_gb300 as oz
    oz.load()
    return oz


def declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"\b(ozemu_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ("ozemu_igemm_s8", "ozemu_dgemm", "ozemu_get_status", "ozemu_max_moduli", "ozemu_release"):
        assert required in names


def test_library_exports_every_declared_symbol(oz):
    lib = oz.load()
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_mirrors_every_declared_symbol(oz):
    missing = [n for n in declared_functions() if not callable(getattr(oz, n, None))]
    assert not missing, missing


def test_moduli_match_oracle(oz):
    assert oz.ozemu_max_moduli() == 16
    assert oz.ozemu_moduli(16) == oracle.moduli(16)


@pytest.mark.parametrize("k", [1, 2, 255, 256, 4096, 8192, 16384, 65536, 131071])
@pytest.mark.parametrize("r", [3, 8, 11, 12, 13, 16])
def test_bit_budget_matches_oracle(oz, k, r):
    try:
        _, pa, pb = oracle.bit_budget(k, r)
    except ValueError:
        with pytest.raises(oz.OzemuError):
            oz.ozemu_bit_budget(k, r)
        return
    assert oz.ozemu_bit_budget(k, r) == (pa, pb)


def test_layout_sizes(oz):
    assert oz.ozemu_plane_bytes(1, 1, 1) == 3 * 128 * 64
    assert oz.ozemu_plane_bytes(129, 300, 13) == 3 * 13 * 256 * 192
    assert oz.ozemu_residue_bytes(5, 17, 2) == 2 * 5 * 32
    assert oz.ozemu_plane_bytes(-1, 1, 1) == 0
    assert oz.ozemu_residue_bytes(1, 1, 20) == 20 * 16  # r up to 20: the mixed-digit list
    assert oz.ozemu_residue_bytes(1, 1, 21) == 0


def test_two_limb_moduli_match_oracle(oz):
    assert oz.ozemu_moduli_2limb(16) == oracle.moduli(16, oracle.MODULUS_CEILING_2LIMB)


@pytest.mark.parametrize("k", [1, 2, 255, 256, 4096, 8192, 65536, 131071])
@pytest.mark.parametrize("r", [1, 3, 8, 13, 16])
def test_two_limb_bit_budget_matches_oracle(oz, k, r):
    try:
        _, pa, pb = oracle.bit_budget(k, r, oracle.MODULUS_CEILING_2LIMB)
    except ValueError:
        with pytest.raises(oz.OzemuError):
            oz.ozemu_bit_budget_2limb(k, r)
        return
    assert oz.ozemu_bit_budget_2limb(k, r) == (pa, pb)


def test_mixed_moduli_products_and_budget_match_oracle(oz):
    assert oz.ozemu_max_moduli_mixed() == 20 and oz.ozemu_single_digit_moduli_mixed() == 6
    assert oz.ozemu_moduli_mixed(20) == oracle.moduli(20, oracle.MIXED)
    for r in range(1, 21):
        assert oz.ozemu_products_mixed(r) == sum(oracle.products_per_modulus(l, oracle.MIXED) for l in range(r))
    assert oz.ozemu_products_mixed(0) == oz.OZEMU_ERR_INVALID_ARG
    for k in (1, 2, 300, 8192, 65536, 131071):
        for r in (1, 4, 6, 7, 13, 19, 20):
            try:
                _, pa, pb = oracle.bit_budget(k, r, oracle.MIXED)
            except ValueError:
                with pytest.raises(oz.OzemuError):
                    oz.ozemu_bit_budget_mixed(k, r)
                continue
            assert oz.ozemu_bit_budget_mixed(k, r) == (pa, pb)


def test_mixed_layout_sizes(oz):
    # single-digit moduli: one plane each; two-digit moduli: two
    assert oz.ozemu_plane_bytes_mixed(1, 1, 1) == 128 * 64
    assert oz.ozemu_plane_bytes_mixed(129, 300, 6) == 6 * 256 * 192
    assert oz.ozemu_plane_bytes_mixed(129, 300, 19) == (6 + 2 * 13) * 256 * 192
    assert oz.ozemu_plane_bytes_mixed(1, 1, 21) == 0


def test_two_limb_layout_sizes(oz):
    assert oz.ozemu_plane_bytes_2limb(1, 1, 1) == 2 * 128 * 64
    assert oz.ozemu_plane_bytes_2limb(129, 300, 16) == 2 * 16 * 256 * 192
    assert oz.ozemu_plane_bytes_2limb(1, 1, 17) == 0


NULL = None
FAKE = 0x10000  # a non-null, 16-byte aligned value; never dereferenced


@pytest.mark.parametrize("call", [
    lambda oz: oz.ozemu_dgemm(-1, 1, 1, FAKE, 1, FAKE, 1, FAKE, 1, 13, NULL),
    lambda oz: oz.ozemu_dgemm(4, 4, 4, FAKE, 3, FAKE, 4, FAKE, 4, 13, NULL),      # lda < k
    lambda oz: oz.ozemu_dgemm(4, 4, 4, FAKE, 4, FAKE, 3, FAKE, 4, 13, NULL),      # ldb < n
    lambda oz: oz.ozemu_dgemm(4, 4, 4, FAKE, 4, FAKE, 4, FAKE, 3, 13, NULL),      # ldc < n
    lambda oz: oz.ozemu_dgemm(4, 4, 4, FAKE, 4, FAKE, 4, FAKE, 4, 0, NULL),       # r < 1
    lambda oz: oz.ozemu_dgemm(4, 4, 4, FAKE, 4, FAKE, 4, FAKE, 4, 17, NULL),      # r > 16
    lambda oz: oz.ozemu_dgemm(4, 4, 4, NULL, 4, FAKE, 4, FAKE, 4, 13, NULL),      # null A
    lambda oz: oz.ozemu_dgemm(4, 4, 4, FAKE, 4, FAKE, 4, NULL, 4, 13, NULL),      # null C
    lambda oz: oz.ozemu_dgemm(4, 4, 200, FAKE, 200, FAKE, 4, FAKE, 4, 1, NULL),   # 2k >= 256
    lambda oz: oz.ozemu_igemm_s8(-1, 2, 2, FAKE, FAKE, FAKE, NULL),
    lambda oz: oz.ozemu_igemm_s8(2, 2, 2, NULL, FAKE, FAKE, NULL),
    lambda oz: oz.ozemu_split_rows_f64(4, 4, FAKE, 4, 63, 13, FAKE, FAKE, NULL),  # p > 62
    lambda oz: oz.ozemu_split_rows_f64(4, 4, FAKE, 4, 40, 13, FAKE + 8, FAKE, NULL),  # unaligned planes
    lambda oz: oz.ozemu_split_cols_f64(4, 4, FAKE, 3, 40, 13, FAKE, FAKE, NULL),  # ldx < cols
    lambda oz: oz.ozemu_split_rows_s8(4, 4, FAKE, 3, FAKE, NULL),
    lambda oz: oz.ozemu_split_cols_s8(4, 4, NULL, 4, FAKE, NULL),
    lambda oz: oz.ozemu_residue_gemm(4, 4, 4, 0, FAKE, FAKE, FAKE, NULL),
    lambda oz: oz.ozemu_residue_gemm(4, 4, 4, 13, FAKE, FAKE, FAKE + 4, NULL),    # unaligned residues
    lambda oz: oz.ozemu_limb_gemm_s32(4, 4, 4, FAKE, FAKE, FAKE, 3, NULL),        # ldc < n
    lambda oz: oz.ozemu_crt_f64(4, 4, 13, FAKE, FAKE, NULL, FAKE, 4, NULL),
    lambda oz: oz.ozemu_dgemm_host(4, 4, 4, FAKE, 3, FAKE, 4, FAKE, 4, 13, NULL),  # lda < k
    lambda oz: oz.ozemu_dgemm_host(4, 4, 4, FAKE, 4, FAKE, 4, NULL, 4, 13, NULL),  # null C
    lambda oz: oz.ozemu_dgemm_host(4, 4, 200, FAKE, 200, FAKE, 4, FAKE, 4, 1, NULL),  # 2k >= 256
    lambda oz: oz.ozemu_residues_narrow_f64(4, 3, 4, 13, FAKE, 4, FAKE, 3, FAKE, FAKE, FAKE, NULL),  # n > 2
    lambda oz: oz.ozemu_residues_narrow_f64(4, 1, 0, 13, FAKE, 1, FAKE, 1, FAKE, FAKE, FAKE, NULL),  # k < 1
    lambda oz: oz.ozemu_residues_narrow_f64(4, 1, 1 << 25, 16, FAKE, 1 << 25, FAKE, 1, FAKE, FAKE, FAKE, NULL),
    lambda oz: oz.ozemu_residues_narrow_f64(4, 2, 4, 13, FAKE, 4, FAKE, 1, FAKE, FAKE, FAKE, NULL),  # ldb < n
    lambda oz: oz.ozemu_residues_narrow_f64(4, 1, 4, 13, FAKE, 4, FAKE, 1, FAKE + 8, FAKE, FAKE, NULL),
    lambda oz: oz.ozemu_residues_narrow_f64(4, 1, 200, 1, FAKE, 200, FAKE, 1, FAKE, FAKE, FAKE, NULL),  # 2k >= M
    lambda oz: oz.ozemu_residues_narrow_f64(4, 1, 5, 16, FAKE, 5, FAKE, 1, FAKE, FAKE, FAKE, NULL),  # p_A > 52
    lambda oz: oz.ozemu_dgemm_2limb(4, 4, 4, FAKE, 3, FAKE, 4, FAKE, 4, 16, NULL),  # lda < k
    lambda oz: oz.ozemu_dgemm_2limb(4, 4, 4, FAKE, 4, FAKE, 4, FAKE, 4, 17, NULL),  # r > 16
    lambda oz: oz.ozemu_dgemm_2limb(4, 4, 4, FAKE, 4, FAKE, 4, NULL, 4, 16, NULL),  # null C
    lambda oz: oz.ozemu_dgemm_2limb(4, 4, 60, FAKE, 60, FAKE, 4, FAKE, 4, 1, NULL),  # 2k >= 113
    lambda oz: oz.ozemu_split_rows_f64_2limb(4, 4, FAKE, 4, 63, 16, FAKE, FAKE, NULL),  # p > 62
    lambda oz: oz.ozemu_split_cols_f64_2limb(4, 4, FAKE, 3, 40, 16, FAKE, FAKE, NULL),  # ldx < cols
    lambda oz: oz.ozemu_residue_gemm_2limb(4, 4, 4, 16, FAKE, FAKE, FAKE + 4, NULL),  # unaligned residues
    lambda oz: oz.ozemu_crt_f64_2limb(4, 4, 0, FAKE, FAKE, FAKE, FAKE, 4, NULL),  # r < 1
    lambda oz: oz.ozemu_dgemm_host_2limb(4, 4, 60, FAKE, 60, FAKE, 4, FAKE, 4, 1, NULL),  # 2k >= 113
    lambda oz: oz.ozemu_dgemm_host_2limb(4, 4, 4, FAKE, 4, FAKE, 4, NULL, 4, 16, NULL),  # null C
    lambda oz: oz.ozemu_igemm_s4s8(-1, 4, 4, FAKE, FAKE, FAKE, NULL),
    lambda oz: oz.ozemu_igemm_s4s8(4, 4, 4, FAKE, FAKE, NULL, NULL),                # null C32
    lambda oz: oz.ozemu_igemm_s4s8(4, 4, 4, NULL, FAKE, FAKE, NULL),                # null A
    lambda oz: oz.ozemu_split_rows_s4(4, 4, FAKE, 3, FAKE, NULL),                   # ldx < k
    lambda oz: oz.ozemu_split_rows_s4(4, 4, FAKE, 4, FAKE + 8, NULL),               # unaligned planes
    lambda oz: oz.ozemu_split_cols_s8_four(4, 4, FAKE, 3, FAKE, NULL),              # ldx < cols
    lambda oz: oz.ozemu_split_cols_s8_four(4, 4, NULL, 4, FAKE, NULL),              # null X
])
def test_invalid_arguments_rejected_on_host(oz, call):
    assert call(oz) == oz.OZEMU_ERR_INVALID_ARG


def test_k_overflow_rejected_on_host(oz):
    assert oz.ozemu_igemm_s8(4, 4, 131072, FAKE, FAKE, FAKE, NULL) == oz.OZEMU_ERR_K_OVERFLOW
    assert oz.ozemu_limb_gemm_s32(4, 4, 131072, FAKE, FAKE, FAKE, 4, NULL) == oz.OZEMU_ERR_K_OVERFLOW
    # INT4 x INT8: |C| <= 1024 k must stay below 2^31.
    assert oz.ozemu_igemm_s4s8(4, 4, 2097152, FAKE, FAKE, FAKE, NULL) == oz.OZEMU_ERR_K_OVERFLOW


def test_four_plane_layout_size(oz):
    # [rows_p][k_p/128][4][64]: 2 k_p bytes per padded row.
    assert oz.ozemu_four_plane_bytes(1, 1) == 128 * 2 * 128
    assert oz.ozemu_four_plane_bytes(129, 129) == 256 * 2 * 256
    assert oz.ozemu_four_plane_bytes(-1, 4) == 0
    assert oz.OZEMU_ERR_RANGE == -9


def test_narrow_limit(oz):
    assert oz.ozemu_narrow_max_n() == 2


def test_empty_problems_are_noops(oz):
    assert oz.ozemu_dgemm(0, 5, 5, NULL, 5, NULL, 5, NULL, 5, 13, NULL) == oz.OZEMU_OK
    assert oz.ozemu_dgemm(5, 0, 5, NULL, 5, NULL, 1, NULL, 1, 13, NULL) == oz.OZEMU_OK
    assert oz.ozemu_dgemm_host(0, 5, 5, NULL, 5, NULL, 5, NULL, 5, 13, NULL) == oz.OZEMU_OK
    assert oz.ozemu_igemm_s8(0, 0, 7, NULL, NULL, NULL, NULL) == oz.OZEMU_OK
    assert oz.ozemu_split_rows_f64(0, 9, NULL, 9, 30, 13, NULL, NULL, NULL) == oz.OZEMU_OK
    assert oz.ozemu_residue_gemm(0, 3, 3, 13, NULL, NULL, NULL, NULL) == oz.OZEMU_OK
    assert oz.ozemu_igemm_s4s8(0, 3, 3, NULL, NULL, NULL, NULL) == oz.OZEMU_OK
    assert oz.ozemu_split_rows_s4(0, 9, NULL, 9, NULL, NULL) == oz.OZEMU_OK


def test_product_path_has_no_fallback():
    # The package never imports the oracle and never computes on the host.
    pkg = os.path.join(ROOT, "ozaki_ii_fp64_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, fn)).read()
                assert "import oracle" not in text and "from oracle" not in text, fn


def test_header_and_library_usable_from_plain_c(oz, tmp_path):
    # The boundary is a C ABI: a C99 program includes the header, links the
    # library and calls host-side entry points (no device work).
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    lib = oz.library_path()
    cuda_inc = "/usr/local/cuda/include"
    src = tmp_path / "use.c"
    src.write_text(
        '#include "ozemu.h"\n'
        "#include <stdio.h>\n"
        "int main(void) {\n"
        "  int pa = 0, pb = 0, m[16];\n"
        "  if (ozemu_max_moduli() != 16) return 1;\n"
        "  if (ozemu_moduli(3, m) != OZEMU_OK || m[0] != 256 || m[1] != 255 || m[2] != 253) return 2;\n"
        "  if (ozemu_bit_budget(8192, 13, &pa, &pb) != OZEMU_OK) return 3;\n"
        "  if (ozemu_dgemm(4, 4, 4, 0, 3, 0, 4, 0, 4, 13, 0) != OZEMU_ERR_INVALID_ARG) return 4;\n"
        '  printf("%d %d\\n", pa, pb);\n'
        "  return 0;\n"
        "}\n")
    exe = tmp_path / "use"
    cmd = [gcc, "-std=c99", "-I", os.path.join(ROOT, "include"), "-I", cuda_inc, str(src), "-o", str(exe),
           "-L", os.path.dirname(lib), "-lozemu", "-Wl,-rpath," + os.path.dirname(lib)]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0 and "cuda_runtime_api.h" in res.stderr:
        pytest.skip("CUDA headers not found")
    assert res.returncode == 0, res.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True)
    assert run.returncode == 0, run.stdout + run.stderr
    _, pa, pb = oracle.bit_budget(8192, 13)
    assert run.stdout.split() == [str(pa), str(pb)]
