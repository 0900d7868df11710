"""The NVFP4 element code is e2m1 of the quotient v / s, computed without a
division instruction (an FMA-corrected product, Markstein's method).  This
checks it against CUDA's correctly rounded division for every positive e4m3
block scale and every float a block with that scale can hold: bit for bit
wherever the element is at least 2^-100 and the quotient a normal float
(below that the remainder underflows, outside the theorem's assumptions, and
every quotient is below 2^-91, code 0), and in the e2m1 code everywhere.  It
also counts how many codes the plain product v * RN(1/s) would get wrong, the
cases the correction exists for."""
import ctypes
import os
import subprocess

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "..", "norm_quant_gb300", "csrc")


def test_nvfp4_quotient_matches_the_correctly_rounded_division(tmp_path):
    so = tmp_path / "libquot.so"
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-shared",
                    "-Xcompiler", "-fPIC", "-I", CSRC, "-o", str(so),
                    os.path.join(HERE, "cuda", "nvfp4_quotient_check.cu")], check=True)
    lib = ctypes.CDLL(str(so))
    lib.nvfp4_quotient_expected_count.restype = ctypes.c_ulonglong
    res = (ctypes.c_ulonglong * 7)()
    assert lib.nvfp4_quotient_check(res) == 0
    bad_normal, bad_sub_input, bad_sub_quotient, bad_codes, product_codes, checked, first = list(res)
    print(f"checked {checked}; quotients differing: v and quotient normal {bad_normal} "
          f"(first: scale code {first >> 32}, v bits {first & 0xFFFFFFFF:#010x}), v below 2^-100 {bad_sub_input}, "
          f"quotient subnormal {bad_sub_quotient}; codes differing {bad_codes}; codes the plain product "
          f"would change: {product_codes}")
    assert checked == lib.nvfp4_quotient_expected_count()
    assert bad_codes == 0
    assert bad_normal == 0
    assert product_codes > 0   # the midpoint cases exist, so the check can see them
