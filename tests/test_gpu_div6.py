"""The NVFP4 block scale divides amax by 6 without a division instruction
(an FMA-corrected product, Markstein's method).  This checks it against
CUDA's correctly rounded division on every finite non-negative fp32 value:
bit for bit wherever the quotient is a normal float, and in the e4m3 block
scale it becomes everywhere (below 2^-126 every quotient's code is 0), so the
kernel's scale bytes are exactly those of amax / 6 rounded once."""
import ctypes
import os
import subprocess

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "..", "norm_quant_gb300", "csrc")


def test_div6_matches_the_correctly_rounded_division_everywhere(tmp_path):
    so = tmp_path / "libdiv6.so"
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-shared",
                    "-Xcompiler", "-fPIC", "-I", CSRC, "-o", str(so),
                    os.path.join(HERE, "cuda", "div6_check.cu")], check=True)
    lib = ctypes.CDLL(str(so))
    res = (ctypes.c_ulonglong * 4)()
    assert lib.div6_check(res) == 0
    bad_normal, bad_subnormal, bad_codes, checked = list(res)
    assert checked == 0x7F7FFFFF + 1
    assert bad_normal == 0
    assert bad_codes == 0
    print(f"quotients differing below 2^-126 (all e4m3 code 0): {bad_subnormal}")
