"""The RMSNorm scale 1/sqrt(mean(x^2) + eps) comes from the hardware's
reciprocal square root refined by one Newton step.  This checks it on every
positive normal fp32 value against CUDA's correctly rounded reciprocal square
root: never more than one ulp away.  Zero still gives infinity (a zero row
with eps = 0 normalises as 0 * inf, as 1 / sqrtf(0) would) and infinity 0."""
import ctypes
import os
import subprocess

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "..", "norm_quant_gb300", "csrc")


def test_rsqrt_newton_within_one_ulp_of_the_correctly_rounded_value(tmp_path):
    so = tmp_path / "librsqrt.so"
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-shared",
                    "-Xcompiler", "-fPIC", "-I", CSRC, "-o", str(so),
                    os.path.join(HERE, "cuda", "rsqrt_check.cu")], check=True)
    lib = ctypes.CDLL(str(so))
    res = (ctypes.c_ulonglong * 4)()
    assert lib.rsqrt_check(res) == 0
    differ, beyond_one_ulp, checked, specials_wrong = list(res)
    print(f"checked {checked}; differing from the correctly rounded value: {differ} "
          f"({differ / checked:.4%}); beyond one ulp: {beyond_one_ulp}")
    assert checked == 0x7F7FFFFF - 0x00800000 + 1
    assert beyond_one_ulp == 0
    assert specials_wrong == 0
