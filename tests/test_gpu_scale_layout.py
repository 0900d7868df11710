"""An outside pin of the 128x4 scale layout: the oracle's swizzled scales,
read by cuBLAS's block-scaled matmul (torch._scaled_mm), mean what the
oracle's linear scales mean.

The 128x4 layout is named on the pages without a definition (the
block-scaling-factor layout of cuBLAS).  Here the oracle quantises rows whose
blocks span a range of exponents, so a scale byte that lands in the wrong
place changes the value.  Its codes and swizzled scales go into a
block-scaled matmul against an identity operand with unit scales.  Each output
element then has exactly one non-zero product, and every product is exact in
fp32 and in bf16 (e4m3 codes times a power of two; e2m1 codes times an e4m3
scale).  So the product must equal, bit for bit, the oracle's dequantisation
through its linear scales.  Nothing from the CUDA path takes part; the
combine's own swizzled scales are compared with the oracle's byte for byte in
the parity tests."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

_VEC = {"mxfp8": 32, "mxfp4": 32, "nvfp4": 16}


def _oracle_quant(M, K, quant, seed):
    """Codes, swizzled scales and the linear-layout dequantisation of an
    M x K matrix, all from the oracle's quant-without-norm path (top_k = 1,
    unit weight, no norm)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    vec = _VEC[quant]
    lo, hi = (-4, 8) if quant == "nvfp4" else (-12, 12)   # NVFP4: block scales in e4m3's normal range
    expo = rng.integers(lo, hi + 1, (M, K // vec))
    x = rng.standard_normal((M, K)) * np.repeat(2.0 ** expo, vec, axis=1)
    ex = oracle.f64_to_bf16(x)
    rm = np.arange(M, dtype=np.int32).reshape(M, 1)
    w = np.ones((M, 1), np.float32)
    swz = oracle.combine(ex, rm, w, quant=quant, sf_layout="swizzled", outputs=("quant",))
    lin = oracle.combine(ex, rm, w, quant=quant, sf_layout="linear", outputs=("quant",))
    assert swz["status"] == 0 and lin["status"] == 0
    assert np.array_equal(swz["quant"], lin["quant"])
    want = oracle.dequant(lin["quant"], lin["scales"], M, K, quant, "linear", 1.0)
    return swz["quant"], swz["scales"], want


def _identity(K, quant):
    """The second operand as [K, N] column-major (N = K): identity codes,
    and unit scales (UE8M0 127 or e4m3 1.0) of the size the 128x4 layout of
    an N-row operand needs."""
    shape = _scale_shape(K, K, quant)
    if quant == "mxfp8":
        bt = np.zeros((K, K), np.uint8)
        np.fill_diagonal(bt, 0x38)                  # e4m3 1.0
        return bt, np.full(shape, 127, np.uint8)
    bt = np.zeros((K, K // 2), np.uint8)            # e2m1 pairs, element 2i in the low nibble
    n = np.arange(K)
    bt[n, n // 2] = np.where(n % 2 == 0, 0x02, 0x20)  # e2m1 1.0
    return bt, np.full(shape, 127 if quant == "mxfp4" else 0x38, np.uint8)


def _scale_shape(rows, K, quant):
    """[rows rounded up to 128, scale columns rounded up to 4]."""
    return (rows + 127) // 128 * 128, (K // _VEC[quant] + 3) // 4 * 4


@pytest.mark.parametrize("quant,M,K", [("mxfp8", 144, 480), ("mxfp8", 256, 128),
                                       ("nvfp4", 144, 224), ("nvfp4", 384, 64),
                                       ("mxfp4", 144, 480)])
def test_cublas_reads_the_oracles_swizzled_scales(quant, M, K):
    for name in ("float8_e4m3fn", "float8_e8m0fnu", "float4_e2m1fn_x2"):
        if not hasattr(torch, name):
            pytest.skip(f"torch {torch.__version__} has no {name}")
    q, s_swz, want = _oracle_quant(M, K, quant, seed=4200 + M + K)
    bt, s_b = _identity(K, quant)
    code_t = torch.float8_e4m3fn if quant == "mxfp8" else torch.float4_e2m1fn_x2
    scale_t = torch.float8_e4m3fn if quant == "nvfp4" else torch.float8_e8m0fnu
    a = torch.from_numpy(q).cuda().view(code_t)
    b = torch.from_numpy(bt).cuda().view(code_t).t()      # [K(/2), N], column-major
    sa = torch.from_numpy(s_swz.reshape(_scale_shape(M, K, quant))).cuda().view(scale_t)
    sb = torch.from_numpy(s_b).cuda().view(scale_t)
    try:
        out = torch._scaled_mm(a, b, sa, sb, out_dtype=torch.bfloat16)
    except (RuntimeError, NotImplementedError) as e:
        pytest.skip(f"no block-scaled {quant} matmul in torch {torch.__version__} here: "
                    f"{str(e).splitlines()[0]}")
    torch.cuda.synchronize()
    got = out.float().cpu().numpy().astype(np.float64)
    assert got.shape == (M, K)
    bad = got != want
    assert not bad.any(), (f"{int(bad.sum())} of {bad.size} differ; first "
                           f"{[(tuple(i), got[tuple(i)], want[tuple(i)]) for i in np.argwhere(bad)[:4]]}")
