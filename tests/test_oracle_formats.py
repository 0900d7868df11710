"""Pins for the oracle's number formats and scale layouts (CPU only).

Each check compares the oracle with something other than itself: torch's
own float -> bf16 / float8_e4m3fn conversions (library routines), exact
rational brute force over every representable value, the value table of the
OCP Microscaling spec for FP4, and an index-free reshape/transpose statement
of the 128x4 scale layout.
"""
import bisect
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

RNG = np.random.Generator(np.random.PCG64(7))


# ------------------------------------------------------------------ bf16 --

def _all_bf16_values():
    bits = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    vals = bits.double().numpy()
    pos = sorted({float(v) for v in vals if np.isfinite(v) and v >= 0})
    return pos


_BF16_POS = None


def _bf16_nearest_even_bits(x: float) -> int:
    """Brute force: nearest bf16 to the exact value x, ties to even bits."""
    global _BF16_POS
    if _BF16_POS is None:
        _BF16_POS = _all_bf16_values()
    a = abs(x)
    i = bisect.bisect_right(_BF16_POS, a) - 1
    lo = _BF16_POS[i]
    hi = _BF16_POS[i + 1]
    dlo, dhi = Fraction(a) - Fraction(lo), Fraction(hi) - Fraction(a)

    def bits(v):
        return int(torch.tensor(v, dtype=torch.float64).to(torch.bfloat16).view(torch.int16)) & 0xFFFF

    blo, bhi = bits(lo), bits(hi)
    pick = blo if dlo < dhi else bhi if dhi < dlo else (blo if blo % 2 == 0 else bhi)
    return pick | (0x8000 if x < 0 else 0)


def test_bf16_from_float32_matches_torch():
    x = np.concatenate([
        RNG.standard_normal(4000).astype(np.float32),
        (RNG.standard_normal(2000) * 1e-30).astype(np.float32),
        (RNG.standard_normal(2000) * 1e30).astype(np.float32),
    ])
    # exact midpoints between adjacent bf16 values: ties must go to even
    base = torch.from_numpy(RNG.standard_normal(2000).astype(np.float32)).to(torch.bfloat16)
    u = base.view(torch.int16).numpy().astype(np.uint16).astype(np.uint32)
    mids = ((u << 16) | 0x8000).astype(np.uint32).view(np.float32)
    x = np.concatenate([x, mids])
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.f64_to_bf16(x.astype(np.float64))
    assert np.array_equal(got, want)


def test_bf16_from_double_brute_force():
    # doubles carry more bits than float32, so single rounding matters here
    xs = list(RNG.standard_normal(300)) + [1 + 2.0 ** -8, 1 + 2.0 ** -8 + 2.0 ** -40,
                                           1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8 - 2.0 ** -45)]
    for x in xs:
        assert int(oracle.f64_to_bf16(np.array([x]))[0]) == _bf16_nearest_even_bits(float(x)), x


def test_bf16_decode_roundtrip_all_finite():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = oracle.bf16_to_f64(bits)
    fin = np.isfinite(vals)
    back = oracle.f64_to_bf16(vals[fin])
    # -0.0 keeps its sign bit; every finite pattern survives the round trip
    assert np.array_equal(back, bits[fin])


# ------------------------------------------------------------------ e4m3 --

def test_e4m3_decode_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    got = oracle.e4m3_to_f64(codes)
    nan = np.isnan(want)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(got[~nan], want[~nan])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x08] == 2.0 ** -6


def test_e4m3_encode_matches_torch_in_range():
    # torch rounds to nearest even and turns |x| >= 464 into NaN; below that
    # it agrees with round-to-nearest-even-satfinite, which the oracle uses.
    vals = oracle.e4m3_to_f64(np.arange(0, 0x7F, dtype=np.uint8))
    mids = (vals[:-1] + vals[1:]) / 2
    x = np.concatenate([vals, mids, -mids, -vals,
                        RNG.uniform(-463, 463, 5000), RNG.standard_normal(3000) * 1e-2,
                        np.nextafter(mids, 0), np.nextafter(mids, 1000)])
    x = x[np.abs(x) < 464]
    x = x.astype(np.float32).astype(np.float64)
    want = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_from_f64(x)
    assert np.array_equal(got, want)


def test_e4m3_encode_saturates():
    got = oracle.e4m3_from_f64(np.array([448.0, 460.0, 464.0, 470.0, 1e6, -1e30]))
    assert got.tolist() == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE]


# ------------------------------------------------------------------ e2m1 --

# OCP Microscaling Formats v1.0, FP4 E2M1: magnitudes of codes 0..7.
OCP_FP4 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_decode_matches_spec_table():
    got = oracle.e2m1_to_f64(np.arange(16, dtype=np.uint8))
    assert got[:8].tolist() == OCP_FP4
    assert got[8:].tolist() == [-v for v in OCP_FP4]


def _e2m1_brute(x: float) -> int:
    a = Fraction(abs(x))
    if a >= 6:
        code = 7
    else:
        best = None
        for c, v in enumerate(OCP_FP4):
            d = abs(a - Fraction(v))
            if best is None or d < best[0] or (d == best[0] and c % 2 == 0):
                best = (d, c)
        code = best[1]
    return code | (8 if x < 0 or (x == 0 and np.signbit(x)) else 0)


def test_e2m1_encode_brute_force():
    x = np.concatenate([np.arange(-64, 65) / 8.0, RNG.uniform(-8, 8, 2000),
                        [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -2.5, 7.0, 1e9]])
    got = oracle.e2m1_from_f64(x)
    want = np.array([_e2m1_brute(float(v)) for v in x], dtype=np.uint8)
    assert np.array_equal(got, want)
    # the tie rule, spelled out
    ties = oracle.e2m1_from_f64(np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]))
    assert oracle.e2m1_to_f64(ties).tolist() == [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0]


# ----------------------------------------------------------------- UE8M0 --

def _ue8m0_brute(amax: float) -> int:
    if amax == 0:
        return 0
    a = Fraction(amax)
    e = -200
    while Fraction(448) * Fraction(2) ** e < a:
        e += 1
    return max(0, min(254, e + 127))


def test_ue8m0_rule_exact():
    f32 = np.float32
    cases = [0.0, 448.0, 224.0, 1.0, 1.75, 1.7500001, 3.5, 7.0, 1e-30, 1e30, 2.0 ** -140]
    for e in range(-20, 20):
        b = 448.0 * 2.0 ** e
        cases += [b, float(np.nextafter(f32(b), f32(0))), float(np.nextafter(f32(b), f32(np.inf)))]
    cases += list(np.abs(RNG.standard_normal(500)) * 10.0 ** RNG.integers(-10, 10, 500))
    cases = [float(f32(c)) for c in cases]
    got = oracle.ue8m0_for_amax(np.array(cases))
    want = [_ue8m0_brute(c) for c in cases]
    assert got.tolist() == want


def test_ue8m0_never_saturates_block():
    # every element of a block scaled by its UE8M0 scale lands in [-448, 448]
    for amax in np.abs(RNG.standard_normal(300)) * 10.0 ** RNG.integers(-5, 5, 300):
        b = int(oracle.ue8m0_for_amax(np.array([amax]))[0])
        assert amax * 2.0 ** (127 - b) <= 448.0


# ---------------------------------------------------------- scale layout --

def _swizzle_by_reshape(S: np.ndarray) -> np.ndarray:
    """128x4 layout as a reshape: pad to [Rp, Cp], view as
    [Rp/128, 4, 32, Cp/4, 4] (row = rb*128 + r4*32 + r32, col = cb*4 + c4),
    then order the axes (rb, cb, r32, r4, c4)."""
    R, Cc = S.shape
    Rp, Cp = -(-R // 128) * 128, -(-Cc // 4) * 4
    P = np.zeros((Rp, Cp), S.dtype)
    P[:R, :Cc] = S
    return P.reshape(Rp // 128, 4, 32, Cp // 4, 4).transpose(0, 3, 2, 1, 4).reshape(-1)


@pytest.mark.parametrize("R,Cc", [(1, 1), (5, 3), (128, 4), (130, 7), (300, 224), (256, 256)])
def test_swizzle_offset_matches_reshape(R, Cc):
    S = (np.arange(R * Cc) % 251 + 1).astype(np.uint8).reshape(R, Cc)
    want = _swizzle_by_reshape(S)
    got = np.zeros(oracle.scales_bytes(R, Cc * 32, "mxfp8", "swizzled"), np.uint8)
    assert got.size == want.size
    offs = set()
    for r in range(R):
        for c in range(Cc):
            o = oracle.sf_offset(r, c, Cc, "swizzled")
            got[o] = S[r, c]
            offs.add(o)
    assert len(offs) == R * Cc          # injective
    assert np.array_equal(got, want)    # same placement, zero padding


def test_linear_offset_and_sizes():
    assert oracle.sf_offset(3, 5, 224, "linear") == 3 * 224 + 5
    assert oracle.scales_bytes(4096, 7168, "mxfp8", "linear") == 4096 * 224
    assert oracle.scales_bytes(8192, 4096, "nvfp4", "swizzled") == 8192 * 256
    assert oracle.scales_bytes(1, 32, "mxfp8", "swizzled") == 128 * 4


# ------------------------------------------------------------------ fp16 --

def test_fp16_decode_all_codes_match_torch():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    want = torch.from_numpy(bits.view(np.int16)).view(torch.float16).double().numpy()
    got = oracle.f16_to_f64(bits)
    nan = np.isnan(want)
    assert np.array_equal(nan, np.isnan(got)) and np.array_equal(got[~nan], want[~nan])


def test_fp16_encode_matches_torch():
    vals = torch.arange(0, 0x7C00, dtype=torch.int32).to(torch.int16).view(torch.float16).double().numpy()
    mids = (vals[:-1] + vals[1:]) / 2
    x = np.concatenate([vals, mids, -mids, RNG.standard_normal(4000) * 10.0 ** RNG.integers(-8, 5, 4000),
                        [65504.0, 65519.0, 65520.0, 70000.0, 2.0 ** -25, 3 * 2.0 ** -26]])
    x32 = x.astype(np.float32)   # torch converts float32 -> float16 with one rounding
    want = torch.from_numpy(x32).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.f64_to_f16(x32.astype(np.float64))
    assert np.array_equal(got, want)


# --------------------------------------------------------- MXFP4 scale rule --

def _ue8m0_fp4_brute(amax: float) -> int:
    if amax == 0:
        return 0
    a = Fraction(amax)
    e = -200
    while Fraction(6) * Fraction(2) ** e < a:
        e += 1
    return max(0, min(254, e + 127))


def test_ue8m0_fp4_rule_exact():
    f32 = np.float32
    cases = [0.0, 6.0, 3.0, 1.5, 1.5000001, 12.0, 0.75, 1e-30, 1e30]
    for e in range(-20, 20):
        b = 6.0 * 2.0 ** e
        cases += [b, float(np.nextafter(f32(b), f32(0))), float(np.nextafter(f32(b), f32(np.inf)))]
    cases += list(np.abs(RNG.standard_normal(300)) * 10.0 ** RNG.integers(-8, 8, 300))
    cases = [float(f32(c)) for c in cases]
    assert oracle.ue8m0_fp4_for_amax(np.array(cases)).tolist() == [_ue8m0_fp4_brute(c) for c in cases]
