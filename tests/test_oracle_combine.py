"""Pins for the oracle's combine / residual / RMSNorm / quantisation (CPU).

Every check is tied to something outside the oracle: a hand-derived worked
example, closed forms of the norm, exact invariants of the sum (gather,
permutation, partition of unity, one-hot index recovery), the Gemma-form
identity, and inputs already on the fp8 / fp4 grids that must round-trip
exactly.
"""
import json
import os

import numpy as np
import pytest

import oracle
from norm_quant_gb300.synth import f32_to_bf16_bits

HERE = os.path.dirname(os.path.abspath(__file__))
RNG = np.random.Generator(np.random.PCG64(13))


def bf(x):
    return f32_to_bf16_bits(np.asarray(x, np.float32))


def f(bits):
    return oracle.bf16_to_f64(bits)


def _routing(T, k, E, rng=RNG):
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    st, counts, offsets, row_map, _ = oracle.build_row_map(ids, E)
    assert st == 0
    return ids, row_map, int(offsets[E])


# --------------------------------------------------------- worked example --

def _worked_example_inputs():
    g = json.load(open(os.path.join(HERE, "golden", "worked_example.json")))
    H = g["H"]
    h = np.arange(H)
    rows = np.stack([np.ones(H), 2 * np.ones(H), np.where(h % 2 == 0, 1.0, -1.0)])
    shared = np.stack([np.full(H, v) for v in g["shared_per_token"]])
    residual = np.stack([np.full(H, v) for v in g["residual_per_token"]])
    gamma = np.ones(H)
    gamma[:3] = [7.0, 0.5, 2.0]
    return g, rows, shared, residual, gamma


def test_worked_example_golden():
    g, rows, shared, residual, gamma = _worked_example_inputs()
    ex = g["expect"]
    st, counts, offsets, row_map, src_row = oracle.build_row_map(np.array(g["topk_ids"]), g["E"])
    assert st == 0
    assert counts.tolist() == ex["counts"] and offsets.tolist() == ex["offsets"]
    assert row_map.tolist() == ex["row_map"] and src_row.tolist() == ex["src_row"]
    w = np.array(g["router_weights"], np.float32)
    common = dict(shared=bf(shared), residual=bf(residual), gamma=bf(gamma), eps=g["eps"],
                  weight_bias=g["weight_bias"])
    o = oracle.combine(bf(rows), row_map, w, quant="mxfp8", **common)
    assert o["status"] == 0
    comb, res, nrm = f(o["combined"]), f(o["residual"]), f(o["norm"])
    assert np.all(comb[0, 0::2] == ex["combined_t0_even"]) and np.all(comb[0, 1::2] == ex["combined_t0_odd"])
    assert np.all(comb[1] == ex["combined_t1"])
    assert np.all(res[0, 0::2] == ex["residual_out_t0_even"]) and np.all(res[0, 1::2] == ex["residual_out_t0_odd"])
    assert np.all(res[1] == ex["residual_out_t1"])
    assert nrm[0, :6].tolist() == ex["norm_out_t0_head"] and nrm[1, :6].tolist() == ex["norm_out_t1_head"]
    assert o["scales"].tolist() == ex["mxfp8_scale"]
    assert [hex(v).upper().replace("X", "x") for v in o["quant"][0, :6]] == ex["mxfp8_codes_t0_head"]
    assert [hex(v).upper().replace("X", "x") for v in o["quant"][1, :6]] == ex["mxfp8_codes_t1_head"]
    # the rest of the rows follow the same alternating pattern
    assert np.all(o["quant"][0, 4::2] == 0x68) and np.all(o["quant"][0, 3::2] == 0xE8)
    o4 = oracle.combine(bf(rows), row_map, w, quant="nvfp4", global_scale=1.0, **common)
    want_s = [[int(v, 16) for v in r] for r in ex["nvfp4_scales"]]
    assert o4["scales"].reshape(2, 2).tolist() == want_s
    assert o4["quant"][0].tolist() == [int(v, 16) for v in ex["nvfp4_bytes_t0"]]
    assert o4["quant"][1].tolist() == [int(v, 16) for v in ex["nvfp4_bytes_t1"]]


def _nvfp4_midpoint_golden():
    return json.load(open(os.path.join(HERE, "golden", "nvfp4_midpoints.json")))


def _e2m1_rne_f32_codes(x):
    """e2m1 codes of float values by nearest-value search over the grid,
    ties to the even code, saturating at 6 (written out here, not taken from
    the oracle)."""
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float64)
    out = []
    for v in np.asarray(x, np.float64):
        a = min(abs(v), 6.0)
        dist = np.abs(grid - a)
        best = np.flatnonzero(dist == dist.min())
        c = int(best[0]) if best.size == 1 else int(best[best % 2 == 0][0])
        out.append(c | (8 if v < 0 and c else 0))
    return out


def test_nvfp4_midpoint_golden_divides_by_the_block_scale():
    # elements exactly on e2m1 midpoints once divided by the block scale; the
    # expected bytes are hand-derived in the fixture
    g = _nvfp4_midpoint_golden()
    H = g["H"]
    row = bf(np.array(g["row"], np.float64))[None, :]
    assert np.array_equal(f(row)[0], g["row"])           # the row is exact in bf16
    o = oracle.combine(row, np.zeros((1, 1), np.int32), np.ones((1, 1), np.float32), quant="nvfp4",
                       global_scale=g["global_scale"], outputs=("quant",))
    assert o["status"] == 0
    assert o["scales"].tolist() == [int(v, 16) for v in g["expect"]["scales"]]
    assert o["quant"][0].tolist() == [int(v, 16) for v in g["expect"]["bytes"]]
    # the global scale acts before the block scaling: a row 4x smaller with
    # g = 4 gives the same bytes
    o4 = oracle.combine(bf(np.array(g["row"]) / 4)[None, :], np.zeros((1, 1), np.int32),
                        np.ones((1, 1), np.float32), quant="nvfp4", global_scale=4.0, outputs=("quant",))
    assert o4["quant"].tolist() == o["quant"].tolist() and o4["scales"].tolist() == o["scales"].tolist()
    assert H == 32


def test_nvfp4_midpoint_golden_separates_the_reciprocal_reading():
    # the other plausible reading, an element times the fp32 reciprocal of its
    # block scale, written out in float32 arithmetic: it must give the
    # fixture's other bytes, so the golden above cannot pass under it
    g = _nvfp4_midpoint_golden()
    v = np.array(g["row"], np.float32)
    scales = [1.875, 0.234375]
    codes = []
    for b in range(2):
        rs = np.float32(1.0) / np.float32(scales[b])
        codes += _e2m1_rne_f32_codes((v[16 * b:16 * b + 16] * rs).astype(np.float32))
        # and the quotient reading, for the expected bytes
    packed = [codes[2 * i] | (codes[2 * i + 1] << 4) for i in range(16)]
    assert packed == [int(x, 16) for x in g["expect"]["bytes_if_reciprocal"]]
    assert packed != [int(x, 16) for x in g["expect"]["bytes"]]
    qcodes = []
    for b in range(2):
        qcodes += _e2m1_rne_f32_codes(np.array(g["row"][16 * b:16 * b + 16]) / scales[b])
    assert [qcodes[2 * i] | (qcodes[2 * i + 1] << 4) for i in range(16)] == [int(x, 16) for x in g["expect"]["bytes"]]


# -------------------------------------------------------------- the sum ---

def test_top1_unit_weight_is_a_pure_gather():
    T, H, E = 40, 64, 12
    ids, row_map, nv = _routing(T, 1, E)
    rows = RNG.standard_normal((nv, H)).astype(np.float32)
    o = oracle.combine(bf(rows), row_map, np.ones((T, 1), np.float32), outputs=("combined",))
    assert np.array_equal(o["combined"], bf(rows)[row_map[:, 0]])


def test_one_hot_rows_recover_row_map_and_weights():
    # row r is the unit vector e_r; token t must then hold w[t, j] exactly at
    # column row_map[t, j] and zero elsewhere -- any index or operand mix-up
    # between slots, tokens and rows shows.
    T, k, E = 24, 4, 9
    ids, row_map, nv = _routing(T, k, E)
    ids[3, 1] = -1
    row_map[3, 1] = -1
    rows = np.eye(nv, dtype=np.float32)
    w = np.array([[2.0 ** -(j + 1) * (1 + (t % 3)) for j in range(k)] for t in range(T)], np.float32)
    o = oracle.combine(bf(rows), row_map, w, outputs=("combined",))
    want = np.zeros((T, nv))
    for t in range(T):
        for j in range(k):
            if row_map[t, j] >= 0:
                want[t, row_map[t, j]] = w[t, j]
    assert np.array_equal(f(o["combined"]), want)


@pytest.mark.parametrize("quant", [None, "mxfp8", "nvfp4"])
def test_permuting_slots_changes_nothing(quant):
    T, k, E, H = 16, 8, 32, 64
    ids, row_map, nv = _routing(T, k, E)
    rows = bf(RNG.standard_normal((nv, H)))
    w = (2.0 ** -RNG.integers(0, 6, (T, k))).astype(np.float32)   # dyadic: sums exact
    kw = dict(residual=bf(RNG.standard_normal((T, H))), gamma=bf(1 + 0.1 * RNG.standard_normal(H)),
              quant=quant, global_scale=3.0)
    a = oracle.combine(rows, row_map, w, **kw)
    perm = RNG.permutation(k)
    b = oracle.combine(rows, row_map[:, perm], w[:, perm], **kw)
    for key in ("combined", "residual", "norm", "y", "quant", "scales"):
        if key in a:
            assert np.array_equal(a[key], b[key]), key


def test_equal_rows_with_weights_summing_to_one_reproduce_the_row():
    T, k, H = 10, 8, 96
    row = bf(RNG.standard_normal(H))
    rows = np.tile(row, (T * k, 1))
    row_map = np.arange(T * k, dtype=np.int32).reshape(T, k)
    for w in [np.full((T, k), 1.0 / k, np.float32),
              np.array(RNG.dirichlet(np.ones(k), T), np.float32)]:
        o = oracle.combine(rows, row_map, w, outputs=("combined",))
        assert np.array_equal(o["combined"], np.tile(row, (T, 1)))


def test_padded_slots_and_shared_weight_one():
    T, H = 3, 32
    rows = bf(RNG.standard_normal((2, H)))
    shared = bf(RNG.standard_normal((T, H)))
    row_map = np.array([[-1, -1], [0, -1], [-1, 1]], np.int32)
    w = np.array([[5.0, 7.0], [1.0, 9.0], [3.0, 1.0]], np.float32)  # padded weights ignored
    o = oracle.combine(rows, row_map, w, shared=shared, outputs=("combined",))
    c = f(o["combined"])
    assert np.array_equal(o["combined"][0], shared[0])                    # all padded: shared only
    assert np.array_equal(c[1], f(bf(f(rows[0]) + f(shared[1]))))
    assert np.array_equal(c[2], f(bf(f(rows[1]) + f(shared[2]))))


# ------------------------------------------------------------- RMSNorm ----

def test_rmsnorm_unit_gamma_gives_unit_rms():
    T, H, eps = 12, 256, 2.0 ** -10   # eps travels as fp32: keep it exact
    ids, row_map, nv = _routing(T, 4, 16)
    rows = bf(3 * RNG.standard_normal((nv, H)))
    w = np.full((T, 4), 0.25, np.float32)
    res = bf(RNG.standard_normal((T, H)))
    x = oracle.combine(rows, row_map, w, residual=res)["y"]        # no gamma: y is x
    y = oracle.combine(rows, row_map, w, residual=res, gamma=bf(np.ones(H)), eps=eps)["y"]
    m = (x ** 2).mean(axis=1)
    assert np.allclose((y ** 2).mean(axis=1), m / (m + eps), rtol=1e-13, atol=0)
    assert np.allclose(y, x / np.sqrt(m + eps)[:, None], rtol=1e-14, atol=0)


def test_rmsnorm_constant_row_closed_form():
    H = 64
    for c, eps in [(1.0, 3.0), (2.0, 0.0), (0.5, 1e-6), (-1.5, 0.75)]:
        rows = bf(np.full((1, H), c))
        o = oracle.combine(rows, np.array([[0]], np.int32), np.ones((1, 1), np.float32),
                           gamma=bf(np.ones(H)), eps=eps)
        e32 = float(np.float32(eps))
        assert np.allclose(o["y"], c / np.sqrt(c * c + e32), rtol=1e-15, atol=0)
    # eps inside the square root: c = 1, eps = 3 gives exactly 1/2
    o = oracle.combine(bf(np.ones((1, H))), np.array([[0]], np.int32), np.ones((1, 1), np.float32),
                       gamma=bf(np.ones(H)), eps=3.0)
    assert np.all(o["y"] == 0.5)


def test_rmsnorm_gamma_is_per_column():
    H = 64
    gamma = bf(np.arange(1, H + 1) / 8.0)
    rows = bf(np.full((1, H), 2.0))
    o = oracle.combine(rows, np.array([[0]], np.int32), np.ones((1, 1), np.float32),
                       gamma=gamma, eps=0.0)
    assert np.array_equal(o["y"][0], f(gamma))   # x / rms(x) = 1 for a constant row


def test_gemma_form_identity():
    T, H = 8, 128
    ids, row_map, nv = _routing(T, 2, 6)
    rows = bf(RNG.standard_normal((nv, H)))
    w = np.full((T, 2), 0.5, np.float32)
    kw = dict(residual=bf(RNG.standard_normal((T, H))), quant="nvfp4", global_scale=100.0)
    a = oracle.combine(rows, row_map, w, gamma=bf(np.zeros(H)), weight_bias=1.0, **kw)
    b = oracle.combine(rows, row_map, w, gamma=bf(np.ones(H)), weight_bias=0.0, **kw)
    for key in ("norm", "y", "quant", "scales"):
        assert np.array_equal(a[key], b[key]), key
    # a general weight_bias is gamma + weight_bias
    c = oracle.combine(rows, row_map, w, gamma=bf(np.full(H, 0.5)), weight_bias=0.25, **kw)
    d = oracle.combine(rows, row_map, w, gamma=bf(np.full(H, 0.75)), weight_bias=0.0, **kw)
    assert np.array_equal(c["y"], d["y"])


def test_zero_row_normalises_to_zero():
    H = 64
    o = oracle.combine(np.zeros((0, H), np.uint16), np.array([[-1, -1]], np.int32),
                       np.ones((1, 2), np.float32), gamma=bf(np.ones(H)), eps=1e-6,
                       quant="mxfp8")
    assert np.all(o["y"] == 0) and np.all(o["quant"] == 0) and np.all(o["scales"] == 0)


# --------------------------------------------------------- quantisation ---

def test_mxfp8_grid_values_roundtrip_exactly():
    H, T = 128, 6
    e4m3 = oracle.e4m3_to_f64(np.arange(0, 0x7F, dtype=np.uint8))
    rows, codes, scales = [], [], []
    for t in range(T):
        row = []
        for blk in range(H // 32):
            e = int(RNG.integers(-20, 10))
            c = RNG.integers(0, 0x7F, 32).astype(np.uint8)
            c[RNG.integers(0, 32)] = 0x7E                       # amax = 448 * 2^e
            c = c | (RNG.integers(0, 2, 32).astype(np.uint8) << 7)
            vals = np.where(c & 0x80, -1.0, 1.0) * e4m3[c & 0x7F] * 2.0 ** e
            row.append(vals)
            codes.append(c)
            scales.append(e + 127)
        rows.append(np.concatenate(row))
    rows = np.array(rows)
    bits = bf(rows)
    assert np.array_equal(f(bits), rows)                       # grid values are bf16-exact
    o = oracle.combine(bits, np.arange(T, dtype=np.int32)[:, None], np.ones((T, 1), np.float32),
                       quant="mxfp8")
    want_codes = np.concatenate(codes).reshape(T, H)
    zero = (want_codes & 0x7F) == 0
    assert np.array_equal(o["quant"][~zero], want_codes[~zero])
    assert np.all((o["quant"][zero] & 0x7F) == 0)
    assert o["scales"].tolist() == scales
    assert np.array_equal(oracle.dequant(o["quant"], o["scales"], T, H, "mxfp8"), rows)


def test_nvfp4_grid_values_roundtrip_exactly():
    H, T = 64, 5
    e4m3 = oracle.e4m3_to_f64(np.arange(0, 0x7F, dtype=np.uint8))
    fp4 = oracle.e2m1_to_f64(np.arange(8, dtype=np.uint8))
    rows, scales, codes = [], [], []
    for t in range(T):
        for blk in range(H // 16):
            sc = int(RNG.integers(0x20, 0x60))                # normal e4m3 scale
            c = RNG.integers(0, 8, 16).astype(np.uint8)
            c[RNG.integers(0, 16)] = 7                          # amax = 6 * s
            c = c | (RNG.integers(0, 2, 16).astype(np.uint8) << 3)
            rows.append(np.where(c & 8, -1.0, 1.0) * fp4[c & 7] * e4m3[sc])
            scales.append(sc)
            codes.append(c)
    rows = np.concatenate(rows).reshape(T, H)
    bits = bf(rows)
    assert np.array_equal(f(bits), rows)
    for g in (1.0, 4.0):
        # a power-of-two global scale on inputs divided by it leaves codes alone
        inp = bf(rows / g)
        o = oracle.combine(inp, np.arange(T, dtype=np.int32)[:, None], np.ones((T, 1), np.float32),
                           quant="nvfp4", global_scale=g)
        assert o["scales"].tolist() == scales
        c = np.concatenate(codes).reshape(T, H)
        got = np.stack([o["quant"] & 15, o["quant"] >> 4], axis=-1).reshape(T, H)
        nz = (c & 7) != 0
        assert np.array_equal(got[nz], c[nz]) and np.all((got[~nz] & 7) == 0)
        assert np.array_equal(oracle.dequant(o["quant"], o["scales"], T, H, "nvfp4",
                                              global_scale=g), rows / g)


def test_swizzled_scales_are_the_linear_scales_relocated():
    T, H = 130, 96
    ids, row_map, nv = _routing(T, 2, 8)
    rows = bf(RNG.standard_normal((nv, H)))
    w = np.full((T, 2), 0.5, np.float32)
    for quant, vec in (("mxfp8", 32), ("nvfp4", 16)):
        lin = oracle.combine(rows, row_map, w, quant=quant, sf_layout="linear", global_scale=7.0)
        swz = oracle.combine(rows, row_map, w, quant=quant, sf_layout="swizzled", global_scale=7.0)
        assert np.array_equal(lin["quant"], swz["quant"])
        Cc = H // vec
        moved = np.zeros_like(swz["scales"])
        for r in range(T):
            for c in range(Cc):
                moved[oracle.sf_offset(r, c, Cc, "swizzled")] = lin["scales"][r * Cc + c]
        assert np.array_equal(moved, swz["scales"])


def test_mxfp8_dequant_within_half_a_step_of_input():
    # e4m3 keeps 3 mantissa bits, so in the top binade of a block with scale
    # 2^e the spacing is 2^(e + 8 - 3); rounding is within half of that.
    T, H = 20, 256
    x = RNG.standard_normal((T, H)) * 10.0 ** RNG.integers(-3, 3, (T, 1))
    o = oracle.combine(bf(x), np.arange(T, dtype=np.int32)[:, None], np.ones((T, 1), np.float32),
                       quant="mxfp8")
    dq = oracle.dequant(o["quant"], o["scales"], T, H, "mxfp8")
    e = o["scales"].reshape(T, H // 32).astype(float) - 127
    half = np.repeat(2.0 ** (e + 5), 32, axis=1) / 2
    assert np.all(np.abs(dq - f(bf(x))) <= half)


def test_empty_batch():
    o = oracle.combine(np.zeros((0, 32), np.uint16), np.zeros((0, 2), np.int32),
                       np.zeros((0, 2), np.float32), quant="mxfp8")
    assert o["status"] == 0 and o["quant"].shape == (0, 32)


# ------------------------------------------------------- slot-major layout --

def test_slot_major_is_the_grouped_layout_with_row_map_j_T_plus_t():
    # the slot-major buffer [k, T, H] is a grouped buffer whose row_map is
    # row_map[t, j] = j * T + t; both index paths must agree bit for bit
    T, k, H = 37, 4, 64
    rows = bf(RNG.standard_normal((k, T, H)))
    w = np.array(RNG.dirichlet(np.ones(k), T), np.float32)
    kw = dict(shared=bf(RNG.standard_normal((T, H))), residual=bf(RNG.standard_normal((T, H))),
              gamma=bf(1 + 0.1 * RNG.standard_normal(H)), quant="mxfp8")
    a = oracle.combine(rows, None, w, expert_layout="slot_major", **kw)
    rm = (np.arange(k)[None, :] * T + np.arange(T)[:, None]).astype(np.int32)
    b = oracle.combine(rows.reshape(k * T, H), rm, w, **kw)
    for key in ("combined", "residual", "norm", "y", "quant", "scales"):
        assert np.array_equal(a[key], b[key]), key


def test_slot_major_one_hot_recovers_slot_and_token():
    # slot j of token t is the unit vector e_(j*T + t) in H = k*T columns
    T, k = 6, 3
    H = k * T + 6
    rows = np.zeros((k, T, H), np.float32)
    for j in range(k):
        for t in range(T):
            rows[j, t, j * T + t] = 1.0
    w = np.array([[2.0 ** -(j + 1) for j in range(k)] for _ in range(T)], np.float32)
    w[2, 1] = 0.0
    o = oracle.combine(bf(rows), None, w, expert_layout="slot_major", outputs=("combined",))
    want = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            want[t, j * T + t] = w[t, j]
    assert np.array_equal(f(o["combined"]), want)


# --------------------------------------------------------- dtype variants --

def test_mxfp4_grid_values_roundtrip_exactly():
    H, T = 96, 5
    fp4 = oracle.e2m1_to_f64(np.arange(8, dtype=np.uint8))
    rows, codes, scales = [], [], []
    for t in range(T):
        for blk in range(H // 32):
            e = int(RNG.integers(-12, 12))
            c = RNG.integers(0, 8, 32).astype(np.uint8)
            c[RNG.integers(0, 32)] = 7                          # amax = 6 * 2^e
            c = c | (RNG.integers(0, 2, 32).astype(np.uint8) << 3)
            rows.append(np.where(c & 8, -1.0, 1.0) * fp4[c & 7] * 2.0 ** e)
            codes.append(c)
            scales.append(e + 127)
    rows = np.concatenate(rows).reshape(T, H)
    o = oracle.combine(bf(rows), np.arange(T, dtype=np.int32)[:, None], np.ones((T, 1), np.float32),
                       quant="mxfp4")
    assert o["scales"].tolist() == scales
    got = np.stack([o["quant"] & 15, o["quant"] >> 4], axis=-1).reshape(T, H)
    c = np.concatenate(codes).reshape(T, H)
    nz = (c & 7) != 0
    assert np.array_equal(got[nz], c[nz]) and np.all((got[~nz] & 7) == 0)
    assert np.array_equal(oracle.dequant(o["quant"], o["scales"], T, H, "mxfp4"), rows)


def test_low_precision_weights_equal_their_fp32_values():
    T, k, E, H = 20, 4, 8, 64
    ids, row_map, nv = _routing(T, k, E)
    rows = bf(RNG.standard_normal((nv, H)))
    w32 = np.array(RNG.dirichlet(np.ones(k), T), np.float32)
    for name, enc, dec in (("bf16", bf, f), ("fp16", oracle.f64_to_f16, oracle.f16_to_f64)):
        wbits = enc(w32)
        a = oracle.combine(rows, row_map, wbits, weight_dtype=name, quant="mxfp8")
        b = oracle.combine(rows, row_map, dec(wbits).astype(np.float32), quant="mxfp8")
        for key in ("combined", "y", "quant", "scales"):
            assert np.array_equal(a[key], b[key]), (name, key)


def test_fp16_io_agrees_with_bf16_on_values_both_hold_exactly():
    # small dyadic values are exact in both formats and so are their sums,
    # so the fp16 and bf16 paths must produce the same numbers
    T, k, E, H = 12, 3, 6, 32
    ids, row_map, nv = _routing(T, k, E)
    vals = RNG.integers(-16, 17, (nv, H)) / 8.0
    w = (2.0 ** -RNG.integers(0, 3, (T, k))).astype(np.float32)
    res = RNG.integers(-8, 9, (T, H)) / 4.0
    ob = oracle.combine(bf(vals), row_map, w, residual=bf(res), outputs=("combined", "residual"))
    oh = oracle.combine(oracle.f64_to_f16(vals), row_map, w, residual=oracle.f64_to_f16(res),
                        outputs=("combined", "residual"), io_dtype="fp16")
    for key in ("combined", "residual"):
        assert np.array_equal(f(ob[key]), oracle.f16_to_f64(oh[key])), key
