"""Shared machinery of the parity tests: run a workload through the C ABI on
the GPU and through the oracle on the CPU, and compare with the stated
tolerances.

Tolerances (the accuracy bar for this path, with the fp32 rounding terms of
the kernel's sums added):
  * routing (counts, offsets, row_map, src_row): bit-exact;
  * bf16 outputs: |gpu - oracle| <= 2 bf16 ulps of the oracle value plus
    gamma_k * (sum of |terms|), gamma_k = (k + 3) * 2^-24 the fp32 forward
    error bound of the (k + 2)-term sum, carried through the norm's scale;
  * block scales: identical bytes except in at most 0.01 % of blocks, which
    may differ by one step;
  * dequantised values: within one quantisation step of the coarser of the
    two block scales.
"""
from __future__ import annotations

import numpy as np
import torch

import norm_quant_gb300 as nqg
import oracle

DEV = "cuda"


def d(a: np.ndarray) -> torch.Tensor:
    """numpy -> CUDA tensor, byte-for-byte (uint16 bf16 bits travel as int16)."""
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def h(t: torch.Tensor, dtype=None) -> np.ndarray:
    a = t.cpu().numpy()
    if dtype is not None:
        a = a.view(dtype)
    return a


def gpu_route(ids: np.ndarray, E: int, stream=None):
    T, k = ids.shape
    d_ids = d(ids.astype(np.int32))
    counts = torch.full((E,), -7, dtype=torch.int32, device=DEV)
    offsets = torch.full((E + 1,), -7, dtype=torch.int32, device=DEV)
    row_map = torch.full((T, k), -7, dtype=torch.int32, device=DEV)
    src_row = torch.full((max(T * k, 1),), -7, dtype=torch.int32, device=DEV)
    ws = torch.zeros(nqg.moe_build_row_map_workspace_size(T, k, E), dtype=torch.uint8, device=DEV)
    nqg.moe_build_row_map(d_ids, E, counts, offsets, row_map, src_row, ws, stream=stream)
    st = nqg.moe_build_row_map_check(ws, stream=stream)
    return st, counts, offsets, row_map, src_row


def gpu_combine(wl, inp, d_row_map, *, global_scale=1.0, outputs=None, stream=None,
                canary=False, expert_layout="grouped"):
    """Runs moe_combine for workload `wl` on device copies of `inp`.
    Returns host numpy outputs (bf16 as uint16 bits) and the status word."""
    T, H, k = wl.T, wl.H, wl.k
    outputs = outputs or wl.outputs
    ex = d(inp["expert_out"]) if inp["n_valid"] else torch.zeros((0, H), dtype=torch.int16, device=DEV)
    ex = ex.reshape(-1, H)
    w = d(inp["weights"])
    sh = d(inp["shared"]) if inp["shared"] is not None else None
    rs = d(inp["residual"]) if inp["residual"] is not None else None
    gm = d(inp["gamma"]) if inp["gamma"] is not None else None
    pad = 4096 if canary else 0

    def out(n, dtype):
        buf = torch.full((n + 2 * pad,), 0x5A if dtype == torch.uint8 else 0x5A5A, dtype=dtype,
                         device=DEV)
        return buf, buf[pad:pad + n]

    bufs, views = {}, {}
    for name in ("combined", "residual", "norm"):
        if name in outputs:
            bufs[name], views[name] = out(T * H, torch.int16)
    if wl.quant and "quant" in outputs:
        qn = T * H if wl.quant == "mxfp8" else T * H // 2  # fp4: two codes per byte
        bufs["quant"], views["quant"] = out(qn, torch.uint8)
        sn = nqg.moe_scales_bytes(T, H, wl.quant, wl.sf_layout)
        bufs["scales"], views["scales"] = out(sn, torch.uint8)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    nqg.moe_combine(stream=stream, expert_out=ex, row_map=d_row_map, router_weights=w,
                    shared_out=sh, residual=rs, gamma=gm, eps=wl.eps, weight_bias=wl.weight_bias,
                    quant=wl.quant, sf_layout=wl.sf_layout, global_scale=global_scale,
                    combined_out=views.get("combined"), residual_out=views.get("residual"),
                    norm_out=views.get("norm"), quant_out=views.get("quant"),
                    scales_out=views.get("scales"), status=status, H=H, expert_layout=expert_layout,
                    io_dtype=wl.io_dtype, weight_dtype=wl.weight_dtype)
    torch.cuda.synchronize()
    res = {"status": int(status.item())}
    for name, v in views.items():
        res[name] = h(v, np.uint16 if v.dtype == torch.int16 else np.uint8)
        if canary:
            b = h(bufs[name], np.uint16 if v.dtype == torch.int16 else np.uint8)
            fill = 0x5A5A if v.dtype == torch.int16 else 0x5A
            assert np.all(b[:pad] == fill) and np.all(b[pad + v.numel():] == fill), f"{name} overrun"
    for name in ("combined", "residual", "norm"):
        if name in res:
            res[name] = res[name].reshape(T, H)
    if "quant" in res:
        res["quant"] = res["quant"].reshape(T, -1)
    return res


def oracle_combine(wl, inp, row_map, *, tokens=None, global_scale=1.0,
                   sf_layout=None, expert_layout="grouped"):
    """Oracle outputs for all tokens, or for the listed token rows only
    (then in linear scale layout, indexed by position in `tokens`)."""
    sel = slice(None) if tokens is None else np.asarray(tokens)
    pick = (lambda a: a) if tokens is None else (lambda a: None if a is None else a[sel])
    if expert_layout == "slot_major":
        assert tokens is None, "the slot-major oracle runs on whole batches"
        return oracle.combine(
            inp["expert_out"], None, inp["weights"], shared=inp["shared"], residual=inp["residual"],
            gamma=inp["gamma"], eps=wl.eps, weight_bias=wl.weight_bias, quant=wl.quant,
            sf_layout=sf_layout or wl.sf_layout, global_scale=global_scale, expert_layout="slot_major",
            io_dtype=wl.io_dtype, weight_dtype=wl.weight_dtype)
    return oracle.combine(
        inp["expert_out"], row_map[sel], inp["weights"][sel], shared=pick(inp["shared"]),
        residual=pick(inp["residual"]), gamma=inp["gamma"], eps=wl.eps,
        weight_bias=wl.weight_bias, quant=wl.quant,
        sf_layout=(sf_layout or (wl.sf_layout if tokens is None else "linear")),
        global_scale=global_scale, io_dtype=wl.io_dtype, weight_dtype=wl.weight_dtype)


def bf16_ulp(x: np.ndarray, io="bf16") -> np.ndarray:
    """Spacing of the 16-bit output format at |x| (bf16: 8 significant bits,
    normal down to 2^-126; fp16: 11 bits, normal down to 2^-14)."""
    a = np.abs(x)
    if io == "fp16":
        e = np.floor(np.log2(np.maximum(a, 2.0 ** -14)))
        return 2.0 ** (e - 10)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return 2.0 ** (e - 7)


def dec16(bits, io="bf16") -> np.ndarray:
    return oracle.f16_to_f64(bits) if io == "fp16" else oracle.bf16_to_f64(bits)


def dec_weights(w, dtype="fp32") -> np.ndarray:
    if dtype == "fp32":
        return np.asarray(w, np.float64)
    return dec16(w, "fp16" if dtype == "fp16" else "bf16")


def sum_magnitude(inp, row_map, tokens, io="bf16", weight_dtype="fp32") -> np.ndarray:
    """Per element sum of |terms| of x = sum_j w x_j + shared + residual
    (row_map None: the slot-major layout [k, T, H])."""
    tokens = np.asarray(tokens)
    H = inp["expert_out"].shape[-1] if inp["n_valid"] else (
        inp["residual"].shape[1] if inp["residual"] is not None else 1)
    mag = np.zeros((tokens.size, H))
    rows = inp["expert_out"]
    wts = dec_weights(inp["weights"], weight_dtype)
    if row_map is None:
        k, T = rows.shape[0], rows.shape[1]
        row_map = (np.arange(k)[None, :] * T + np.arange(T)[:, None]).astype(np.int32)
        rows = rows.reshape(k * T, H)
    for i, t in enumerate(tokens):
        for j in range(row_map.shape[1]):
            r = row_map[t, j]
            if r >= 0:
                mag[i] += abs(float(wts[t, j])) * np.abs(dec16(rows[r], io))
        if inp["shared"] is not None:
            mag[i] += np.abs(dec16(inp["shared"][t], io))
        if inp["residual"] is not None:
            mag[i] += np.abs(dec16(inp["residual"][t], io))
    return mag


def assert_bf16_close(got: np.ndarray, want: np.ndarray, abs_floor, what: str, io="bf16"):
    g = dec16(got, io)
    w = dec16(want, io)
    tol = 2 * bf16_ulp(w, io) + abs_floor
    bad = np.abs(g - w) > tol
    if bad.any():
        i = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} beyond tolerance; "
                             f"first {[(tuple(x), g[tuple(x)], w[tuple(x)]) for x in i]}")


def quant_step(codes_deq_scaled: np.ndarray, quant: str) -> np.ndarray:
    """Spacing of the element grid at a scaled magnitude (e4m3 or e2m1)."""
    a = np.abs(codes_deq_scaled)
    if quant == "mxfp8":
        e = np.floor(np.log2(np.maximum(a, 2.0 ** -6)))
        return 2.0 ** (e - 3)          # subnormal spacing 2^-9 below 2^-6
    return np.where(a < 2.0, 0.5, np.where(a < 4.0, 1.0, 2.0))   # e2m1 (NVFP4, MXFP4)


def assert_quant_close(wl, got_q, got_s, want_q, want_s, T, H, global_scale, what,
                       layout=None):
    layout = layout or wl.sf_layout
    vec = 16 if wl.quant == "nvfp4" else 32
    Cc = H // vec
    idx = oracle.sf_offsets(T, Cc, layout)
    gs, ws = got_s[idx], want_s[idx]
    diff = gs.astype(np.int64) - ws.astype(np.int64)
    n_bad = int((diff != 0).sum())
    assert n_bad <= int(1e-4 * diff.size), f"{what}: {n_bad} of {diff.size} scale bytes differ"
    assert np.all(np.abs(diff) <= 1), f"{what}: a scale byte differs by more than one step"
    dg = oracle.dequant(got_q, got_s, T, H, wl.quant, layout, global_scale)
    dw = oracle.dequant(want_q, want_s, T, H, wl.quant, layout, global_scale)
    if wl.quant in ("mxfp8", "mxfp4"):
        sc = 2.0 ** (np.maximum(gs, ws).astype(np.float64) - 127)
    else:
        sc = np.maximum(oracle.e4m3_to_f64(gs), oracle.e4m3_to_f64(ws)) / global_scale
    sc = np.repeat(sc, vec, axis=1)
    with np.errstate(divide="ignore", invalid="ignore"):
        scaled = np.where(sc > 0, np.maximum(np.abs(dg), np.abs(dw)) / sc, 0.0)
    step = quant_step(scaled, wl.quant) * sc
    bad = np.abs(dg - dw) > step
    assert not bad.any(), f"{what}: {int(bad.sum())} dequantised values beyond one step"
    same = (got_q == want_q).mean()
    assert same >= 0.999, f"{what}: only {same:.5f} of code bytes identical"


def nvfp4_global_scale(wl, inp, row_map, expert_layout="grouped") -> float:
    """g = fp32(448 * 6 / amax(y)) over the whole tensor, from the oracle's y."""
    o = oracle.combine(inp["expert_out"], row_map, inp["weights"], shared=inp["shared"],
                       residual=inp["residual"], gamma=inp["gamma"], eps=wl.eps,
                       weight_bias=wl.weight_bias, outputs=("y",), expert_layout=expert_layout,
                       io_dtype=wl.io_dtype, weight_dtype=wl.weight_dtype)
    amax = float(np.abs(o["y"]).max())
    return float(np.float32(448.0 * 6.0 / amax)) if amax > 0 else 1.0
