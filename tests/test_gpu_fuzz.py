"""Randomised parity: seeded draws over the combine's whole configuration
space (shape, quantiser and scale layout, I/O and router-weight dtypes,
optional inputs and outputs, expert layout, padding, routing skew and launch
plan, split rows included), each compared with the oracle element by element.
The draws are fixed by the seed, so a failure names a reproducible case."""
import dataclasses

import numpy as np
import pytest
import torch

import norm_quant_gb300 as nqg
from norm_quant_gb300 import synth

from _helpers import gpu_combine, nvfp4_global_scale
from test_gpu_parity import compare, route_and_check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from norm_quant_gb300.build import build
    build()
    nqg.lib()


_BLOCK = {None: 8, "mxfp8": 32, "mxfp4": 32, "nvfp4": 16}
_PLANS = [None, (2, 0, 0, 0, 0), (1, 3, 0, 0, 0), (4, 6, 0, 0, 0), (8, 8, 0, 0, 0), (0, 12, 0, 0, 0),
          (0, 0, 48, 0, 0), (0, 2, 0, 2, 0), (0, 0, 0, 0, 2), (0, 0, 0, 0, 4)]


def _draw(i, rng):
    quant = [None, "mxfp8", "nvfp4", "mxfp4"][int(rng.integers(4))]
    blk = _BLOCK[quant]
    H = int(blk * rng.integers(1, 16384 // blk + 1)) if rng.random() < 0.2 else \
        int(blk * rng.integers(1, 4096 // blk + 1))
    k = int(rng.integers(1, 13))
    E = int(rng.integers(k, 300))
    T = int(rng.integers(1, max(2, min(600, 1_500_000 // H))))
    gamma = rng.random() < 0.7
    outs = [o for o in ("combined", "residual", "norm") if rng.random() < 0.5 and (o != "norm" or gamma)]
    if quant:
        outs.append("quant")
    if not outs:
        outs = ["combined"]
    wl = synth.Workload(
        name=f"fuzz{i}", T=T, H=H, E=E, k=k,
        dist="zipf" if rng.random() < 0.3 else "uniform", zipf_s=1.2,
        pad_frac=float([0.0, 0.0, 0.1, 0.5][int(rng.integers(4))]),
        shared_std=0.5 if rng.random() < 0.5 else None, residual=bool(rng.random() < 0.7),
        gamma_mean=(0.0 if rng.random() < 0.3 else 1.0) if gamma else None,
        weight_bias=float([0.0, 1.0, 0.375][int(rng.integers(3))]), quant=quant,
        sf_layout=["linear", "swizzled"][int(rng.integers(2))], outputs=tuple(outs), seed=5000 + i,
        io_dtype=["bf16", "fp16"][int(rng.integers(2))],
        weight_dtype=["fp32", "bf16", "fp16"][int(rng.integers(3))])
    layout = "slot_major" if rng.random() < 0.2 else "grouped"
    plan = _PLANS[int(rng.integers(len(_PLANS)))]
    return wl, layout, plan


@pytest.mark.parametrize("i", range(160))
def test_random_configuration_matches_the_oracle(i):
    wl, layout, plan = _draw(i, np.random.Generator(np.random.PCG64(7700 + i)))
    if layout == "slot_major":
        wl = dataclasses.replace(wl, E=1, pad_frac=0.0)
        inp = synth.make_slot_major_inputs(wl)
        d_rm, orm = None, None
    else:
        inp = synth.make_inputs(wl)
        d_rm, orm = route_and_check(inp["topk_ids"], wl.E)
    g = nvfp4_global_scale(wl, inp, orm, layout) if wl.quant == "nvfp4" else 1.0
    try:
        if plan is not None:
            vpt, rows, ring, cta, split = plan
            nqg.moe_tuning_set(vpt, rows, ring, cta, 0, split)
        got = gpu_combine(wl, inp, d_rm, global_scale=g, canary=True, expert_layout=layout)
    finally:
        nqg.moe_tuning_set()
    torch.cuda.synchronize()
    assert got["status"] == 0, (wl, layout, plan)
    compare(wl, inp, orm, got, global_scale=g, expert_layout=layout)


@pytest.mark.parametrize("i", range(60))
def test_random_routing_build_matches_the_oracle(i):
    """Seeded draws of T, top_k, E, padding, invalid ids and routing path
    (automatic, three kernels, or a cluster cap); counts, offsets, row_map
    and src_row bit-exact against the oracle."""
    rng = np.random.Generator(np.random.PCG64(9100 + i))
    k = int(rng.integers(1, 33))
    E = int([rng.integers(1, 9), rng.integers(1, 300), rng.integers(1, 8193)][int(rng.integers(3))])
    T = int([rng.integers(1, 300), rng.integers(1, 5000), rng.integers(1, 500_000 // k + 1)][int(rng.integers(3))])
    ids = rng.integers(0, E, (T, k)).astype(np.int32)
    ids[rng.random((T, k)) < rng.choice([0.0, 0.1, 0.5])] = -1
    if rng.random() < 0.15:
        ids[rng.random((T, k)) < 0.001] = E + 3  # out of range: reported, treated as padding
    cluster = int(rng.choice([0, 0, 0, -1, 1, 2, 4, 8, 16]))
    try:
        nqg.moe_tuning_set(route_cluster=cluster)
        route_and_check(ids, E)
    finally:
        nqg.moe_tuning_set()


@pytest.mark.parametrize("i", range(30))
def test_random_dispatch_permute_matches_the_oracle(i):
    """Seeded draws of T, H, top_k and E; the dispatch permute writes every
    grouped row bit-exactly as the oracle does, and leaves the others."""
    from _helpers import d, h
    import oracle
    rng = np.random.Generator(np.random.PCG64(9300 + i))
    k = int(rng.integers(1, 17))
    E = int(rng.integers(k, 400))
    H = int(8 * rng.integers(1, 16384 // 8 + 1)) if rng.random() < 0.3 else int(8 * rng.integers(1, 1025))
    T = int(rng.integers(1, max(2, min(3000, 4_000_000 // (H * k)))))
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    ids[rng.random((T, k)) < 0.1] = -1
    d_rm, orm = route_and_check(ids, E)
    x = synth.bf16_normal(rng, (T, H))
    n_rows = int((ids >= 0).sum()) + int(rng.integers(0, 4))
    xg = torch.full((max(n_rows, 1), H), 0x3F80, dtype=torch.int16, device="cuda")[:n_rows]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    nqg.moe_dispatch_permute(d(x), d_rm, xg, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    st, want = oracle.dispatch_permute(x, orm, n_rows, fill=0x3F80)
    assert np.array_equal(h(xg, np.uint16), want)
