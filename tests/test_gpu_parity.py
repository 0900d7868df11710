"""GPU parity: the CUDA path through the C ABI against the oracle, element by
element, on the seeded synthetic workloads and on edge cases.

Routing is compared bit-exactly.  Combine outputs use the tolerances stated
in tests/_helpers.py.  The largest workloads (T = 16384) are compared on a
sample of token rows, which the oracle computes one by one; everything else
is compared in full.
"""
import dataclasses

import numpy as np
import pytest
import torch

import norm_quant_gb300 as nqg
import oracle
from norm_quant_gb300 import synth
from norm_quant_gb300.build import build

from _helpers import (DEV, assert_bf16_close, assert_quant_close, d, dec16, gpu_combine, gpu_route, h,
                      nvfp4_global_scale, oracle_combine, sum_magnitude)

pytestmark = pytest.mark.gpu

GAMMA_K = lambda k: (k + 3) * 2.0 ** -24  # noqa: E731


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build()
    nqg.lib()


def route_and_check(ids, E, stream=None):
    st, counts, offsets, row_map, src_row = gpu_route(ids, E, stream=stream)
    ost, oc, oo, orm, osr = oracle.build_row_map(ids, E)
    assert st == (nqg.MOE_OK if ost == 0 else nqg.MOE_ERR_INVALID_EXPERT)
    assert np.array_equal(h(counts), oc)
    assert np.array_equal(h(offsets), oo)
    assert np.array_equal(h(row_map), orm)
    assert np.array_equal(h(src_row)[: oo[E]], osr)
    return row_map, orm


def compare(wl, inp, orm, got, tokens=None, global_scale=1.0, expert_layout="grouped"):
    T, H, k = wl.T, wl.H, wl.k
    tok = np.arange(T) if tokens is None else np.asarray(tokens)
    o = oracle_combine(wl, inp, orm, tokens=None if tokens is None else tok, global_scale=global_scale,
                       expert_layout=expert_layout)
    assert o["status"] == 0
    io = wl.io_dtype
    mag = sum_magnitude(inp, orm, tok, io, wl.weight_dtype)
    floor = GAMMA_K(k) * mag
    for name in ("combined", "residual"):
        if name in got:
            assert_bf16_close(got[name][tok], o[name], floor, f"{wl.name}:{name}", io)
    if "norm" in got:
        res = dec16(o["residual"], io)
        rinv = 1.0 / np.sqrt((res ** 2).mean(axis=1, keepdims=True) + wl.eps)
        g = np.abs(dec16(inp["gamma"], io) + wl.weight_bias)[None, :]
        # the sum's bound carried through y = x * rinv * (gamma + wb): once
        # directly and once through rinv's dependence on x; the fp32 rounding
        # of rinv and of the two products (a few parts in 2^24) lies far
        # inside the 2 ulps of the 16-bit output
        nfloor = 2 * floor * rinv * g
        assert_bf16_close(got["norm"][tok], o["norm"], nfloor, f"{wl.name}:norm", io)
    if wl.quant and "quant" in got:
        vec = 16 if wl.quant == "nvfp4" else 32
        Cc = H // vec
        if tokens is None:
            assert_quant_close(wl, got["quant"], got["scales"], o["quant"], o["scales"], T, H,
                               global_scale, f"{wl.name}:quant")
            if wl.sf_layout == "swizzled":
                # every byte outside the real (row, column) cells is zero padding
                used = np.zeros(got["scales"].size, bool)
                used[oracle.sf_offsets(T, Cc, "swizzled").ravel()] = True
                assert np.all(got["scales"][~used] == 0)
        else:
            lin = got["scales"][oracle.sf_offsets(T, Cc, wl.sf_layout)][tok].ravel()
            assert_quant_close(wl, got["quant"][tok], lin, o["quant"], o["scales"], tok.size, H,
                               global_scale, f"{wl.name}:quant", layout="linear")


def run_workload(wl, sample=None, canary=False):
    inp = synth.make_inputs(wl)
    d_rm, orm = route_and_check(inp["topk_ids"], wl.E)
    g = nvfp4_global_scale(wl, inp, orm) if wl.quant == "nvfp4" else 1.0
    got = gpu_combine(wl, inp, d_rm, global_scale=g, canary=canary)
    assert got["status"] == 0
    tokens = None
    if sample is not None and wl.T > sample:
        rng = np.random.Generator(np.random.PCG64(wl.seed + 7))
        tokens = np.unique(np.concatenate([[0, wl.T - 1], rng.choice(wl.T, sample, replace=False)]))
    compare(wl, inp, orm, got, tokens=tokens, global_scale=g)
    return inp, orm, got


# ---------------------------------------------------------------- workloads

@pytest.mark.parametrize("wl", synth.WORKLOADS, ids=lambda w: w.name)
def test_workload_parity(wl):
    run_workload(wl, sample=384 if wl.T > 8192 else None, canary=wl.T <= 4096)


@pytest.mark.parametrize("T", synth.SWEEP_T)
def test_padded_sweep_parity(T):
    run_workload(synth.sweep_point(T), sample=256 if T > 4096 else None)


# -------------------------------------------------------------- edge cases

def _wl(**kw):
    base = dict(name="edge", T=37, H=256, E=16, k=4, residual=True, gamma_mean=1.0,
                outputs=("combined", "residual", "norm"), seed=77)
    base.update(kw)
    return synth.Workload(**base)


@pytest.mark.parametrize("kw", [
    dict(k=1), dict(k=32, E=64), dict(E=1, k=1), dict(H=8, outputs=("combined",), gamma_mean=None),
    dict(H=32, quant="mxfp8", outputs=("combined", "quant")),
    dict(H=16, quant="nvfp4", outputs=("residual", "quant"), gamma_mean=0.0, weight_bias=1.0),
    dict(H=7200, T=19, quant="mxfp8", outputs=("residual", "norm", "quant")),   # ragged last slot
    dict(H=16384, T=9, k=8, E=32, quant="mxfp8", outputs=("residual", "quant")),  # largest H
    # every limit at once (largest H, top_k and E): a few tokens (split over
    # clusters), then enough for whole rows
    dict(H=16384, T=5, k=32, E=8192, shared_std=0.5, quant="nvfp4", sf_layout="swizzled",
         outputs=("residual", "norm", "quant")),
    dict(H=16384, T=200, k=32, E=8192, quant="mxfp8", outputs=("combined", "residual", "norm", "quant")),
    dict(H=8192, T=13, quant="nvfp4", sf_layout="swizzled", outputs=("residual", "quant")),
    dict(H=96, T=130, quant="mxfp8", sf_layout="swizzled", outputs=("norm", "quant")),  # C = 3 pads
    dict(H=48, T=200, quant="nvfp4", sf_layout="swizzled", outputs=("combined", "quant")),
    dict(pad_frac=1.0, shared_std=0.5, quant="mxfp8", outputs=("combined", "residual", "quant")),
    dict(pad_frac=0.5, outputs=("combined", "residual", "norm")),
    dict(T=1, H=7168, E=256, k=8, shared_std=0.5, quant="mxfp8", outputs=("residual", "norm", "quant")),
    dict(T=3000, H=512, E=8, k=8, dist="zipf", zipf_s=2.0, weight_bias=0.375),
    dict(eps=0.5, gamma_std=1.0),
], ids=lambda kw: ",".join(f"{a}={b}" for a, b in kw.items()))
def test_edge_parity(kw):
    wl = _wl(**kw)
    inp = synth.make_inputs(wl)
    d_rm, orm = route_and_check(inp["topk_ids"], wl.E)
    g = nvfp4_global_scale(wl, inp, orm) if wl.quant == "nvfp4" else 1.0
    got = gpu_combine(wl, inp, d_rm, global_scale=g, canary=True)
    assert got["status"] == 0
    compare(wl, inp, orm, got, global_scale=g)


def test_duplicate_experts_in_a_token():
    rng = np.random.Generator(np.random.PCG64(5))
    ids = rng.integers(0, 4, (300, 8)).astype(np.int32)
    ids[rng.random((300, 8)) < 0.1] = -1
    route_and_check(ids, 4)


@pytest.mark.parametrize("cluster", [0, -1, 1, 4, 8])
def test_routing_paths_and_determinism(cluster):
    nqg.moe_tuning_set(route_cluster=cluster)
    try:
        _routing_sizes()
    finally:
        nqg.moe_tuning_set()


def _routing_sizes():
    rng = np.random.Generator(np.random.PCG64(6))
    # the one-CTA path (T * k <= 2048, E <= 1024, automatic plan), the
    # single-launch cluster path and (E > 512 or N > 262144) the three-kernel path
    for T, k, E in [(1, 1, 1), (3, 2, 8192), (1000, 32, 5), (5000, 8, 1024), (70000, 2, 3),
                    (40000, 8, 256), (33000, 8, 16), (2000, 8, 2048), (32768, 8, 256),
                    (16384, 8, 256), (70000, 8, 64), (64, 8, 256), (256, 8, 256), (257, 8, 256),
                    (200, 10, 1024), (7, 3, 1), (97, 1, 33), (128, 16, 1000)]:
        ids = rng.integers(-1, E, (T, k)).astype(np.int32)
        a = route_and_check(ids, E)[0]
        b = gpu_route(ids, E)[3]
        assert torch.equal(a, b)


def test_single_launch_routing_is_planned_at_the_workload_sizes():
    """The one-cluster routing build is the plan at every workload's size
    (a plan that silently fell back to three kernels would still pass the
    parity tests), and route_cluster = -1 selects the three kernels."""
    for wl in synth.WORKLOADS:
        assert nqg.moe_build_row_map_launches(wl.T, wl.k, wl.E) == 1, wl.name
    assert nqg.moe_build_row_map_launches(16384, 8, 256) == 1
    assert nqg.moe_build_row_map_launches(40000, 8, 256) == 3  # beyond one cluster's slots
    try:
        nqg.moe_tuning_set(route_cluster=-1)
        assert nqg.moe_build_row_map_launches(64, 8, 256) == 3
    finally:
        nqg.moe_tuning_set()


def test_routing_duplicate_heavy_small_builds_match_the_oracle():
    """Small builds where most slots share one expert (long runs of equal
    keys within and across warps of the one-CTA kernel)."""
    rng = np.random.Generator(np.random.PCG64(61))
    for T, k, E in [(256, 8, 4), (100, 8, 2), (2048 // 8, 8, 1024)]:
        ids = np.where(rng.random((T, k)) < 0.9, 1 % E, rng.integers(-1, E, (T, k))).astype(np.int32)
        route_and_check(ids, E)


def test_invalid_expert_ids_are_flagged():
    ids = np.array([[0, 1], [9, -1], [-5, 2]], np.int32)
    st, counts, offsets, row_map, _ = gpu_route(ids, 4)
    assert st == nqg.MOE_ERR_INVALID_EXPERT
    assert h(row_map).tolist() == [[0, 1], [-1, -1], [-1, 2]]
    assert h(counts).tolist() == [1, 1, 1, 0]


@pytest.mark.parametrize("bad", ["E", "E+1000", "-2", "-1000"])
@pytest.mark.parametrize("path", ["one_cta", "cluster", "three_kernels"])
def test_each_kind_of_invalid_id_alone_on_every_routing_path(bad, path):
    """One invalid id (at or above E, or below -1) among valid ones is
    reported and treated as padding by each routing kernel; everything else
    matches the oracle bit for bit."""
    T, k, E = (64, 8, 256) if path == "one_cta" else (1024, 8, 256)
    rng = np.random.Generator(np.random.PCG64(4040))
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    ids[T // 2, k // 2] = {"E": E, "E+1000": E + 1000, "-2": -2, "-1000": -1000}[bad]
    try:
        nqg.moe_tuning_set(route_cluster=-1 if path == "three_kernels" else 0)
        assert nqg.moe_build_row_map_launches(T, k, E) == (3 if path == "three_kernels" else 1)
        route_and_check(ids, E)
    finally:
        nqg.moe_tuning_set()
    ost = oracle.build_row_map(ids, E)[0]
    assert ost == 4


def test_empty_batch_is_a_noop():
    st, counts, offsets, row_map, _ = gpu_route(np.zeros((0, 4), np.int32), 8)
    assert st == 0 and h(counts).tolist() == [0] * 8 and h(offsets).tolist() == [0] * 9
    out = torch.full((16,), 0x1234, dtype=torch.int16, device="cuda")
    nqg.moe_combine(expert_out=torch.zeros((0, 64), dtype=torch.int16, device="cuda"),
                    row_map=torch.zeros((0, 2), dtype=torch.int32, device="cuda"),
                    router_weights=torch.zeros((0, 2), dtype=torch.float32, device="cuda"),
                    combined_out=out, H=64)
    torch.cuda.synchronize()
    assert torch.all(out == 0x1234)


def test_row_out_of_range_is_reported_and_skipped():
    wl = _wl(T=8, H=64, outputs=("combined",), residual=False, gamma_mean=None)
    inp = synth.make_inputs(wl)
    _, orm = route_and_check(inp["topk_ids"], wl.E)
    bad = orm.copy()
    bad[2, 1] = inp["n_valid"] + 5
    got = gpu_combine(wl, inp, d(bad))
    assert got["status"] == nqg.MOE_ERR_ROW_OUT_OF_RANGE
    skip = orm.copy()
    skip[2, 1] = -1
    o = oracle_combine(wl, inp, skip)
    assert_bf16_close(got["combined"], o["combined"], GAMMA_K(wl.k) * sum_magnitude(inp, skip, range(8)),
                      "skipped slot")


def test_bounded_wait_timeout_is_reported_and_the_context_survives():
    """A wait that runs out (CTA 0's producer stops staging rows through the
    test hook) is reported as MOE_ERR_DEVICE_TIMEOUT after the 2 s limit,
    without a fault; the next call on the same context is fully correct."""
    wl = _wl(T=300, H=7168, k=8, E=256, shared_std=0.5, quant="mxfp8", outputs=("residual", "quant"))
    inp = synth.make_inputs(wl)
    d_rm, orm = route_and_check(inp["topk_ids"], wl.E)
    try:
        nqg.moe_debug_stall(1)
        got = gpu_combine(wl, inp, d_rm)
    finally:
        nqg.moe_debug_stall(-1)
    assert got["status"] == nqg.MOE_ERR_DEVICE_TIMEOUT
    again = gpu_combine(wl, inp, d_rm, canary=True)
    assert again["status"] == 0
    compare(wl, inp, orm, again)


def test_split_rows_timeout_is_reported_and_the_context_survives():
    """At decode sizes a token is split over a cluster.  The test hook stops
    CTA 0's producer, so CTA 0's consumers give up on their first slot and
    never send their partial sums; its peers send theirs and give up on the
    exchange after 2 s.  Every thread still completes the cluster's
    arrive-wait sequence, so the call ends, reports MOE_ERR_DEVICE_TIMEOUT,
    and the next call on the same context is exact."""
    wl = _wl(T=8, H=7168, k=8, E=256, outputs=("residual", "norm"))
    assert nqg.moe_build_row_map_launches(wl.T, wl.k, wl.E) >= 1
    inp = synth.make_inputs(wl)
    d_rm, orm = route_and_check(inp["topk_ids"], wl.E)
    try:
        nqg.moe_debug_stall(0)
        got = gpu_combine(wl, inp, d_rm)
    finally:
        nqg.moe_debug_stall(-1)
    assert got["status"] == nqg.MOE_ERR_DEVICE_TIMEOUT
    again = gpu_combine(wl, inp, d_rm, canary=True)
    assert again["status"] == 0
    compare(wl, inp, orm, again)


def test_concurrent_calls_from_two_host_threads():
    """Two host threads call the combine at once, on their own streams, with
    workloads that need different shared-memory sizes (and so different
    kernel attributes); both match the oracle."""
    import threading
    cases = [dataclasses.replace(synth.PREFILL, T=200, name="thread_mxfp8"),
             dataclasses.replace(synth.GEMMA_NVFP4, T=150, name="thread_nvfp4")]
    prepared = []
    for wl in cases:
        inp = synth.make_inputs(wl)
        d_rm, orm = route_and_check(inp["topk_ids"], wl.E)
        g = nvfp4_global_scale(wl, inp, orm) if wl.quant == "nvfp4" else 1.0
        prepared.append((wl, inp, d_rm, orm, g))
    results, errors = [None] * len(cases), []

    def run(i):
        try:
            wl, inp, d_rm, orm, g = prepared[i]
            s = torch.cuda.Stream()
            out = []
            for _ in range(3):
                with torch.cuda.stream(s):
                    out.append(gpu_combine(wl, inp, d_rm, global_scale=g, stream=s))
            results[i] = out
        except Exception as e:  # reported below, in the main thread
            errors.append(e)

    threads = [threading.Thread(target=run, args=(i,)) for i in range(len(cases))]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    for (wl, inp, d_rm, orm, g), outs in zip(prepared, results):
        for got in outs:
            assert got["status"] == 0
            compare(wl, inp, orm, got, global_scale=g)


def test_repeat_runs_identical_and_side_stream():
    wl = dataclasses.replace(synth.PREFILL, T=700, name="repeat")
    inp = synth.make_inputs(wl)
    d_rm, orm = route_and_check(inp["topk_ids"], wl.E)
    a = gpu_combine(wl, inp, d_rm)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        d_rm2, _ = route_and_check(inp["topk_ids"], wl.E, stream=s)
        b = gpu_combine(wl, inp, d_rm2, stream=s)
    for key in ("residual", "quant", "scales"):
        assert np.array_equal(a[key], b[key])


@pytest.mark.parametrize("mode", ["eager", "graph"])
@pytest.mark.parametrize("T", [64, 4096], ids=["one_cta_build", "cluster_build"])
def test_consecutive_layers_on_one_stream(T, mode):
    """Two routings alternate on one stream, as consecutive MoE layers do: a
    kernel writes each build's ids just before it, and each build overwrites
    the row_map that the previous combine is reading.  Builds and combines are
    launched as programmatic dependents of their predecessors, so their
    launches overlap the previous kernel; neither order may break, launched
    directly or replayed from a CUDA graph (where the dependencies become
    programmatic graph edges)."""
    wl = dataclasses.replace(synth.DECODE, T=T, name=f"layers_T{T}")
    E, k, H = wl.E, wl.k, wl.H
    inps = [synth.make_inputs(wl, seed=wl.seed + 11 * i) for i in range(2)]
    key = 0x35A5A  # the ids are stored scrambled and restored by a kernel
    enc = [d(inp["topk_ids"].astype(np.int32) ^ key) for inp in inps]
    dev = [{n: d(inp[n]) for n in ("expert_out", "weights", "residual", "gamma")} for inp in inps]
    ids = torch.empty((T, k), dtype=torch.int32, device=DEV)
    counts = torch.empty(E, dtype=torch.int32, device=DEV)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    row_map = torch.empty((T, k), dtype=torch.int32, device=DEV)
    ws = torch.zeros(nqg.moe_build_row_map_workspace_size(T, k, E), dtype=torch.uint8, device=DEV)
    seq = [0, 1, 0, 1, 0, 1]
    outs = [{n: torch.full((T, H), 0x5A5A, dtype=torch.int16, device=DEV) for n in ("residual", "norm")}
            for _ in seq]
    s = torch.cuda.Stream()

    def layers():
        for i, which in enumerate(seq):
            torch.bitwise_xor(enc[which], key, out=ids)
            nqg.moe_build_row_map(ids, E, counts, offsets, row_map, None, ws, stream=s.cuda_stream)
            x = dev[which]
            nqg.moe_combine(stream=s.cuda_stream, expert_out=x["expert_out"].reshape(-1, H), row_map=row_map,
                            router_weights=x["weights"], residual=x["residual"], gamma=x["gamma"], eps=wl.eps,
                            residual_out=outs[i]["residual"], norm_out=outs[i]["norm"], H=H)

    torch.cuda.synchronize()
    if mode == "graph":
        with torch.cuda.stream(s):
            layers()  # the first calls configure the kernels, outside the capture
        torch.cuda.synchronize()
        for o in outs:
            for t in o.values():
                t.fill_(0x5A5A)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            layers()
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            g.replay()
    else:
        with torch.cuda.stream(s):
            layers()
    torch.cuda.synchronize()
    assert nqg.moe_build_row_map_check(ws) == nqg.MOE_OK
    got = [{n: h(t, np.uint16) for n, t in o.items()} for o in outs]
    for which in (0, 1):
        _, _, _, orm, _ = oracle.build_row_map(inps[which]["topk_ids"], E)
        compare(wl, inps[which], orm, got[which])
    for i in range(2, len(seq)):
        for n in ("residual", "norm"):
            assert np.array_equal(got[i][n], got[i - 2][n]), f"call {i}: {n}"
    assert not np.array_equal(got[0]["residual"], got[1]["residual"])


@pytest.mark.parametrize("mode", ["eager", "graph"])
@pytest.mark.parametrize("T", [64, 2048], ids=["one_cta_build", "cluster_build"])
def test_layer_with_identity_experts(T, mode):
    """A whole MoE layer on one stream with identity experts: the routing
    build, the dispatch permute of the token rows, then the combine reading
    the rows the permute has just written, each launch a programmatic
    dependent of the one before.  The permuted rows must equal the oracle's
    permute, and the combine's outputs the oracle's combine of those rows."""
    wl = dataclasses.replace(synth.DECODE, T=T, name=f"identity_layer_T{T}")
    E, k, H = wl.E, wl.k, wl.H
    inp = synth.make_inputs(wl)
    x = synth.bf16_normal(np.random.Generator(np.random.PCG64(T + 5)), (T, H))  # the token rows
    _, _, oo, orm, _ = oracle.build_row_map(inp["topk_ids"], E)
    nv = int(oo[E])
    st, xg_want = oracle.dispatch_permute(x, orm, nv)
    assert st == 0
    d_ids, d_x, d_w, d_res, d_g = (d(a) for a in (inp["topk_ids"], x, inp["weights"], inp["residual"], inp["gamma"]))
    counts = torch.empty(E, dtype=torch.int32, device=DEV)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    row_map = torch.empty((T, k), dtype=torch.int32, device=DEV)
    ws = torch.zeros(nqg.moe_build_row_map_workspace_size(T, k, E), dtype=torch.uint8, device=DEV)
    xg = torch.empty((nv, H), dtype=torch.int16, device=DEV)
    outs = {n: torch.empty((T, H), dtype=torch.int16, device=DEV) for n in ("residual", "norm")}
    s = torch.cuda.Stream()

    def layer():
        nqg.moe_build_row_map(d_ids, E, counts, offsets, row_map, None, ws, stream=s.cuda_stream)
        nqg.moe_dispatch_permute(d_x, row_map, xg, stream=s.cuda_stream)
        nqg.moe_combine(stream=s.cuda_stream, expert_out=xg, row_map=row_map, router_weights=d_w,
                        residual=d_res, gamma=d_g, eps=wl.eps, residual_out=outs["residual"],
                        norm_out=outs["norm"], H=H)

    def clear():
        for t in (row_map, xg, *outs.values()):
            t.fill_(-1)

    torch.cuda.synchronize()
    if mode == "graph":
        with torch.cuda.stream(s):
            layer()  # the first calls configure the kernels, outside the capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            layer()
        clear()
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            g.replay()
    else:
        clear()
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            layer()
    torch.cuda.synchronize()
    assert nqg.moe_build_row_map_check(ws) == nqg.MOE_OK
    assert np.array_equal(h(row_map), orm)
    assert np.array_equal(h(xg, np.uint16), xg_want)
    compare(wl, dict(inp, expert_out=xg_want, n_valid=nv), orm, {n: h(t, np.uint16) for n, t in outs.items()})


@pytest.mark.parametrize("plan", [(1, 1, 0, 0), (1, 4, 0, 0), (2, 1, 0, 0), (2, 4, 32, 0), (4, 1, 0, 0),
                                  (4, 2, 200, 0), (8, 1, 0, 0), (2, 2, 64, 2), (2, 2, 16, 3),
                                  (2, 8, 0, 0), (1, 5, 0, 0), (4, 6, 0, 0), (8, 8, 0, 0), (2, 3, 0, 0),
                                  (1, 12, 0, 0), (2, 9, 0, 0)],
                         ids=lambda p: "vpt%d_rows%d_ring%d_cta%d" % p)
def test_every_launch_plan_matches_the_oracle(plan):
    """moe_tuning_set changes only how the work is laid out on the GPU."""
    cases = [dataclasses.replace(synth.PREFILL, T=300, name="plan_mxfp8"),
             dataclasses.replace(synth.GEMMA_NVFP4, T=257, name="plan_nvfp4")]
    try:
        nqg.moe_tuning_set(*plan)
        for wl in cases:
            run_workload(wl, canary=True)
    finally:
        nqg.moe_tuning_set()


@pytest.mark.parametrize("kw", [
    dict(T=300, H=7168, k=8, shared_std=0.5, quant="mxfp8", outputs=("residual", "quant")),
    dict(T=257, H=4096, k=8, gamma_mean=0.0, weight_bias=1.0, quant="nvfp4", sf_layout="swizzled",
         outputs=("residual", "quant")),
    dict(T=33, H=7200, k=4, shared_std=0.5, outputs=("combined", "residual", "norm")),
    dict(T=5, H=64, k=1, residual=False, gamma_mean=None, outputs=("combined",)),
], ids=["prefill_like_mxfp8", "gemma_like_nvfp4", "ragged_h", "k1_gather"])
def test_slot_major_layout_parity(kw):
    """The slot-major expert layout [k, T, H] with per-(token, slot) scales
    (trtllm_moe_allreduce_fusion's moe_reduction_* inputs) against the oracle."""
    wl = _wl(**{"E": 1, **kw})
    inp = synth.make_slot_major_inputs(wl)
    g = nvfp4_global_scale(wl, inp, None, "slot_major") if wl.quant == "nvfp4" else 1.0
    got = gpu_combine(wl, inp, None, global_scale=g, canary=True, expert_layout="slot_major")
    assert got["status"] == 0
    compare(wl, inp, None, got, global_scale=g, expert_layout="slot_major")


@pytest.mark.parametrize("T,H,k,E", [(4096, 7168, 8, 256), (1, 8, 1, 1), (333, 7200, 4, 16),
                                     (2000, 4096, 8, 128), (64, 16384, 8, 256)])
def test_dispatch_permute_parity(T, H, k, E):
    """Every expert-grouped row gets its token's row, bit for bit; rows no
    slot names keep their previous contents."""
    rng = np.random.Generator(np.random.PCG64(T + H))
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    ids[rng.random((T, k)) < 0.1] = -1
    d_rm, orm = route_and_check(ids, E)
    nv = int((ids >= 0).sum())
    x = synth.bf16_normal(rng, (T, H))
    n_rows = nv + 5
    xg = torch.full((n_rows, H), 0x3F80, dtype=torch.int16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    nqg.moe_dispatch_permute(d(x), d_rm, xg, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    st, want = oracle.dispatch_permute(x, orm, n_rows, fill=0x3F80)
    assert st == 0
    assert np.array_equal(h(xg, np.uint16), want)


def test_dispatch_bounded_wait_timeout_is_reported():
    """The permute's bounded wait runs out when CTA 0 issues no more row
    loads (test hook): MOE_ERR_DEVICE_TIMEOUT, no fault, and the next call on
    the same context is exact."""
    T, H, k, E = 500, 1024, 8, 64
    rng = np.random.Generator(np.random.PCG64(12))
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    d_rm, orm = route_and_check(ids, E)
    x = synth.bf16_normal(rng, (T, H))
    xg = torch.zeros((T * k, H), dtype=torch.int16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    try:
        nqg.moe_debug_stall(0)  # CTA 0 owns one token here (one CTA per token): load none
        nqg.moe_dispatch_permute(d(x), d_rm, xg, status=status)
        torch.cuda.synchronize()
    finally:
        nqg.moe_debug_stall(-1)
    assert int(status.item()) == nqg.MOE_ERR_DEVICE_TIMEOUT
    status.zero_()
    nqg.moe_dispatch_permute(d(x), d_rm, xg, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    st, want = oracle.dispatch_permute(x, orm, T * k)
    assert np.array_equal(h(xg, np.uint16), want)


def test_dispatch_permute_reports_out_of_range_rows():
    T, H, k = 8, 64, 2
    x = synth.bf16_normal(np.random.Generator(np.random.PCG64(3)), (T, H))
    rm = np.arange(T * k, dtype=np.int32).reshape(T, k)
    rm[3, 1] = 10_000
    xg = torch.zeros((T * k, H), dtype=torch.int16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    nqg.moe_dispatch_permute(d(x), d(rm), xg, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == nqg.MOE_ERR_ROW_OUT_OF_RANGE
    st, want = oracle.dispatch_permute(x, rm, T * k)
    assert np.array_equal(h(xg, np.uint16), want)


@pytest.mark.parametrize("kw", [
    dict(T=300, H=7168, k=8, E=64, shared_std=0.5, quant="mxfp4", outputs=("residual", "quant")),
    dict(T=130, H=96, k=4, quant="mxfp4", sf_layout="swizzled", outputs=("norm", "quant")),
    dict(T=200, H=4096, k=8, E=128, gamma_mean=0.0, weight_bias=1.0, quant="mxfp4", sf_layout="swizzled",
         outputs=("residual", "quant")),
    dict(T=257, H=7168, k=8, E=256, shared_std=0.5, io_dtype="fp16",
         outputs=("combined", "residual", "norm")),
    dict(T=257, H=4096, k=8, E=128, io_dtype="fp16", gamma_mean=0.0, weight_bias=1.0, quant="nvfp4",
         sf_layout="swizzled", outputs=("residual", "quant")),
    dict(T=300, H=7168, k=8, E=256, shared_std=0.5, weight_dtype="bf16", quant="mxfp8",
         outputs=("residual", "quant")),
    dict(T=100, H=2048, k=6, E=32, weight_dtype="fp16", io_dtype="fp16", quant="mxfp4",
         outputs=("combined", "norm", "quant")),
], ids=["mxfp4_prefill_like", "mxfp4_swizzled_pad", "mxfp4_gemma_like", "fp16_io_norm",
        "fp16_io_nvfp4", "bf16_weights_mxfp8", "fp16_weights_fp16_io_mxfp4"])
def test_dtype_and_mxfp4_parity(kw):
    """MXFP4 output (UE8M0 per 32, e2m1 codes), fp16 inputs and outputs, and
    bf16 / fp16 router weights, against the oracle."""
    wl = _wl(**kw)
    inp = synth.make_inputs(wl)
    d_rm, orm = route_and_check(inp["topk_ids"], wl.E)
    g = nvfp4_global_scale(wl, inp, orm) if wl.quant == "nvfp4" else 1.0
    got = gpu_combine(wl, inp, d_rm, global_scale=g, canary=True)
    assert got["status"] == 0
    compare(wl, inp, orm, got, global_scale=g)



def _f16_edge_inputs(wl, seed):
    """fp16 inputs with the values an unwidened fp16 product must get right:
    subnormal and large row elements, negative zeros, and subnormal, negative
    and greater-than-one fp16 router weights."""
    inp = synth.make_inputs(wl)
    rng = np.random.Generator(np.random.PCG64(seed))
    ex = inp["expert_out"].copy()
    u = rng.random(ex.shape)
    sign = (rng.integers(0, 2, ex.shape) << 15).astype(np.uint16)
    sub = rng.integers(1, 0x400, ex.shape).astype(np.uint16) | sign       # subnormal
    big = rng.integers(0x6400, 0x6C00, ex.shape).astype(np.uint16) | sign  # [1024, 4096)
    ex = np.where(u < 0.02, sub, np.where(u < 0.03, big, np.where(u < 0.035, np.uint16(0x8000), ex)))
    inp["expert_out"] = ex.astype(np.uint16)
    w = inp["weights"].copy()
    v = rng.random(w.shape)
    w = np.where(v < 0.1, rng.integers(1, 0x400, w.shape).astype(np.uint16),  # subnormal weight
                 np.where(v < 0.15, np.uint16(0x4300),                         # 3.5
                          np.where(v < 0.2, np.uint16(0xBA00), w)))            # -0.75
    inp["weights"] = w.astype(np.uint16)
    return inp


@pytest.mark.parametrize("plan", [None, (1, 3, 0), (2, 8, 0), (4, 6, 0), (8, 12, 0), (0, 0, 2), (0, 0, 4)],
                         ids=["auto", "vpt1_r3", "vpt2_r8", "vpt4_r6", "vpt8_r12", "split2", "split4"])
def test_fp16_weights_kernel_matches_widening_bit_for_bit(plan):
    """fp16 rows with fp16 weights run a kernel that multiplies without
    widening (mixed-precision fma).  On edge values it agrees with the
    oracle, and bit for bit with the widening kernel given the same weights
    as fp32, in every launch plan."""
    wl = _wl(T=37, H=2048, k=8, E=64, shared_std=0.5, io_dtype="fp16", weight_dtype="fp16",
             quant="mxfp8", outputs=("combined", "residual", "norm", "quant"), seed=91)
    inp = _f16_edge_inputs(wl, seed=92)
    d_rm, orm = route_and_check(inp["topk_ids"], wl.E)
    wl32 = dataclasses.replace(wl, weight_dtype="fp32")
    inp32 = dict(inp, weights=inp["weights"].view(np.float16).astype(np.float32))
    try:
        if plan is not None:
            vpt, rows, split = plan
            nqg.moe_tuning_set(vpt, rows, 0, 0, 0, split)
        got = gpu_combine(wl, inp, d_rm, canary=True)
        ref = gpu_combine(wl32, inp32, d_rm, canary=True)
    finally:
        nqg.moe_tuning_set()
    assert got["status"] == 0 and ref["status"] == 0
    for name in ("combined", "residual", "norm", "quant", "scales"):
        assert np.array_equal(got[name], ref[name]), name
    compare(wl, inp, orm, got)



@pytest.mark.parametrize("io,wdt", [("fp16", "fp32"), ("fp16", "fp16"), ("bf16", "fp32"), ("bf16", "bf16")])
def test_pure_gather_returns_every_finite_code(io, wdt):
    """top_k = 1 with weight 1, no other rows and no norm: the combined
    output is the expert row itself, so every finite 16-bit code (all 63,488
    of fp16, all 65,280 of bf16) comes back unchanged, except -0, which
    becomes +0 (the sum starts from +0).  This checks the widening of rows
    and weights and the rounding back, exhaustively."""
    H = 2048 if io == "fp16" else 256
    n_exp = 31 if io == "fp16" else 255             # biased exponents of the finite codes
    mant = 1024 if io == "fp16" else 128
    shift = 10 if io == "fp16" else 7
    e = np.repeat(np.arange(n_exp, dtype=np.uint32), 2 * mant)
    m = np.tile(np.arange(mant, dtype=np.uint32), 2 * n_exp)
    sg = np.tile(np.repeat(np.array([0, 0x8000], np.uint32), mant), n_exp)
    codes = (sg | (e << shift) | m).astype(np.uint16).reshape(n_exp, H)
    T = n_exp
    one = {"fp32": np.float32(1.0), "fp16": np.uint16(0x3C00), "bf16": np.uint16(0x3F80)}[wdt]
    weights = np.full((T, 1), one)
    ids = np.zeros((T, 1), np.int32)
    d_rm, orm = route_and_check(ids, 1)
    rows = np.empty_like(codes)
    rows[orm[:, 0]] = codes                          # expert row row_map[t] holds token t's codes
    ex = torch.from_numpy(rows.view(np.int16)).cuda()
    out = torch.full((T, H), 0x5A5A, dtype=torch.int16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    nqg.moe_combine(expert_out=ex, row_map=d_rm, router_weights=torch.from_numpy(weights).cuda(),
                    combined_out=out, status=status, H=H, io_dtype=io, weight_dtype=wdt)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    want = np.where(codes == 0x8000, np.uint16(0), codes)
    got = h(out, np.uint16)
    bad = got != want
    assert not bad.any(), [(hex(int(want[i])), hex(int(got[i]))) for i in map(tuple, np.argwhere(bad)[:5])]


# ------------------------------------------------- split rows (decode sizes)

SPLIT_CASES = [
    # the decode workload's shape: residual + norm, bf16 outputs
    dict(T=64, H=7168, k=8, E=256, outputs=("residual", "norm")),
    # shared row and combined_out (stored before the residual row lands), MXFP8
    dict(T=23, H=7168, k=8, E=256, shared_std=0.5, quant="mxfp8",
         outputs=("combined", "residual", "quant")),
    # Gemma form, NVFP4 with swizzled scales (pad rows and columns)
    dict(T=5, H=4096, k=8, E=128, gamma_mean=0.0, weight_bias=1.0, quant="nvfp4", sf_layout="swizzled",
         outputs=("residual", "norm", "quant")),
    # fp16 inputs and outputs, fp16 router weights, MXFP4
    dict(T=7, H=2048, k=6, E=32, io_dtype="fp16", weight_dtype="fp16", quant="mxfp4",
         outputs=("combined", "norm", "quant")),
    # many tokens per cluster: the reduction buffers alternate many times
    dict(T=700, H=4096, k=8, E=128, shared_std=0.5, quant="mxfp8", outputs=("residual", "norm", "quant")),
    # padded tokens (no expert rows) and no residual
    dict(T=40, H=1024, k=4, E=16, pad_frac=0.5, residual=False, outputs=("combined", "norm")),
]


@pytest.mark.parametrize("split", [0, 1, 2, 4, 8, 16])
@pytest.mark.parametrize("kw", SPLIT_CASES,
                         ids=["decode", "shared_mxfp8", "gemma_nvfp4", "fp16_mxfp4", "many_tokens", "padded"])
def test_split_rows_parity(kw, split):
    """A token's row split by columns over a cluster of 2..16 CTAs (their
    sums of squares exchanged through distributed shared memory) gives the
    oracle's outputs, as whole rows do."""
    wl = _wl(**kw)
    inp = synth.make_inputs(wl)
    d_rm, orm = route_and_check(inp["topk_ids"], wl.E)
    g = nvfp4_global_scale(wl, inp, orm) if wl.quant == "nvfp4" else 1.0
    try:
        nqg.moe_tuning_set(combine_split=split)
        got = gpu_combine(wl, inp, d_rm, global_scale=g, canary=True)
    finally:
        nqg.moe_tuning_set()
    assert got["status"] == 0
    compare(wl, inp, orm, got, global_scale=g)


@pytest.mark.parametrize("split", [2, 16])
def test_split_rows_slot_major_and_unsplittable_h(split):
    """The split path with the slot-major layout, and a forced split on an H
    that no cluster divides into whole MXFP8 blocks (whole rows are used)."""
    wl = _wl(T=9, H=7168, k=8, E=1, shared_std=0.5, quant="mxfp8", outputs=("residual", "quant"))
    inp = synth.make_slot_major_inputs(wl)
    wl2 = _wl(T=11, H=7200, k=8, E=64, quant="mxfp8", outputs=("residual", "norm", "quant"))
    inp2 = synth.make_inputs(wl2)
    d_rm2, orm2 = route_and_check(inp2["topk_ids"], wl2.E)
    try:
        nqg.moe_tuning_set(combine_split=split)
        got = gpu_combine(wl, inp, None, canary=True, expert_layout="slot_major")
        got2 = gpu_combine(wl2, inp2, d_rm2, canary=True)
    finally:
        nqg.moe_tuning_set()
    assert got["status"] == 0 and got2["status"] == 0
    compare(wl, inp, None, got, expert_layout="slot_major")
    compare(wl2, inp2, orm2, got2)


def test_split_rows_repeatable():
    """The cross-CTA norm adds the partials in one fixed order: two runs of
    the split path are bit-identical."""
    wl = _wl(T=64, H=7168, k=8, E=256, quant="mxfp8", outputs=("residual", "norm", "quant"))
    inp = synth.make_inputs(wl)
    d_rm, _ = route_and_check(inp["topk_ids"], wl.E)
    try:
        nqg.moe_tuning_set(combine_split=8)
        a = gpu_combine(wl, inp, d_rm)
        b = gpu_combine(wl, inp, d_rm)
    finally:
        nqg.moe_tuning_set()
    for key in ("residual", "norm", "quant", "scales"):
        assert np.array_equal(a[key], b[key])


# ------------------------------------------------- NVFP4 midpoint golden --

def test_nvfp4_midpoint_golden_exact_on_gpu():
    # hand-derived blocks whose elements divided by their block scale sit
    # exactly on e2m1 midpoints (tests/golden/nvfp4_midpoints.json): the
    # kernel divides, so its bytes are the golden ones, not the bytes that
    # multiplying by the scale's reciprocal would give
    import json
    import os
    g = json.load(open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                                    "nvfp4_midpoints.json")))
    H = g["H"]
    row = synth.f32_to_bf16_bits(np.array(g["row"], np.float32))[None, :]
    q = torch.full((H // 2,), 0x5A, dtype=torch.uint8, device="cuda")
    sc = torch.full((nqg.moe_scales_bytes(1, H, "nvfp4", "linear"),), 0x5A, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    nqg.moe_combine(expert_out=d(row), row_map=d(np.zeros((1, 1), np.int32)),
                    router_weights=d(np.ones((1, 1), np.float32)), quant="nvfp4", sf_layout="linear",
                    global_scale=g["global_scale"], quant_out=q, scales_out=sc, status=status, H=H)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert h(sc).tolist() == [int(v, 16) for v in g["expect"]["scales"]]
    assert h(q).tolist() == [int(v, 16) for v in g["expect"]["bytes"]]


# ------------------------------------- exact sums: quantisers bit for bit --

def _exact_sum_inputs(T, H, k, E, seed, shared=True):
    """Inputs whose weighted sums are exact in fp32 whatever the order: rows of
    6-bit integers times 2^-6..2^2 (exact in bf16), weights 2^-0..2^-3.  The
    kernel then quantises exactly the oracle's value, so every code and scale
    byte must agree; integer-valued data also puts many elements exactly on
    rounding midpoints of the e4m3 and e2m1 grids."""
    rng = np.random.Generator(np.random.PCG64(seed))
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    ids[rng.random((T, k)) < 0.05] = -1
    ost, oc, oo, orm, osr = oracle.build_row_map(ids, E)
    nv = int(oo[E])

    def vals(shape):
        m = rng.integers(-48, 49, shape).astype(np.float64)
        e = rng.integers(-6, 3, shape[:-1] + (1,)).astype(np.float64)   # one exponent per row
        return synth.f32_to_bf16_bits((m * 2.0 ** e).astype(np.float32))

    inp = {"topk_ids": ids, "n_valid": nv, "expert_out": vals((nv, H)),
           "weights": (2.0 ** -rng.integers(0, 4, (T, k))).astype(np.float32),
           "shared": vals((T, H)) if shared else None, "residual": vals((T, H)), "gamma": None}
    return inp, orm


@pytest.mark.parametrize("quant,layout", [("mxfp8", "linear"), ("mxfp8", "swizzled"), ("nvfp4", "linear"),
                                          ("nvfp4", "swizzled"), ("mxfp4", "linear")])
def test_quantisers_bit_exact_on_exact_sums(quant, layout):
    T, H, k, E = 301, 512, 8, 32
    inp, orm = _exact_sum_inputs(T, H, k, E, seed=11 + len(quant) + len(layout))
    wl = synth.Workload(name=f"exact_{quant}_{layout}", T=T, H=H, E=E, k=k, shared_std=1.0, residual=True,
                        quant=quant, sf_layout=layout, outputs=("combined", "residual", "quant"))
    g = 1.0   # NVFP4's global scale: a power of two keeps g * y exact (other g: the workload tests)
    got = gpu_combine(wl, inp, d(orm), global_scale=g, canary=True)
    assert got["status"] == 0
    o = oracle_combine(wl, inp, orm, global_scale=g)
    assert np.array_equal(got["combined"], o["combined"])
    assert np.array_equal(got["residual"], o["residual"])
    assert np.array_equal(got["scales"], o["scales"]), "scale bytes"
    assert np.array_equal(got["quant"], o["quant"]), f"{int((got['quant'] != o['quant']).sum())} code bytes differ"
    if quant == "nvfp4":
        # the data reaches the case the element quotient exists for: elements
        # exactly on an e2m1 midpoint of their block scale
        y = oracle.combine(inp["expert_out"], orm, inp["weights"], shared=inp["shared"],
                           residual=inp["residual"], outputs=("y",))["y"]
        v = (np.float32(g) * y.astype(np.float32)).astype(np.float64).reshape(T, H // 16, 16)
        s = oracle.e4m3_to_f64(o["scales"][oracle.sf_offsets(T, H // 16, layout)])[:, :, None]
        mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
        on_mid = np.any(np.abs(v)[..., None] == mids * s[..., None], axis=-1)
        assert on_mid.sum() > 50, on_mid.sum()


# ----------------------------- swizzled scales: pad rows at any alignment --

@pytest.mark.parametrize("offset", [0, 1, 4, 8])
@pytest.mark.parametrize("quant,T", [("nvfp4", 1), ("nvfp4", 37), ("mxfp8", 5), ("mxfp8", 130)])
def test_swizzled_scales_pad_rows_at_any_alignment(quant, T, offset):
    # the scale buffer may start at any byte; its pad rows (T % 128 .. 127 of
    # the last row tile) are zeroed with 16-byte, 4-byte or 1-byte stores as
    # the start allows, and no byte outside the buffer is touched
    H = 208 if quant == "nvfp4" else 224   # 13 or 7 scale columns, padded to 16 / 8
    wl = synth.Workload(name=f"swz_{quant}_{T}_{offset}", T=T, H=H, E=8, k=2, residual=True,
                        quant=quant, sf_layout="swizzled", outputs=("residual", "quant"), seed=T + offset)
    inp = synth.make_inputs(wl)
    d_rm, orm = route_and_check(inp["topk_ids"], wl.E)
    g = nvfp4_global_scale(wl, inp, orm) if quant == "nvfp4" else 1.0
    n = nqg.moe_scales_bytes(T, H, quant, "swizzled")
    buf = torch.full((n + 64,), 0x5A, dtype=torch.uint8, device="cuda")
    scales = buf[offset:offset + n]
    q = torch.empty((T, H if quant == "mxfp8" else H // 2), dtype=torch.uint8, device="cuda")
    res = torch.empty((T, H), dtype=torch.int16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    nqg.moe_combine(expert_out=d(inp["expert_out"]), row_map=d_rm, router_weights=d(inp["weights"]),
                    residual=d(inp["residual"]), quant=quant, sf_layout="swizzled", global_scale=g,
                    residual_out=res, quant_out=q, scales_out=scales, status=status, H=H)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    o = oracle_combine(wl, inp, orm, global_scale=g)
    b = h(buf)
    assert np.all(b[:offset] == 0x5A) and np.all(b[offset + n:] == 0x5A), "bytes outside the scale buffer"
    got = b[offset:offset + n]
    used = np.zeros(n, bool)
    used[oracle.sf_offsets(T, H // (16 if quant == "nvfp4" else 32), "swizzled").ravel()] = True
    assert np.all(got[~used] == 0), "pad bytes not zero"
    assert_quant_close(wl, h(q), got, o["quant"], o["scales"], T, H, g, wl.name)
