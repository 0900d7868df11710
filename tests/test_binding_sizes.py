"""The Python binding's buffer-size checks, on the CPU.

The kernels take plain pointers, so the binding refuses (ValueError) a
tensor smaller than the call reads or writes.  The checks run before any
pointer is taken, so CPU tensors reach them: a well-sized call then stops at
the "must be CUDA tensors" check, a short buffer at its own name."""
import numpy as np
import pytest
import torch

import norm_quant_gb300 as nqg
import oracle
from norm_quant_gb300 import synth
from norm_quant_gb300.build import build

import _helpers


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build()
    nqg.lib()


def _combine_kw(T=5, H=64, k=2, quant="mxfp8", sf_layout="swizzled", weight_dtype="fp32"):
    z = lambda *shape, dt=torch.int16: torch.zeros(shape, dtype=dt)  # noqa: E731
    return dict(expert_out=z(T * k, H), row_map=z(T, k, dt=torch.int32),
                router_weights=z(T, k, dt=torch.float32 if weight_dtype == "fp32" else torch.int16),
                shared_out=z(T, H), residual=z(T, H), gamma=z(H), combined_out=z(T, H), residual_out=z(T, H),
                norm_out=z(T, H), quant=quant, sf_layout=sf_layout,
                quant_out=z(T * (H if quant == "mxfp8" else H // 2), dt=torch.uint8),
                scales_out=z(nqg.moe_scales_bytes(T, H, quant, sf_layout), dt=torch.uint8),
                status=z(1, dt=torch.int32), weight_dtype=weight_dtype)


def _expect(kw, what):
    with pytest.raises(ValueError) as e:
        nqg.combine_args(**kw)
    assert what in str(e.value), str(e.value)


@pytest.mark.parametrize("quant,layout", [("mxfp8", "swizzled"), ("nvfp4", "linear"), ("mxfp4", "swizzled")])
def test_well_sized_buffers_pass_and_short_ones_are_named(quant, layout):
    kw = _combine_kw(quant=quant, sf_layout=layout)
    _expect(kw, "CUDA")  # every size is right: stops at the device check
    # (router_weights sets T and top_k by its shape; its dtype case is below)
    for name in ("row_map", "shared_out", "residual", "gamma", "combined_out",
                 "residual_out", "norm_out", "quant_out", "scales_out", "status"):
        short = dict(kw)
        short[name] = kw[name].flatten()[:-1]
        _expect(short, name)


def test_two_byte_weights_declared_fp32_are_refused():
    kw = _combine_kw(weight_dtype="fp16")
    _expect(kw, "CUDA")
    _expect(dict(kw, weight_dtype="fp32"), "router_weights")


def test_slot_major_needs_every_slot_row():
    kw = _combine_kw()
    kw.update(row_map=None, expert_layout="slot_major")
    _expect(kw, "CUDA")
    _expect(dict(kw, expert_out=kw["expert_out"][:-1]), "expert_out")


@pytest.mark.parametrize("T,H,quant", [(1, 32, "mxfp8"), (130, 96, "mxfp8"), (7, 48, "nvfp4"),
                                       (300, 224, "nvfp4"), (70, 64, "mxfp4"), (0, 64, "nvfp4")])
def test_scale_size_rule_matches_the_library_and_the_oracle(T, H, quant):
    vec = 16 if quant == "nvfp4" else 32
    for layout in ("linear", "swizzled"):
        n = nqg._scales_bytes(T, H, vec, layout)
        assert n == nqg.moe_scales_bytes(T, H, quant, layout) == oracle.scales_bytes(T, H, quant, layout)


def test_routing_and_dispatch_buffers():
    ids = torch.zeros((4, 2), dtype=torch.int32)
    ok = dict(counts=torch.zeros(8, dtype=torch.int32), offsets=torch.zeros(9, dtype=torch.int32),
              row_map=torch.zeros((4, 2), dtype=torch.int32))
    for name in ok:
        args = dict(ok, **{name: ok[name].flatten()[:-1]})
        with pytest.raises(ValueError, match=name):
            nqg.moe_build_row_map(ids, 8, args["counts"], args["offsets"], args["row_map"])
    with pytest.raises(ValueError, match="CUDA"):
        nqg.moe_build_row_map(ids, 8, ok["counts"], ok["offsets"], ok["row_map"])
    x = torch.zeros((4, 64), dtype=torch.int16)
    with pytest.raises(ValueError, match="status"):
        nqg.moe_dispatch_permute(x, ok["row_map"], torch.zeros((8, 64), dtype=torch.int16),
                                 status=torch.zeros(0, dtype=torch.int32))


def test_every_parity_test_buffer_passes_the_size_checks(monkeypatch):
    """The GPU parity tests' own allocation helper, pointed at the CPU, on
    the tiny and decode workloads and on every fourth randomised draw: each
    call gets through the size checks (it stops at the device check)."""
    import test_gpu_fuzz
    monkeypatch.setattr(_helpers, "DEV", "cpu")
    cases = [(synth.TINY, "grouped"), (synth.DECODE, "grouped")]
    cases += [test_gpu_fuzz._draw(i, np.random.Generator(np.random.PCG64(7700 + i)))[:2] for i in range(0, 160, 4)]
    for wl, layout in cases:
        if layout == "slot_major":
            import dataclasses
            wl = dataclasses.replace(wl, E=1, pad_frac=0.0)
            inp, d_rm = synth.make_slot_major_inputs(wl), None
        else:
            inp = synth.make_inputs(wl)
            d_rm = _helpers.d(oracle.build_row_map(inp["topk_ids"], wl.E)[3])
        with pytest.raises(ValueError, match="CUDA"):
            _helpers.gpu_combine(wl, inp, d_rm, global_scale=1.0, canary=True, expert_layout=layout)
