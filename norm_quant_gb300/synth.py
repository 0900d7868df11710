"""Seeded synthetic inputs for the MoE combine/finalize step.

This module only draws random numbers.  It holds none of the combine's
arithmetic, and both the CUDA path's tests/bench and the CPU oracle consume
what it makes.  Everything comes from ``numpy.random.Generator(PCG64(seed))``.

Workload shapes follow the pages' setting: DeepSeek-style hidden 7168 with 256
experts and top_k 8, decode to prefill token counts, plus a Gemma-style
(weight_bias = 1) NVFP4 case at hidden 4096 with 128 experts.

* expert picks: k distinct experts per token.  Uniform, or Zipf-skewed with
  p(e) proportional to (e + 1)^-s (expert 0 hottest).  Sampling without
  replacement by sequential renormalised draws is done with the Gumbel-top-k
  construction, which has exactly that distribution.
* router weights: fp32 softmax of N(0, 1) logits over the k picks.
* padded tokens (when pad_frac > 0): floor(pad_frac * T) token rows, picked
  by a seeded permutation, get all ids = -1 and weight 0.
* expert_out: bf16 N(0, 1) rows, one per valid (token, slot) entry.  Rows are
  i.i.d., so their order in the expert-grouped buffer does not change the
  distribution.
* shared: bf16 N(0, shared_std); residual: bf16 N(0, 1);
  gamma: bf16 N(gamma_mean, gamma_std).  The second parameter is the standard
  deviation.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    E: int
    k: int
    dist: str = "uniform"          # "uniform" | "zipf"
    zipf_s: float = 0.0
    pad_frac: float = 0.0
    shared_std: Optional[float] = None   # None: no shared-expert row
    residual: bool = False
    gamma_mean: Optional[float] = None   # None: no RMSNorm
    gamma_std: float = 0.1
    eps: float = 1e-6
    weight_bias: float = 0.0
    quant: Optional[str] = None          # None | "mxfp8" | "nvfp4"
    sf_layout: str = "linear"            # "linear" | "swizzled"
    outputs: tuple = ("combined",)       # subset of combined/residual/norm/quant
    seed: int = 0
    io_dtype: str = "bf16"               # element type of the 16-bit tensors: bf16 | fp16
    weight_dtype: str = "fp32"           # router weights: fp32 | bf16 | fp16

    def with_T(self, T: int, seed: Optional[int] = None) -> "Workload":
        return dataclasses.replace(self, T=T, seed=self.seed if seed is None else seed)


# The five workloads.  Seeds: 1000 + index; sweep points use 2000 + T.
TINY = Workload("tiny_combine_T16_H256_E8_k2", T=16, H=256, E=8, k=2,
                outputs=("combined",), seed=1001)
DECODE = Workload("decode_T64_H7168_E256_k8_rmsnorm_bf16", T=64, H=7168, E=256, k=8,
                  residual=True, gamma_mean=1.0, gamma_std=0.1, eps=1e-6,
                  outputs=("residual", "norm"), seed=1002)
PREFILL = Workload("prefill_T4096_H7168_E256_k8_zipf1.1_shared_rmsnorm_mxfp8",
                   T=4096, H=7168, E=256, k=8, dist="zipf", zipf_s=1.1,
                   shared_std=0.5, residual=True, gamma_mean=1.0, gamma_std=0.1,
                   eps=1e-6, quant="mxfp8", sf_layout="linear",
                   outputs=("residual", "quant"), seed=1003)
GEMMA_NVFP4 = Workload("gemma_T8192_H4096_E128_k8_wb1_nvfp4_128x4",
                       T=8192, H=4096, E=128, k=8, residual=True, gamma_mean=0.0,
                       gamma_std=0.1, eps=1e-6, weight_bias=1.0, quant="nvfp4",
                       sf_layout="swizzled", outputs=("residual", "quant"), seed=1004)
PADDED = Workload("padded_T16384_H7168_E256_k8_zipf1.3_pad10_rmsnorm_mxfp8",
                  T=16384, H=7168, E=256, k=8, dist="zipf", zipf_s=1.3, pad_frac=0.1,
                  residual=True, gamma_mean=1.0, gamma_std=0.1, eps=1e-6,
                  quant="mxfp8", sf_layout="linear", outputs=("residual", "quant"),
                  seed=1005)
WORKLOADS = [TINY, DECODE, PREFILL, GEMMA_NVFP4, PADDED]
SWEEP_T = (1, 8, 64, 512, 4096, 16384)


def sweep_point(T: int) -> Workload:
    return dataclasses.replace(PADDED, name=f"padded_sweep_T{T}", T=T, seed=2000 + T)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def draw_routing(wl: Workload, rng: np.random.Generator):
    """topk_ids int32 [T, k] (-1 = padded) and router weights fp32 [T, k]."""
    T, E, k = wl.T, wl.E, wl.k
    if k > E:
        raise ValueError("top_k must not exceed the number of experts")
    if wl.dist == "zipf":
        logp = -wl.zipf_s * np.log(np.arange(1, E + 1, dtype=np.float64))
    else:
        logp = np.zeros(E)
    ids = np.empty((T, k), np.int32)
    step = 4096
    for t0 in range(0, T, step):
        t1 = min(T, t0 + step)
        keys = logp[None, :] + rng.gumbel(size=(t1 - t0, E))
        ids[t0:t1] = np.argsort(-keys, axis=1, kind="stable")[:, :k]
    logits = rng.standard_normal((T, k))
    w = np.exp(logits - logits.max(axis=1, keepdims=True))
    w = (w / w.sum(axis=1, keepdims=True)).astype(np.float32)
    n_pad = int(np.floor(wl.pad_frac * T))
    if n_pad:
        pad = rng.permutation(T)[:n_pad]
        ids[pad] = -1
        w[pad] = 0.0
    return ids, w


def f32_to_f16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> IEEE binary16 bit patterns, round to nearest even."""
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def bf16_normal(rng: np.random.Generator, shape, std=1.0, mean=0.0, io="bf16") -> np.ndarray:
    """bf16 (or, with io="fp16", binary16) bit patterns of N(mean, std)
    draws, generated in row blocks."""
    out = np.empty(shape, np.uint16)
    flat = out.reshape(-1, shape[-1]) if len(shape) > 1 else out.reshape(1, -1)
    rows_per = max(1, (1 << 24) // max(1, flat.shape[1]))
    for r0 in range(0, flat.shape[0], rows_per):
        r1 = min(flat.shape[0], r0 + rows_per)
        x = rng.standard_normal((r1 - r0, flat.shape[1]), dtype=np.float32)
        if std != 1.0 or mean != 0.0:
            x = x * np.float32(std) + np.float32(mean)
        flat[r0:r1] = f32_to_f16_bits(x) if io == "fp16" else f32_to_bf16_bits(x)
    return out


def weights_as(w: np.ndarray, dtype: str) -> np.ndarray:
    """fp32 router weights stored as fp32, or as bf16 / fp16 bit patterns."""
    if dtype == "bf16":
        return f32_to_bf16_bits(w)
    if dtype == "fp16":
        return f32_to_f16_bits(w)
    return w


def make_inputs(wl: Workload, seed: Optional[int] = None) -> dict:
    """All host inputs of one workload as numpy arrays (bf16 as uint16 bits)."""
    rng = np.random.Generator(np.random.PCG64(wl.seed if seed is None else seed))
    ids, w = draw_routing(wl, rng)
    n_valid = int((ids >= 0).sum())
    io = wl.io_dtype
    d = dict(topk_ids=ids, weights=weights_as(w, wl.weight_dtype), n_valid=n_valid)
    d["expert_out"] = bf16_normal(rng, (n_valid, wl.H), io=io)
    d["shared"] = (bf16_normal(rng, (wl.T, wl.H), std=wl.shared_std, io=io)
                   if wl.shared_std is not None else None)
    d["residual"] = bf16_normal(rng, (wl.T, wl.H), io=io) if wl.residual else None
    d["gamma"] = (bf16_normal(rng, (wl.H,), std=wl.gamma_std, mean=wl.gamma_mean, io=io)
                  if wl.gamma_mean is not None else None)
    return d


def make_slot_major_inputs(wl: Workload, seed: Optional[int] = None) -> dict:
    """Inputs for the slot-major layout: every token has one expert row per
    slot, stored as bf16 [k, T, H] (no routing ids, no padding); weights are
    the softmax of N(0, 1) logits per token as in make_inputs."""
    rng = np.random.Generator(np.random.PCG64((wl.seed if seed is None else seed) + 500))
    logits = rng.standard_normal((wl.T, wl.k))
    w = np.exp(logits - logits.max(axis=1, keepdims=True))
    w = (w / w.sum(axis=1, keepdims=True)).astype(np.float32)
    io = wl.io_dtype
    d = dict(weights=weights_as(w, wl.weight_dtype), n_valid=wl.T * wl.k)
    d["expert_out"] = bf16_normal(rng, (wl.k, wl.T, wl.H), io=io)
    d["shared"] = (bf16_normal(rng, (wl.T, wl.H), std=wl.shared_std, io=io)
                   if wl.shared_std is not None else None)
    d["residual"] = bf16_normal(rng, (wl.T, wl.H), io=io) if wl.residual else None
    d["gamma"] = (bf16_normal(rng, (wl.H,), std=wl.gamma_std, mean=wl.gamma_mean, io=io)
                  if wl.gamma_mean is not None else None)
    return d
