"""Benchmark of the MoE combine/finalize step on GB300.

One step = one pass of the whole hot path over one batch: the routing build
(moe_build_row_map: histogram, scan, stable scatter) and the combine
(moe_combine: gather + weighted sum + shared + residual + RMSNorm + MXFP8),
on the prefill workload T=4096, H=7168, E=256, top_k=8 (Zipf 1.1 experts,
shared expert row, residual, RMSNorm, MXFP8 with linear UE8M0 scales).

Timing: inputs resident in HBM.  Each step streams 676 MB (587 MB read, 89 MB
written), over five times the 129 MB L2, so no step finds the previous
step's data in L2; `--l2 write` instead writes a 256 MB buffer before each
step, outside the timed events (its dirty lines are then written back during
the next step, which the default avoids).  Each step is bracketed by CUDA
events on the launching stream; `value` = tokens / summed step time.  The
combine kernel is also bracketed on its own for the roofline line.  `e2e`
repeats the step through the same C ABI from pinned host buffers, with the
host->device copy of the step's inputs and the device->host copy of its
outputs inside the timed region.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun each rank runs an independent replica on its own GPU (the
tokens of a batch are independent; there is no data-path collective), and
rank 0 prints one JSON line with the max-over-ranks time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import time
import types

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE combine tokens/s and achieved HBM GB/s vs peak (T=4096,H=7168,k=8)"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0   # GB300's HBM3e, NVIDIA's nominal figure (8 stacks)
L2_FLUSH_BYTES = 256 << 20
# every source the combine kernels are compiled from
KERNEL_SOURCES = ["norm_quant_gb300/csrc/combine.cu", "norm_quant_gb300/csrc/combine_impl.cuh",
                  "norm_quant_gb300/csrc/ptx.cuh", "norm_quant_gb300/csrc/combine_f16.cu",
                  "norm_quant_gb300/csrc/combine_f16w.cu", "norm_quant_gb300/csrc/common.h"]
# the committed ncu summary of each workload whose combine traffic was captured
TRAFFIC_FILES = {"prefill": "profiles/combine_prefill_T4096_H7168_k8_mxfp8.md",
                 "fp16": "profiles/combine_prefill_fp16io_fp16weights_T4096_H7168_k8_mxfp8.md",
                 "gemma": "profiles/combine_gemma_T8192_H4096_nvfp4_128x4.md",
                 "decode": "profiles/combine_decode_T64_H7168_k8.md"}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--workload", choices=["tiny", "decode", "prefill", "gemma", "padded",
                                           "slot_major", "dispatch", "mxfp4", "fp16", "fp16_fp32w"],
                    default="prefill", help="the headline is prefill; the others are for analysis "
                    "(slot_major: the prefill shape with [k, T, H] expert rows; dispatch: the "
                    "prefill shape's dispatch-side permute; mxfp4: the prefill shape with MXFP4 "
                    "output; fp16: the prefill shape with fp16 inputs, outputs and router weights; fp16_fp32w: "
                    "the same with fp32 router weights)")
    ap.add_argument("--T", type=int, default=None,
                    help="with --workload padded: a point of its token-count sweep (seed 2000 + T)")
    ap.add_argument("--seed", type=int, default=None,
                    help="another seed for the workload's synthetic inputs (default: the workload's own)")
    ap.add_argument("--l2", choices=["none", "write", "read"], default="none",
                    help="none: inputs larger than L2; write: 256 MB write before each step (leaves L2 "
                    "full of dirty lines); read: 256 MB read before each step (leaves it full of clean lines)")
    return ap.parse_args()


def max_over_ranks(x: float, device=None) -> float:
    """The largest of every rank's x (x itself when not distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, tokens_per_rank: int, steps: int, max_seconds: float) -> float:
    """Whole-job tokens/s: every rank's tokens over the slowest rank's time."""
    return world * tokens_per_rank * steps / max_seconds


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def args_workload(args):
    """The workload the command line names: --workload, or a point of the
    padded workload's token-count sweep with --T."""
    import dataclasses
    from norm_quant_gb300 import synth
    if args.T is None:
        wl = workload(args.workload)
    elif args.workload != "padded" or args.T < 1:
        raise SystemExit("bench.py: --T takes a positive token count and goes with --workload padded")
    else:
        wl = synth.sweep_point(args.T)
    if args.seed is not None:
        wl = dataclasses.replace(wl, seed=args.seed, name=f"{wl.name}_seed{args.seed}")
    return wl


def workload(name="prefill"):
    import dataclasses
    from norm_quant_gb300 import synth
    P = synth.PREFILL
    return {"tiny": synth.TINY, "decode": synth.DECODE, "prefill": P,
            "gemma": synth.GEMMA_NVFP4, "padded": synth.PADDED, "slot_major": P, "dispatch": P,
            "mxfp4": dataclasses.replace(P, quant="mxfp4", name=P.name.replace("mxfp8", "mxfp4")),
            "fp16": dataclasses.replace(P, io_dtype="fp16", weight_dtype="fp16",
                                        name=P.name.replace("rmsnorm", "fp16io_fp16weights_rmsnorm")),
            "fp16_fp32w": dataclasses.replace(P, io_dtype="fp16",
                                              name=P.name.replace("rmsnorm", "fp16io_rmsnorm"))}[name]


def algorithmic_bytes(wl, n_valid: int, expert_layout: str = "grouped") -> dict:
    """Bytes one combine launch must move at least (reads + writes).  The
    slot-major layout reads no row_map; 128x4 scales include their pad bytes
    (rows to a multiple of 128, scale columns to a multiple of 4)."""
    T, H, k = wl.T, wl.H, wl.k
    rows = n_valid * 2 * H
    other = (2 * H * T if wl.shared_std is not None else 0) + (2 * H * T if wl.residual else 0)
    weight_bytes = 4 if wl.weight_dtype == "fp32" else 2
    map_bytes = 0 if expert_layout == "slot_major" else 4
    meta = (map_bytes + weight_bytes) * k * T + (2 * H if wl.gamma_mean is not None else 0)
    writes = 2 * H * T * len([o for o in wl.outputs if o in ("combined", "residual", "norm")])
    if wl.quant:
        writes += (H if wl.quant == "mxfp8" else H // 2) * T           # codes
        cols = H // (16 if wl.quant == "nvfp4" else 32)
        if wl.sf_layout == "swizzled":
            writes += -(-T // 128) * 128 * (-(-cols // 4) * 4)
        else:
            writes += cols * T
    return {"rows": rows, "other_reads": other, "meta": meta, "writes": writes,
            "total": rows + other + meta + writes}


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        return float(json.load(open(p))["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def code_only(text: str) -> str:
    """C++ source without its comments and whitespace: edits to comments alone
    leave the compiled kernel, and so this text, unchanged."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return re.sub(r"\s+", "", text)


def kernel_hash(read=None) -> str:
    """Hash of the combine kernel's code (comments and whitespace ignored)."""
    read = read or (lambda f: open(os.path.join(ROOT, f)).read())
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        h.update(code_only(read(f)).encode())
    return h.hexdigest()[:16]


def recorded_traffic(kind="prefill", read=None):
    """DRAM bytes per combine launch from the workload's committed ncu
    summary, with the summary's capture date and kernel source hash; None if
    there is no summary or the kernel source changed since those counters
    were taken."""
    read = read or (lambda f: open(os.path.join(ROOT, f)).read())
    if kind not in TRAFFIC_FILES:
        return None
    try:
        text = read(TRAFFIC_FILES[kind])
    except OSError:
        return None
    m = re.search(r"dram_bytes_per_launch:\s*([0-9]+)", text)
    hsh = re.search(r"kernel_source_hash:\s*([0-9a-f]+)", text)
    when = re.search(r"captured:\s*([0-9-]+)", text)
    if not m or not hsh or hsh.group(1) != kernel_hash():
        return None
    return {"bytes": int(m.group(1)), "file": TRAFFIC_FILES[kind], "kernel_source_hash": hsh.group(1),
            "captured": when.group(1) if when else None}


def traffic_provenance(kind, traffic):
    """Where roofline.traffic comes from (or why it is null)."""
    if traffic:
        return {"how": "dram__bytes_read.sum + dram__bytes_write.sum of one launch, from the committed ncu "
                       "summary of this kernel source (not measured in this run)",
                "file": traffic["file"], "kernel_source_hash": traffic["kernel_source_hash"],
                "captured": traffic["captured"]}
    if kind not in TRAFFIC_FILES:
        return {"how": "null: no committed ncu summary for this workload"}
    return {"how": "null: the committed ncu summary was taken on other kernel source (hash "
                   f"{kernel_hash()} now), or the run flushes L2 between steps"}


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.p = None

    def __enter__(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "100"],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.p = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.p is not None:
            time.sleep(0.2)
            self.p.terminate()
            out, _ = self.p.communicate(timeout=10)
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        mhz, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                mhz.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": float(np.median(mhz)) if mhz else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(mhz)}


def cpu_oracle_rate(wl, inp, orm, seconds: float):
    """Tokens/s of the oracle on a bounded sample of this workload's tokens."""
    import oracle
    n = 16
    while True:
        t0 = time.perf_counter()
        oracle.combine(inp["expert_out"], orm[:n], inp["weights"][:n], shared=inp["shared"][:n],
                       residual=inp["residual"][:n], gamma=inp["gamma"], eps=wl.eps,
                       weight_bias=wl.weight_bias, quant=wl.quant, sf_layout="linear",
                       outputs=("residual", "quant"))
        dt = time.perf_counter() - t0
        if dt >= seconds or n >= wl.T:
            return n / dt, n, dt
        n = min(wl.T, max(n * 2, int(n * seconds / max(dt, 1e-3) * 1.1)))


# ---- the oracle on all host cores: token slices in spawned worker processes

_POOL_ARRAYS = {}


def _pool_init(specs, params):
    """Worker start: attach the shared input arrays; import the oracle."""
    from multiprocessing import shared_memory
    import oracle  # noqa: F401  (built by the parent)
    for name, (shm_name, shape, dtype) in specs.items():
        shm = shared_memory.SharedMemory(name=shm_name)
        _POOL_ARRAYS[name] = (shm, np.ndarray(shape, dtype=dtype, buffer=shm.buf))
    _POOL_ARRAYS["_params"] = params


def _pool_slice(bounds):
    """The oracle's routing build and combine of tokens [a, b), as it stands."""
    import oracle
    a, b = bounds
    A = {n: v[1] for n, v in _POOL_ARRAYS.items() if n != "_params"}
    P = _POOL_ARRAYS["_params"]
    oracle.build_row_map(A["topk_ids"][a:b], P["E"])
    oracle.combine(A["expert_out"], A["row_map"][a:b], A["weights"][a:b],
                   shared=A["shared"][a:b] if "shared" in A else None,
                   residual=A["residual"][a:b] if "residual" in A else None, gamma=A.get("gamma"),
                   eps=P["eps"], weight_bias=P["weight_bias"], quant=P["quant"],
                   sf_layout=P["sf_layout"], outputs=P["outputs"], io_dtype=P["io_dtype"],
                   weight_dtype=P["weight_dtype"])
    return b - a


class OraclePool:
    """A spawn-started process pool (one worker per host core) over shared
    copies of the workload's inputs; `run(a, b)` splits tokens [a, b) evenly
    over the workers and returns the wall-clock seconds it took."""

    def __init__(self, wl, inp, orm, workers=None):
        import multiprocessing as mp
        from multiprocessing import shared_memory
        self.workers = workers or len(os.sched_getaffinity(0))
        arrays = {"topk_ids": inp["topk_ids"], "row_map": orm, "weights": inp["weights"],
                  "expert_out": inp["expert_out"], "shared": inp.get("shared"),
                  "residual": inp.get("residual"), "gamma": inp.get("gamma")}
        self.shms, specs = [], {}
        for name, arr in arrays.items():
            if arr is None:
                continue
            arr = np.ascontiguousarray(arr)
            shm = shared_memory.SharedMemory(create=True, size=max(1, arr.nbytes))
            np.ndarray(arr.shape, dtype=arr.dtype, buffer=shm.buf)[...] = arr
            self.shms.append(shm)
            specs[name] = (shm.name, arr.shape, arr.dtype.str)
        params = {"E": wl.E, "eps": wl.eps, "weight_bias": wl.weight_bias, "quant": wl.quant,
                  "sf_layout": wl.sf_layout, "outputs": tuple(wl.outputs), "io_dtype": wl.io_dtype,
                  "weight_dtype": wl.weight_dtype}
        self.pool = mp.get_context("spawn").Pool(self.workers, initializer=_pool_init, initargs=(specs, params))
        self.pool.map(_pool_slice, [(0, 1)] * self.workers)  # every worker started and warm

    def run(self, a, b):
        n = b - a
        cuts = [a + (n * i) // self.workers for i in range(self.workers + 1)]
        t0 = time.perf_counter()
        self.pool.map(_pool_slice, [(cuts[i], cuts[i + 1]) for i in range(self.workers) if cuts[i + 1] > cuts[i]])
        return time.perf_counter() - t0

    def close(self):
        self.pool.close()
        self.pool.join()
        for shm in self.shms:
            shm.close()
            shm.unlink()


def cpu_oracle_rate_all_cores(wl, inp, orm, seconds: float):
    """Tokens/s of the oracle over all host cores: whole passes over the
    workload's tokens (routing build + combine) until `seconds` have passed."""
    pool = OraclePool(wl, inp, orm)
    try:
        done, total = 0, 0.0
        while total < seconds:
            total += pool.run(0, wl.T)
            done += wl.T
        return done / total, done, total, pool.workers
    finally:
        pool.close()


def run_reference(args):
    """The reference arm: the CPU oracle timed as it stands, on all host cores
    (token slices in spawned processes), on the same workload as our arm
    (the headline unless --workload names another routing + combine one)."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    if args.workload in ("slot_major", "dispatch"):
        raise SystemExit(f"bench.py --impl reference times the routing build + combine workloads; "
                         f"--workload {args.workload} has no reference arm")
    import oracle
    from norm_quant_gb300 import synth
    wl = args_workload(args)
    inp = synth.make_inputs(wl)
    st, _, _, orm, _ = oracle.build_row_map(inp["topk_ids"], wl.E)
    pool = OraclePool(wl, inp, orm)
    try:
        probe = min(wl.T, 64 * pool.workers)
        rate = probe / pool.run(0, probe)
        budget = 90.0
        per_step = max(1, min(wl.T, int(rate * budget / max(1, args.steps + args.warmup))))

        def step(i):
            t0 = (i * per_step) % max(1, wl.T - per_step + 1)
            return pool.run(t0, t0 + per_step)

        for i in range(args.warmup):
            step(i)
        t0 = time.perf_counter()
        for i in range(args.steps):
            step(i)
        dt = time.perf_counter() - t0
        cores = pool.workers
    finally:
        pool.close()
    value = per_step * args.steps / dt
    sample = (f"{per_step} of {wl.T} tokens per step (routing build + combine of that slice), "
              f"split over {cores} spawned processes")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "T": wl.T, "H": wl.H, "E": wl.E, "top_k": wl.k,
                   "sample": sample},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def run_ours(args):
    import torch
    import torch.distributed as dist

    import norm_quant_gb300 as nqg
    from norm_quant_gb300 import synth
    from norm_quant_gb300.build import build

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        build()
    if world > 1:
        dist.barrier()
    build()
    nqg.lib()

    kind = args.workload
    wl = args_workload(args)
    T, H, E, k = wl.T, wl.H, wl.E, wl.k
    inp = synth.make_slot_major_inputs(wl) if kind == "slot_major" else synth.make_inputs(wl)
    if kind == "dispatch":  # the residual stream is the token input of the permute
        inp = {"topk_ids": inp["topk_ids"], "x": inp["residual"], "n_valid": inp["n_valid"]}

    def pinned(a):
        a = a.view(np.int16) if a.dtype == np.uint16 else a
        return torch.from_numpy(np.ascontiguousarray(a)).pin_memory()

    names = [n for n in ("topk_ids", "weights", "expert_out", "shared", "residual", "gamma", "x")
             if inp.get(n) is not None]
    host = {n: pinned(inp[n]) for n in names}
    flush = torch.zeros(L2_FLUSH_BYTES if args.l2 != "none" else 16, dtype=torch.uint8, device=dev)
    flush_sum = torch.zeros((), dtype=torch.int64, device=dev)

    def flush_l2():
        """Evicts the step's data from L2: by writing 256 MB (the lines it
        leaves are dirty and are written back during the next step) or by
        reading it (the lines it leaves are clean)."""
        if args.l2 == "write":
            flush.zero_()
        elif args.l2 == "read":
            flush_sum.copy_(flush.view(torch.int64).max())
    stream = torch.cuda.current_stream(dev)
    route_kernels = 0 if kind == "slot_major" else nqg.moe_build_row_map_launches(T, k, E)

    def buffer_set():
        """Device inputs, outputs and the calls of one step over them."""
        b = types.SimpleNamespace()
        b.dv = {n: t.to(dev) for n, t in host.items()}
        b.counts = torch.empty(E, dtype=torch.int32, device=dev)
        b.offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
        b.row_map = torch.empty((T, k), dtype=torch.int32, device=dev)
        b.ws = torch.empty(nqg.moe_build_row_map_workspace_size(T, k, E), dtype=torch.uint8, device=dev)
        b.outs = {}
        if kind == "dispatch":
            b.outs["x_grouped"] = torch.empty((inp["n_valid"], H), dtype=torch.int16, device=dev)
        for o in ("combined", "residual", "norm"):
            if kind != "dispatch" and o in wl.outputs:
                b.outs[o] = torch.empty((T, H), dtype=torch.int16, device=dev)
        if kind != "dispatch" and wl.quant:
            b.outs["quant"] = torch.empty((T, H if wl.quant == "mxfp8" else H // 2), dtype=torch.uint8,
                                          device=dev)
            b.outs["scales"] = torch.empty(nqg.moe_scales_bytes(T, H, wl.quant, wl.sf_layout),
                                           dtype=torch.uint8, device=dev)
        b.args_c = None
        if kind != "dispatch":
            # NVFP4's per-tensor scale only changes which codes come out, not the work
            b.args_c = nqg.combine_args(
                expert_out=b.dv["expert_out"].reshape(-1, H), row_map=None if kind == "slot_major" else b.row_map,
                router_weights=b.dv["weights"], shared_out=b.dv.get("shared"), residual=b.dv.get("residual"),
                gamma=b.dv.get("gamma"), eps=wl.eps, weight_bias=wl.weight_bias, quant=wl.quant,
                sf_layout=wl.sf_layout, global_scale=1.0, combined_out=b.outs.get("combined"),
                residual_out=b.outs.get("residual"), norm_out=b.outs.get("norm"), quant_out=b.outs.get("quant"),
                scales_out=b.outs.get("scales"), H=H,
                expert_layout="slot_major" if kind == "slot_major" else "grouped",
                io_dtype=wl.io_dtype, weight_dtype=wl.weight_dtype)

        def route(st):
            if kind != "slot_major":
                nqg.moe_build_row_map(b.dv["topk_ids"], E, b.counts, b.offsets, b.row_map, None, b.ws, stream=st)

        def combine(st):  # the dominant kernel of the step
            if kind == "dispatch":
                nqg.moe_dispatch_permute(b.dv["x"], b.row_map, b.outs["x_grouped"], stream=st)
            else:
                nqg.moe_combine(stream=st, args=b.args_c)

        def step(st):
            route(st)
            combine(st)

        b.route, b.combine, b.step = route, combine, step
        return b

    bufs = [buffer_set()]
    route, combine, step, ws = bufs[0].route, bufs[0].combine, bufs[0].step, bufs[0].ws

    gs = torch.cuda.Stream(dev)
    with torch.cuda.stream(gs):
        for _ in range(3):  # first calls configure the kernels; outside capture
            flush_l2()
            step(gs.cuda_stream)
    torch.cuda.synchronize()
    if kind != "slot_major":
        assert nqg.moe_build_row_map_check(ws, stream=gs.cuda_stream) == nqg.MOE_OK

    # G consecutive steps per graph (G divides K), so that the graph's own
    # launch cost is paid once per G steps, as in a serving loop; with an L2
    # flush before every step, one step per graph keeps the flush outside the
    # timed events
    K = args.steps
    G = 1 if args.l2 != "none" else next(g for g in (10, 8, 5, 4, 2, 1) if K % g == 0)

    def graph_of(fn, n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=gs):
            for _ in range(n):
                fn(gs.cuda_stream)
        return g

    g_step, g_comb = graph_of(step, G), graph_of(combine, G)
    g_route = graph_of(route, G) if kind != "slot_major" else None

    replay_s = []  # device seconds of each replay of the last replay() call

    def replay(g, n):
        """n replays on gs, each after an optional L2 flush; device seconds.
        An event after every replay (no synchronisation between them) also
        gives each replay's duration."""
        replay_s.clear()
        with torch.cuda.stream(gs):
            if args.l2 != "none":
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                for _ in range(n):
                    flush_l2()
                    e0.record(gs)
                    g.replay()
                    e1.record(gs)
                    e1.synchronize()
                    replay_s.append(e0.elapsed_time(e1) / 1e3)
                return sum(replay_s)
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
            ev[0].record(gs)
            for i in range(n):
                g.replay()
                ev[i + 1].record(gs)
        ev[-1].synchronize()
        replay_s.extend(ev[i].elapsed_time(ev[i + 1]) / 1e3 for i in range(n))
        return ev[0].elapsed_time(ev[-1]) / 1e3

    replay(g_step, -(-max(3, args.warmup) // G))  # at least W untimed steps
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        total_s = replay(g_step, K // G)       # timed region: exactly K whole steps
        step_pct = np.percentile(np.array(replay_s) / G * 1e6, [10, 50, 90])
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        comb_s = replay(g_comb, K // G) / K    # the combine kernel alone, same count
        route_s = replay(g_route, K // G) / K if g_route is not None else None  # the routing build alone
    total_s = max_over_ranks(total_s, dev)

    # end to end through the C ABI from pinned host buffers: every step copies
    # its inputs in and its outputs out.  Two buffer sets and three streams
    # (copy-in, compute, copy-out) overlap step i + 1's copy-in with step i's
    # compute and copy-out, as a serving loop would; the timed region runs
    # from the first copy-in to the last copy-out.
    bufs.append(buffer_set())
    host_out = [{n: torch.empty_like(t, device="cpu").pin_memory() for n, t in b.outs.items()} for b in bufs]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out[0].values())
    s_in, s_comp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ev = lambda: torch.cuda.Event()  # noqa: E731
    freed = [ev(), ev()]      # a set's inputs were consumed by its last compute
    drained = [ev(), ev()]    # a set's outputs were copied out

    def e2e_steps(n):
        for i in range(n):
            b, j = bufs[i % 2], i % 2
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(freed[j])
                for name, t in host.items():
                    b.dv[name].copy_(t, non_blocking=True)
                loaded = ev()
                loaded.record(s_in)
            with torch.cuda.stream(s_comp):
                s_comp.wait_event(loaded)
                if i >= 2:
                    s_comp.wait_event(drained[j])
                b.step(s_comp.cuda_stream)
                freed[j].record(s_comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(freed[j])
                for name, t in b.outs.items():
                    host_out[j][name].copy_(t, non_blocking=True)
                drained[j].record(s_out)

    e2e_steps(2)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(s_in)
    e2e_steps(args.e2e_steps)
    s_in.wait_stream(s_out)
    t1.record(s_in)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(t0.elapsed_time(t1) / 1e3, dev)

    if rank == 0:
        if kind == "dispatch":
            nv = inp["n_valid"]
            byt = {"total": T * 2 * H + nv * 2 * H + 4 * k * T}
        else:
            byt = algorithmic_bytes(wl, inp["n_valid"], "slot_major" if kind == "slot_major" else "grouped")
        comb_avg_s = comb_s
        achieved = byt["total"] / comb_avg_s / 1e9
        traffic = recorded_traffic(kind) if args.l2 == "none" else None
        peak, peak_kind = measured_peak()
        line = {
            "metric": METRIC, "value": job_throughput(world, T, K, total_s), "unit": "tokens/s", "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": total_s / K * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": wl.name, "T": T, "H": H, "E": E, "top_k": k,
                       "io": ("bf16 token rows copied to expert-grouped rows" if kind == "dispatch" else
                              f"{wl.io_dtype} in ({wl.weight_dtype} router weights), fp32 accumulate, "
                              f"out: {'+'.join(wl.outputs)}"
                              + (f" ({wl.quant}, {wl.sf_layout} scales)" if wl.quant else "")
                              + (", slot-major [k, T, H] expert rows" if kind == "slot_major" else "")),
                       "l2": ({"write": "256 MB L2 write-flush before each step, outside the timed events",
                               "read": "256 MB L2 read-flush before each step, outside the timed events"}
                              .get(args.l2) or
                              f"no flush: each step streams {byt['total'] / 1e6:.0f} MB through the 129 MB L2"),
                       "timing": f"K steps (routing build + combine) as K/{G} replays of a CUDA graph of "
                                 f"{G} consecutive steps, between two events; the roofline times the same "
                                 f"count of combine launches in graphs of {G}, and route_us the routing "
                                 f"build alone the same way",
                       "parallelism": f"{world} independent replicas" if world > 1 else "1 GPU"},
            "achieved_gbs": achieved,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_source": peak_kind,
                         "nominal_peak": NOMINAL_HBM_GBS, "frac_of_nominal": achieved / NOMINAL_HBM_GBS,
                         "kernel": "dispatch_kernel" if kind == "dispatch" else "combine_kernel",
                         "kernel_ms": comb_avg_s * 1e3,
                         "algorithmic_bytes": byt["total"],
                         "traffic": traffic["bytes"] if traffic else None,
                         "traffic_source": traffic_provenance(kind, traffic)},
            "e2e": {"value": job_throughput(world, T, args.e2e_steps, e2e_s), "unit": "tokens/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": (route_kernels + 1) * K,
            "route_us": route_s * 1e6 if route_s is not None else None,
            "step_time_us": {"p10": float(step_pct[0]), "p50": float(step_pct[1]), "p90": float(step_pct[2]),
                             "over": f"{K // G} replays of {G} steps each (rank {rank})"},
            "clocks": clk.summary(),
        }
        if not args.no_cpu_baseline and world == 1 and kind == "prefill":
            import oracle
            st, _, _, orm, _ = oracle.build_row_map(inp["topk_ids"], E)
            rate1, n1, dt1 = cpu_oracle_rate(wl, inp, orm, args.cpu_seconds)
            rate, n, dt, cores = cpu_oracle_rate_all_cores(wl, inp, orm, args.cpu_seconds)
            line["cpu_baseline"] = {
                "value": rate, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                "sample": f"{n // T} pass(es) over all {T} tokens, routing build + combine + MXFP8, "
                          f"token slices over {cores} spawned processes ({dt:.1f} s wall)",
                "single_thread": {"value": rate1, "unit": "tokens/s", "cores": 1,
                                  "sample": f"first {n1} of {T} tokens, combine + MXFP8 ({dt1:.1f} s)"}}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
