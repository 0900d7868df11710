"""The bench's host-side arithmetic, on the CPU: the algorithmic byte counts
behind every roofline fraction, checked against per-workload totals worked
out by hand from the byte formula (reads of the k expert rows at 2H bytes,
the shared and residual rows, 8k bytes of row_map and weights per token and
gamma once; writes of each 16-bit output, the fp8 / fp4 codes and the scale
bytes), and the code-only source hash that decides whether a recorded ncu
traffic figure still applies."""
import os

import pytest

import bench


@pytest.mark.parametrize("name,n_valid,total_mb", [
    # prefill: 469.76 MB rows + 117.44 shared/residual + 0.28 metadata + 89.00 writes
    ("prefill", 4096 * 8, 676.48),
    # Gemma NVFP4: 536.87 + 67.11 + 0.53 + 85.98
    ("gemma", 8192 * 8, 690.49),
    # decode: 7.34 + 0.92 + 0.02 + 1.84
    ("decode", 64 * 8, 10.11),
])
def test_algorithmic_bytes_match_the_workload_table(name, n_valid, total_mb):
    wl = bench.workload(name)
    b = bench.algorithmic_bytes(wl, n_valid)
    assert b["total"] == b["rows"] + b["other_reads"] + b["meta"] + b["writes"]
    assert abs(b["total"] / 1e6 - total_mb) < 0.01


def test_byte_count_follows_dtypes_and_formats():
    base = bench.algorithmic_bytes(bench.workload("prefill"), 32768)
    fp16 = bench.algorithmic_bytes(bench.workload("fp16"), 32768)
    mxfp4 = bench.algorithmic_bytes(bench.workload("mxfp4"), 32768)
    T, H, k = 4096, 7168, 8
    assert base["meta"] - fp16["meta"] == 2 * k * T          # 2-byte router weights
    assert base["writes"] - mxfp4["writes"] == H // 2 * T    # 4-bit codes, same scale bytes
    assert base["rows"] == fp16["rows"] == mxfp4["rows"] == 32768 * 2 * H


def test_byte_count_follows_layouts():
    """Slot-major reads no row_map; 128x4 scales count their pad bytes,
    as the library sizes them (checked against the oracle's sizes)."""
    import dataclasses
    import oracle
    P = bench.workload("prefill")
    grouped = bench.algorithmic_bytes(P, 32768)
    slot = bench.algorithmic_bytes(P, 32768, "slot_major")
    assert grouped["meta"] - slot["meta"] == 4 * P.k * P.T
    for q in ("mxfp8", "nvfp4", "mxfp4"):
        for T, H in ((4096, 7168), (300, 96), (130, 224)):
            wl = dataclasses.replace(P, T=T, H=H, quant=q, sf_layout="swizzled", outputs=("quant",))
            codes = (H if q == "mxfp8" else H // 2) * T
            assert bench.algorithmic_bytes(wl, 8 * T)["writes"] == \
                codes + oracle.scales_bytes(T, H, q, "swizzled")
            wl = dataclasses.replace(wl, sf_layout="linear")
            assert bench.algorithmic_bytes(wl, 8 * T)["writes"] == codes + oracle.scales_bytes(T, H, q, "linear")


def test_code_only_ignores_comments_and_whitespace():
    a = "int f(int x) { // add one\n  return x + 1; /* block\n comment */ }\n"
    b = "int f(int x)\n{\n    return x + 1;\n}"
    c = "int f(int x) { return x + 2; }"
    assert bench.code_only(a) == bench.code_only(b)
    assert bench.code_only(a) != bench.code_only(c)


def test_kernel_hash_changes_with_code_not_with_comments():
    src = {f: open(f"{bench.ROOT}/{f}").read() for f in bench.KERNEL_SOURCES}
    h0 = bench.kernel_hash(lambda f: src[f])
    first = bench.KERNEL_SOURCES[0]
    commented = dict(src, **{first: "// a new comment line\n" + src[first]})
    assert bench.kernel_hash(lambda f: commented[f]) == h0
    edited = dict(src, **{first: src[first] + "\nstatic int extra_symbol = 1;\n"})
    assert bench.kernel_hash(lambda f: edited[f]) != h0


def test_recorded_traffic_needs_a_matching_source_hash():
    """A summary's DRAM bytes count only while its hash is the kernel
    sources' hash; workloads without a summary report none."""
    h = bench.kernel_hash()
    summary = {f: f"x\ndram_bytes_per_launch: 123456\nkernel_source_hash: {h}\ncaptured: 2026-12-02\n"
               for f in bench.TRAFFIC_FILES.values()}
    for kind in ("prefill", "fp16", "gemma", "decode"):
        got = bench.recorded_traffic(kind, summary.__getitem__)
        assert got["bytes"] == 123456 and got["kernel_source_hash"] == h and got["captured"] == "2026-12-02"
        assert got["file"] == bench.TRAFFIC_FILES[kind]
        prov = bench.traffic_provenance(kind, got)
        assert prov["file"] == got["file"] and prov["captured"] == "2026-12-02"
    assert bench.recorded_traffic("tiny", summary.__getitem__) is None
    assert "no committed" in bench.traffic_provenance("tiny", None)["how"]
    stale = {f: t.replace(h, "0" * 16) for f, t in summary.items()}
    assert bench.recorded_traffic("prefill", stale.__getitem__) is None
    assert "other kernel source" in bench.traffic_provenance("prefill", None)["how"]
    assert all(os.path.exists(os.path.join(bench.ROOT, f)) for f in bench.TRAFFIC_FILES.values())


def _reference_arm(*extra, env=None):
    import json
    import subprocess
    import sys
    run = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "3", "--warmup", "3",
                          *extra], cwd=bench.ROOT, capture_output=True, text=True, timeout=600,
                         env={**os.environ, **(env or {})})
    lines = [json.loads(x) for x in run.stdout.splitlines() if x.startswith("{")]
    return run.returncode, lines, run.stderr


@pytest.mark.parametrize("name", ["tiny", "decode"])
def test_reference_arm_line(name):
    """The oracle arm on the CPU: one JSON line with the contract's keys, on
    the requested workload, with no host<->device bytes."""
    rc, lines, err = _reference_arm("--workload", name)
    assert rc == 0, err[-2000:]
    assert len(lines) == 1
    line = lines[0]
    wl = bench.workload(name)
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["config"]["workload"] == wl.name and line["config"]["T"] == wl.T
    assert line["value"] > 0 and line["unit"] == "tokens/s" and line["higher_is_better"] is True
    assert line["steps"] == 3 and line["warmup"] == 3 and line["dtype"] == "f64"
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"] and cb["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": "tokens/s",
                           "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_exit_quietly():
    rc, lines, _ = _reference_arm("--workload", "tiny", env={"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert rc == 0 and lines == []


def test_workload_from_the_command_line():
    import sys
    def parsed(*argv):
        old = sys.argv
        try:
            sys.argv = ["bench.py", *argv]
            return bench.args_workload(bench.parse())
        finally:
            sys.argv = old
    assert parsed() == bench.workload("prefill")                       # the headline, unchanged
    assert parsed("--workload", "gemma") == bench.workload("gemma")
    w = parsed("--workload", "padded", "--T", "512")
    assert (w.T, w.seed) == (512, 2512)
    w = parsed("--workload", "decode", "--seed", "7")
    assert w.seed == 7 and w.name.endswith("_seed7") and w.T == bench.workload("decode").T
    with pytest.raises(SystemExit):
        parsed("--T", "64")                                           # --T goes with padded only
