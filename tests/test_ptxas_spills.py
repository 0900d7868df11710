"""Every kernel compiles for sm_103a without register spills.

The combine's plans rest on the kernels fitting their launch bounds in
registers: with 17 warps a CTA (16 consumer warps and the producer) the cap is
96 registers a thread, and a spill would put local-memory traffic on the path
that is meant to move only the algorithmic bytes.  ptxas reports, per kernel,
its registers and spill bytes (-Xptxas -v); this test reads those counts."""
import importlib
import os
import re
import subprocess

B = importlib.import_module("norm_quant_gb300.build")  # the module (the package exports a build function)


def _ptxas_reports():
    procs = []
    for src in B.sources():
        cmd = [B._nvcc(), *B.ARCH, *B.FLAGS, "-Xptxas", "-v", "-I", os.path.join(B.ROOT, "include"),
               "-c", src, "-o", os.devnull]
        procs.append((os.path.basename(src), subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                                              stderr=subprocess.STDOUT, text=True)))
    out = {}
    for name, p in procs:
        text, _ = p.communicate(timeout=600)
        assert p.returncode == 0, text[-3000:]
        out[name] = text
    return out


def test_no_kernel_spills():
    reports = _ptxas_reports()
    kernels = []
    for name, text in reports.items():
        fn = None
        for line in text.splitlines():
            m = re.search(r"Function properties for (\S+)", line)
            if m:
                fn = m.group(1)
                continue
            m = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", line)
            if m and fn is not None:
                assert (int(m.group(1)), int(m.group(2))) == (0, 0), (name, fn, line.strip())
                kernels.append(fn)
                fn = None
    # three combine forms (bf16; fp16; fp16 with fp16 weights), each with
    # VPT 1/2/4/8 x four quantisers plus split rows (VPT 1) x four quantisers
    assert sum("combine_kernel" in k for k in kernels) == 3 * (4 * 4 + 4)
    assert any("route_fused_kernel" in k for k in kernels) and any("dispatch_kernel" in k for k in kernels)
