"""Source files stand on their own: no code, comment or docstring names the
project's planning documents, the driver's files, the remote-run tool or a
path of the build machine."""
import glob
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
_DOCS = ["SUR" + "VEY", "DES" + "IGN.md", "VER" + "DICT", "ADV" + "ICE", "BASE" + "LINE",
         "north" + "_star", "PA" + "PER.md", "gpu" + "run", "/ro" + "ot/"]


def _sources():
    pats = ["norm_quant_gb300/**/*.py", "norm_quant_gb300/csrc/*", "include/*.h", "oracle/*.py", "oracle/*.c",
            "tests/**/*.py", "tests/cuda/*", "bench.py", "__graft_entry__.py"]
    files = set()
    for p in pats:
        files |= {f for f in glob.glob(os.path.join(ROOT, p), recursive=True) if os.path.isfile(f)}
    files = {f for f in files if "/_build/" not in f and "__pycache__" not in f}
    assert len(files) > 20
    return sorted(files)


def test_sources_name_no_planning_documents_or_machine_paths():
    bad = []
    for f in _sources():
        text = open(f, errors="replace").read()
        for word in _DOCS:
            for m in re.finditer(re.escape(word), text):
                bad.append((os.path.relpath(f, ROOT), text.count("\n", 0, m.start()) + 1, word))
    assert not bad, bad[:10]
