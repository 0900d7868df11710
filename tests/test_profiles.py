"""The committed ncu summaries: short text, each with the full command that
made it, every ncu invocation leaving the GPU clocks alone
(--clock-control none), and every command running committed files only."""
import glob
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _summaries():
    files = sorted(glob.glob(os.path.join(ROOT, "profiles", "*")))
    assert files
    return files


def test_summaries_are_short_text():
    for f in _summaries():
        assert f.endswith((".md", ".txt")), f
        assert os.path.getsize(f) < 16 * 1024, f


def test_every_ncu_command_keeps_the_clocks_and_runs_committed_files():
    for f in _summaries():
        text = open(f).read()
        # an ncu command may continue over lines ending in a backslash
        commands = re.findall(r"ncu (?:[^\n]*\\\n)*[^\n]*", text)
        assert commands, f"{f}: no ncu command"
        for c in commands:
            assert "--clock-control none" in c, (f, c)
            assert "_work" not in c, (f, c)
            for script in re.findall(r"python ([\w/]+\.py)", c):
                assert os.path.exists(os.path.join(ROOT, script)), (f, script)
