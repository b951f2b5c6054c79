"""The committed ncu summaries stay usable: each is a short text file that
gives the ncu command it came from (with --clock-control none), and each
command line runs committed files only, with flags bench.py still accepts."""
import os
import re
import shlex
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILES = os.path.join(ROOT, "profiles")
sys.path.insert(0, ROOT)
import bench  # noqa: E402

SUMMARIES = sorted(f for f in os.listdir(PROFILES) if f.endswith(".md"))


def _commands(text):
    """The indented command blocks of a summary, continuation lines joined."""
    out, cur = [], ""
    for line in text.splitlines():
        if line.startswith("    ") and line.strip():
            cur += " " + line.strip().rstrip("\\").strip()
            if not line.rstrip().endswith("\\"):
                out.append(cur.strip())
                cur = ""
        elif cur:
            out.append(cur.strip())
            cur = ""
    if cur:
        out.append(cur.strip())
    return out


def test_profiles_hold_only_short_text():
    for f in os.listdir(PROFILES):
        assert f.endswith((".md", ".txt", ".json")), f
        assert os.path.getsize(os.path.join(PROFILES, f)) < 16 * 1024, f


@pytest.mark.parametrize("name", SUMMARIES)
def test_summary_gives_a_runnable_ncu_command(name, monkeypatch):
    text = open(os.path.join(PROFILES, name)).read()
    cmds = [c for c in _commands(text) if c.startswith("ncu ")]
    assert cmds, f"{name}: no ncu command"
    for cmd in cmds:
        assert "--clock-control none" in cmd, cmd
        argv = shlex.split(cmd)
        i = argv.index("python")
        script = argv[i + 1]
        assert os.path.exists(os.path.join(ROOT, script)), script
        assert not re.search(r"(^|/)_work/", script), script
        if script == "bench.py":
            monkeypatch.setattr(sys, "argv", ["bench.py", *argv[i + 2:]])
            bench.parse_args()      # exits (SystemExit) on a flag bench.py no longer takes
