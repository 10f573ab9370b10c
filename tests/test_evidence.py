"""CPU checks of the committed profiling evidence under profiles/.

The roofline line's `traffic` figure is read from profiles/traffic.json and is dropped
(null) when the kernel source has changed since the capture; these tests make such a
change visible before a run, and check that every summary's command can be re-run from
committed files with clocks left alone.
"""
import json
import os
import re
import shlex
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILES = os.path.join(ROOT, "profiles")
CSRC = os.path.join(ROOT, "scaled_dot_product_flash_gb300", "csrc")


def _summaries():
    return sorted(f for f in os.listdir(PROFILES) if f.endswith(".md"))


def _commands(text):
    """Lines inside fenced blocks that start a program."""
    out = []
    for block in re.findall(r"```\n(.*?)```", text, flags=re.S):
        for line in block.splitlines():
            line = line.strip()
            if line.startswith(("ncu ", "python ")):
                out.append(line)
    return out


def test_every_summary_gives_its_command():
    names = _summaries()
    assert names, "no ncu summaries committed"
    for name in names:
        with open(os.path.join(PROFILES, name)) as f:
            assert _commands(f.read()), f"{name} gives no command"


def test_summary_commands_run_committed_files_and_leave_clocks_alone():
    for name in _summaries():
        with open(os.path.join(PROFILES, name)) as f:
            cmds = _commands(f.read())
        for cmd in cmds:
            argv = shlex.split(cmd)
            assert "_work" not in cmd, f"{name}: {cmd}"
            if argv[0] == "ncu":
                assert "--clock-control" in argv and argv[argv.index("--clock-control") + 1] == "none", \
                    f"{name}: ncu without --clock-control none"
            scripts = [a for a in argv if a.endswith(".py")]
            for s in scripts:
                assert os.path.exists(os.path.join(ROOT, s)), f"{name}: {s} is not a committed file"


def test_traffic_record_matches_the_current_sources():
    """A kernel source edited after its DRAM capture must be recaptured (or its entry
    removed); otherwise the bench would silently report traffic as null."""
    sys.path.insert(0, ROOT)
    import bench

    with open(os.path.join(PROFILES, "traffic.json")) as f:
        rec = json.load(f)
    assert rec
    for key, d in rec.items():
        assert os.path.exists(os.path.join(CSRC, d["source"])), key
        assert bench.source_digest(d["source"]) == d["source_sha"], \
            f"{key}: {d['source']} changed since its capture"
        assert d["bytes_per_launch"] > 0
        assert bench.ncu_traffic(key) == d["bytes_per_launch"]
