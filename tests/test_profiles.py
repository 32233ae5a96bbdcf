"""The ncu summaries under profiles/ stay reproducible from committed files: each gives the command
that made it, every ncu command leaves the GPU clocks alone (--clock-control none), every
workload it runs is one bench.py still offers as an ncu target, and the committed per-launch
traffic figure is keyed to the decode kernel's current sources (bench.py reports it only then)."""
import glob
import json
import os
import re

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SUMMARIES = sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md")))


def _commands(text: str):
    """ncu command lines of a summary (continuation lines joined)."""
    joined = re.sub(r"\\\s*\n\s*", " ", text)
    return [line for line in joined.splitlines() if re.search(r"\bncu\b\s+--", line)]


def test_summaries_exist():
    assert SUMMARIES, "no ncu summary under profiles/"


def test_every_summary_gives_its_ncu_command():
    for p in SUMMARIES:
        cmds = _commands(open(p).read())
        assert cmds, f"{os.path.basename(p)} gives no ncu command"
        for c in cmds:
            assert "--clock-control none" in c, f"{os.path.basename(p)}: ncu without --clock-control none: {c}"


def test_ncu_targets_exist_in_bench():
    targets = set(bench.NCU_TARGETS)
    for p in SUMMARIES + [os.path.join(ROOT, "profiles", "traffic.json")]:
        for t in re.findall(r"--ncu-target ([A-Za-z0-9_-]+)", open(p).read()):
            assert t in targets, f"{os.path.basename(p)} runs ncu target {t!r}, which bench.py no longer has"


def test_traffic_figure_keyed_to_current_decode_sources():
    d = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    entries = {k: v for k, v in d.items() if isinstance(v, dict) and "source_hash" in v}
    assert entries
    for k, e in entries.items():
        assert e["dram_bytes_per_launch"] > 0
        assert "--clock-control none" in e.get("command", d.get("command", ""))
    # bench.py returns the figure only while the hash matches; the committed one should
    assert any(e["source_hash"] == bench.kernel_source_hash() for e in entries.values()), \
        "profiles/traffic.json was taken on other decode-kernel sources: re-capture it"
