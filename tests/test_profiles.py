"""The ncu summaries under profiles/: each names the command that produced it
(committed files only) and the kernel sources it describes, and bench.py
takes a recorded DRAM traffic figure only while those sources are unchanged."""

import glob
import os
import re
import shutil

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILES = sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md")))


def _fields(text):
    f = re.search(r"src_files:\s*(.+)", text)
    h = re.search(r"src_sha:\s*([0-9a-f]+)", text)
    return (f.group(1).split() if f else None), (h.group(1) if h else None)


def test_there_are_profiles():
    assert PROFILES


@pytest.mark.parametrize("path", PROFILES, ids=os.path.basename)
def test_profile_names_its_command_and_sources(path):
    text = open(path, encoding="utf-8").read()
    assert "ncu " in text and "--clock-control none" in text, "the ncu command that made it"
    assert "_work" not in text, "commands run committed files only"
    files, sha = _fields(text)
    assert files and sha, "src_files / src_sha lines"
    for name in files:
        assert os.path.isfile(os.path.join(ROOT, "paged_kv_cache_98_gb300", "csrc", name)), name


@pytest.mark.parametrize("workload", sorted(bench.TRAFFIC_PROFILES))
def test_traffic_profiles_exist(workload):
    assert os.path.isfile(os.path.join(ROOT, "profiles",
                                       bench.TRAFFIC_PROFILES[workload] + ".md"))


def test_recorded_traffic_follows_the_sources(tmp_path, monkeypatch):
    # a copy of the tree's profile and csrc layout in a scratch root: the
    # figure is returned while the hash matches and dropped once a source changes
    src = os.path.join(ROOT, "profiles", "decode_llama2_7b.md")
    text = open(src, encoding="utf-8").read()
    files, _ = _fields(text)
    root = tmp_path / "root"
    (root / "profiles").mkdir(parents=True)
    csrc = root / "paged_kv_cache_98_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for name in files:
        shutil.copy(os.path.join(ROOT, "paged_kv_cache_98_gb300", "csrc", name), csrc / name)
    monkeypatch.setattr(bench, "ROOT", str(root))
    fresh = re.sub(r"src_sha:\s*[0-9a-f]+", "src_sha: " + bench.source_hash(files), text)
    (root / "profiles" / "p.md").write_text(fresh, encoding="utf-8")
    t = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    assert t, "the headline profile records its traffic"
    assert bench.recorded_traffic("p") == pytest.approx(float(t.group(1)))
    with open(csrc / files[0], "a", encoding="utf-8") as f:
        f.write("\n// changed\n")
    assert bench.recorded_traffic("p") is None
    assert bench.recorded_traffic("absent") is None
