"""The benchmark's bookkeeping that needs no GPU: the DRAM traffic it reads
from the committed ncu summaries is used only while every kernel source the
capture ran is unchanged, and the summaries it relies on parse."""
import os
import shutil

import bench

REPO = bench.ROOT  # the repository itself (tests below point bench.ROOT elsewhere)


def _tree(tmp_path, text, which):
    """A copy of the repository's sources and one summary under tmp_path."""
    name, srcs = bench.PROFILES[which]
    csrc = tmp_path / "long_context_decode_04_b300" / "csrc"
    csrc.mkdir(parents=True)
    for s in srcs:
        shutil.copy(os.path.join(REPO, "long_context_decode_04_b300", "csrc", s), csrc / s)
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / name).write_text(text)
    return csrc, srcs


def _summary(csrc, srcs, dram):
    lines = ["# kernel", "", "Sources at capture:", ""]
    lines += [f"- {s} sha256: `{bench.source_hash(str(csrc / s))}`" for s in srcs]
    lines += [f"- dram bytes per launch: `{dram}`", ""]
    return "\n".join(lines)


def test_traffic_is_read_while_the_sources_match(tmp_path, monkeypatch):
    for which in bench.PROFILES:
        root = tmp_path / which
        csrc, srcs = _tree(root, "", which)
        (root / "profiles" / bench.PROFILES[which][0]).write_text(_summary(csrc, srcs, 123456))
        monkeypatch.setattr(bench, "ROOT", str(root))
        assert bench.profiled_traffic(which) == 123456


def test_traffic_is_dropped_when_a_source_changed(tmp_path, monkeypatch):
    which = "decode"
    csrc, srcs = _tree(tmp_path, "", which)
    (tmp_path / "profiles" / bench.PROFILES[which][0]).write_text(_summary(csrc, srcs, 99))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic(which) == 99
    with open(csrc / srcs[-1], "a") as f:
        f.write("\n// changed\n")
    assert bench.profiled_traffic(which) is None


def test_traffic_is_none_without_a_summary(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("prefill") is None


def test_committed_summaries_name_their_sources_and_traffic():
    for name, srcs in bench.PROFILES.values():
        text = open(os.path.join(REPO, "profiles", name)).read()
        assert "ncu " in text and "--clock-control none" in text
        for s in srcs:
            assert f"- {s} sha256: `" in text
        assert "- dram bytes per launch: `" in text
