"""The kernel-source digest that ties recorded ncu counters to the sources:
comment and layout edits keep it, any code edit changes it, and the
committed counters are keyed to the current sources."""
import json
import os
import shutil

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_comments_and_layout_are_ignored():
    a = "int f(int x) {\n  return x + 1;  // add one\n}\n"
    b = "/* the successor */\nint f(int x) { return x + 1; }\n"
    assert bench._code_only(a) == bench._code_only(b)


def test_code_changes_and_literals_are_kept():
    assert bench._code_only("x = a + 1;") != bench._code_only("x = a + 2;")
    # comment markers inside literals are code
    s = 'const char* p = "a//b/*c*/"; char q = \'/\';'
    assert bench._code_only(s) == s
    assert bench._code_only('s = "\\"//"; // tail') == 's = "\\"//";'


def _copy_sources(tmp_path):
    pkg = os.path.join(ROOT, "eagle_speculative_drafting_gb300")
    dst = tmp_path / "eagle_speculative_drafting_gb300" / "csrc"
    shutil.copytree(os.path.join(pkg, "csrc"), dst)
    shutil.copy(os.path.join(pkg, "_build.py"), tmp_path / "eagle_speculative_drafting_gb300" / "_build.py")
    (tmp_path / "include").mkdir()
    shutil.copy(os.path.join(ROOT, "include", "peagle.h"), tmp_path / "include" / "peagle.h")
    return dst


def test_digest_follows_code_not_comments(tmp_path):
    dst = _copy_sources(tmp_path)
    base = bench.source_digest(str(tmp_path))
    assert base == bench.source_digest()
    f = dst / sorted(os.listdir(dst))[0]
    text = f.read_text()
    f.write_text("// a new comment line\n" + text.replace("\n", "\n\n", 3))
    assert bench.source_digest(str(tmp_path)) == base
    f.write_text(text + "\nstatic int unused_marker_for_the_test = 1;\n")
    assert bench.source_digest(str(tmp_path)) != base


def test_recorded_counters_are_keyed_and_summarised():
    # a record taken on other kernel sources is simply not used (bench
    # reports traffic null); every record names its digest and its summary
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as fh:
        rec = json.load(fh)
    assert rec, "no recorded counters"
    for key, e in rec.items():
        assert len(e["source_digest"]) == 16 and int(e["source_digest"], 16) >= 0, key
        assert e["dram_bytes_per_launch"] > 0, key
        assert os.path.exists(os.path.join(ROOT, e["summary"])), key
        if e["source_digest"] == bench.source_digest():
            workload, op = key.split(":")
            assert bench.recorded_traffic(op, workload) == e["dram_bytes_per_launch"]


def test_digest_covers_the_header_and_build_flags(tmp_path):
    _copy_sources(tmp_path)
    base = bench.source_digest(str(tmp_path))
    hdr = tmp_path / "include" / "peagle.h"
    text = hdr.read_text()
    hdr.write_text(text.replace("#define PEAGLE_DEV_TIMEOUT 0x2", "#define PEAGLE_DEV_TIMEOUT 0x4"))
    assert bench.source_digest(str(tmp_path)) != base
    hdr.write_text(text)
    assert bench.source_digest(str(tmp_path)) == base
    b = tmp_path / "eagle_speculative_drafting_gb300" / "_build.py"
    bt = b.read_text()
    b.write_text(bt.replace('"-O3"', '"-O2"'))
    assert bench.source_digest(str(tmp_path)) != base
