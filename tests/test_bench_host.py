"""Host logic of bench.py that needs no GPU: the DRAM-traffic tables that
feed the roofline's `traffic` field are well formed and used only while the
kernel's translation unit (the source and every header it includes) still
hashes to the one the counters were taken on; the
oracle's thread-rate helper counts the work of every thread."""
import hashlib
import os
import re

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _entries():
    for table, source in ((bench.VERIFY_TRAFFIC, "verify.cu"), (bench.CUT_TRAFFIC, "sampling.cu")):
        for workload, entry in table.items():
            yield table, source, workload, entry


def test_traffic_tables_are_well_formed():
    seen = 0
    for _, source, workload, entry in _entries():
        assert entry["bytes"] > 0, workload
        assert set(entry) == {"bytes", "code_sha256"}, workload
        assert re.fullmatch(r"[0-9a-f]{64}", entry["code_sha256"]), workload
        seen += 1
    assert seen >= 4


def test_traffic_only_for_the_captured_code():
    for table, source, workload, entry in _entries():
        current = bench._tu_code_sha256(source)
        same = {workload: dict(entry, code_sha256=current)}
        other = {workload: dict(entry, code_sha256="0" * 64)}
        assert bench._traffic(same, workload, source) == entry["bytes"]
        assert bench._traffic(other, workload, source) is None
        assert bench._traffic(table, "no_such_workload", source) is None


def test_translation_unit_holds_the_included_headers():
    names = [os.path.basename(p) for p in bench._tu_sources("verify.cu")]
    assert names[0] == "verify.cu"
    assert {"common.cuh", "philox.cuh", "sampling.cuh", "samspec.h"} <= set(names)
    assert len(names) == len(set(names))
    names = [os.path.basename(p) for p in bench._tu_sources("sampling.cu")]
    assert names[0] == "sampling.cu" and "common.cuh" in names and "philox.cuh" not in names


def test_code_hash_ignores_comments_only(tmp_path):
    a = tmp_path / "a.cu"
    a.write_text('int f() {  // one\n  return 1;\n}\nconst char* s = "a // b";\n')
    b = tmp_path / "b.cu"
    b.write_text('/* a new\n   header */\n// line\nint f() {  // two\n\n  return 1;   \n}\n'
                 'const char* s = "a // b";  /* end */\n')
    b2 = tmp_path / "sub"
    b2.mkdir()
    b2 = b2 / "a.cu"  # same name, same code: same hash
    b2.write_text(b.read_text())
    c = tmp_path / "c.cu"
    c.write_text('int f() {  // one\n  return 2;\n}\nconst char* s = "a // b";\n')
    d = tmp_path / "d.cu"  # a code edit inside a string literal
    d.write_text('int f() {  // one\n  return 1;\n}\nconst char* s = "a // c";\n')
    assert bench._code_sha256(a) == bench._code_sha256(b2)
    assert bench._code_sha256(a) != bench._code_sha256(b)  # the file name is part of the hash
    assert bench._code_sha256(a) != bench._code_sha256(c)
    assert bench._code_sha256(a) != bench._code_sha256(d)
    assert bench._code_sha256(a, c) != bench._code_sha256(a)
    assert bench._code_sha256(a) != hashlib.sha256(a.read_bytes()).hexdigest()


def test_a_header_edit_changes_the_translation_unit_hash(tmp_path, monkeypatch):
    csrc, inc = tmp_path / "csrc", tmp_path / "include"
    csrc.mkdir()
    inc.mkdir()
    (csrc / "k.cu").write_text('#include "h.cuh"\n#include "api.h"\nint k() { return H; }\n')
    (csrc / "h.cuh").write_text("#define H 1  // one\n")
    (inc / "api.h").write_text("/* api */\nint k();\n")
    monkeypatch.setattr(bench, "CSRC", str(csrc))
    monkeypatch.setattr(bench, "INCLUDE", str(inc))
    h0 = bench._tu_code_sha256("k.cu")
    (csrc / "h.cuh").write_text("// the constant\n#define H 1\n")
    assert bench._tu_code_sha256("k.cu") == h0
    (csrc / "h.cuh").write_text("#define H 2\n")
    assert bench._tu_code_sha256("k.cu") != h0


def test_thread_rate_counts_every_thread():
    calls = []

    def work(t, i):
        calls.append((t, i))
        return 3

    rate, units, wall = bench._threads_rate(work, 4, 0.2)
    assert units == 3 * len(calls) and wall >= 0.2 and rate > 0
    assert {t for t, _ in calls} == {0, 1, 2, 3}
    assert bench._nproc() >= 1


def test_default_workload_is_the_b1024_verify_point():
    cfg = bench.head_config(1)
    assert cfg["workload"] == bench.HEAD_WORKLOAD
    assert (cfg["B_per_gpu"], cfg["K"], cfg["temperature"]) == (1024, 3, 1.0)
