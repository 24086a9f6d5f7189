"""Host logic of bench.py that needs no GPU: the DRAM-traffic tables that
feed the roofline's `traffic` field are well formed and used only while the
kernel source still hashes to the one the counters were taken on; the
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
        assert set(entry) == {"bytes", source.replace(".", "_") + "_code_sha256"}, workload
        assert re.fullmatch(r"[0-9a-f]{64}", entry[source.replace(".", "_") + "_code_sha256"]), workload
        seen += 1
    assert seen >= 4


def test_traffic_only_for_the_captured_source():
    for table, source, workload, entry in _entries():
        path = os.path.join(ROOT, "sam_drafting_verification_gb300", "csrc", source)
        current = bench._code_sha256(path)
        key = source.replace(".", "_") + "_code_sha256"
        same = {workload: dict(entry, **{key: current})}
        other = {workload: dict(entry, **{key: "0" * 64})}
        assert bench._traffic(same, workload, source) == entry["bytes"]
        assert bench._traffic(other, workload, source) is None
        assert bench._traffic(table, "no_such_workload", source) is None


def test_code_hash_ignores_comments_only(tmp_path):
    a = tmp_path / "a.cu"
    a.write_text("int f() {  // one\n  return 1;\n}\n")
    b = tmp_path / "b.cu"
    b.write_text("// a new header\nint f() {  // two\n\n  return 1;   \n}\n")
    c = tmp_path / "c.cu"
    c.write_text("int f() {  // one\n  return 2;\n}\n")
    assert bench._code_sha256(a) == bench._code_sha256(b)
    assert bench._code_sha256(a) != bench._code_sha256(c)
    assert bench._code_sha256(a) != hashlib.sha256(a.read_bytes()).hexdigest()


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
