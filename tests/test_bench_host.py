"""Host-side pieces of bench.py that decide what a bench line reports: the
source hash that ties the committed ncu traffic record to the kernel it was
taken on (comments and whitespace do not count, code does), and the lookup
that reports that traffic only for a matching hash."""
import importlib.util
import json
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_host_under_test", os.path.join(ROOT, "bench.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    return b


SRC = """// a kernel
__global__ void k(float* y) {   /* one
   thread */
    y[threadIdx.x] = 1.0f;  // store
}
"""


def test_code_hash_ignores_comments_and_whitespace():
    b = _bench()
    h = b.code_hash([SRC])
    assert b.code_hash([SRC.replace("// a kernel", "// the same kernel, reworded")]) == h
    assert b.code_hash([SRC.replace("/* one\n   thread */", "")]) == h
    assert b.code_hash([SRC.replace("    y[", "\ty[")]) == h


def test_code_hash_follows_code():
    b = _bench()
    h = b.code_hash([SRC])
    assert b.code_hash([SRC.replace("1.0f", "2.0f")]) != h
    assert b.code_hash([SRC.replace("threadIdx.x", "threadIdx.y")]) != h
    assert b.code_hash([SRC, ""]) == h and b.code_hash([SRC, "int x;"]) != h


def test_traffic_reported_only_for_the_hash_it_was_taken_on(tmp_path, monkeypatch):
    b = _bench()
    (tmp_path / "profiles").mkdir()
    rec = {"layer_m1": {"dram_read": 300, "dram_write": 7, "dram_bytes_per_launch": 307, "source_hash": "abc",
                        "sources": "token"}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(b, "ROOT", str(tmp_path))
    monkeypatch.setattr(b, "kernel_source_hash", lambda which: "abc" if which == "token" else "zzz")
    assert b.ncu_traffic("layer", 1) == 307.0
    assert b.ncu_traffic("layer", 16) is None        # no record for that workload
    # a record of a smaller case scales with the launch's algorithmic bytes
    rec["layer_m1"]["algorithmic_bytes"] = 100
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    assert b.ncu_traffic("layer", 1, 100) == 307.0
    assert b.ncu_traffic("layer", 1, 200) == 614.0
    monkeypatch.setattr(b, "kernel_source_hash", lambda which: "def")
    assert b.ncu_traffic("layer", 1) is None          # the kernel changed since the capture


def test_committed_traffic_record_is_consistent():
    b = _bench()
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        for e in json.load(f).values():
            assert e["dram_bytes_per_launch"] == e["dram_read"] + e["dram_write"]
            assert len(e["source_hash"]) == 16 and "ncu" in e["command"]
            assert e["sources"] in b.KERNEL_SOURCES
