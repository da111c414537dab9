"""The bench's traffic record: the ncu figure of the dominant kernel is used
only while the hash of the kernel's code matches the one recorded with the
capture; comments and blank space do not count as code."""
import os

import bench


def test_code_of_drops_comments_and_space_but_keeps_strings():
    src = 'int a = 1;  // one\n/* block\n comment */ const char *s = "x // y /* z */";\n\n  b++; // tail'
    assert bench.code_of(src) == 'int a = 1; const char *s = "x // y /* z */"; b++;'
    # an escaped quote inside a string does not end it
    assert bench.code_of('s = "a\\"b // c"; // d') == 's = "a\\"b // c";'


def test_hash_follows_code_not_comments(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (tmp_path / "k.cu").write_text("__global__ void k() { x = 1; }  // v1\n")
    h1 = bench.sources_sha256(["k.cu"])
    (tmp_path / "k.cu").write_text("// a new comment\n__global__ void k() {\n  x = 1;\n}\n")
    assert bench.sources_sha256(["k.cu"]) == h1
    (tmp_path / "k.cu").write_text("__global__ void k() { x = 2; }\n")
    assert bench.sources_sha256(["k.cu"]) != h1


def test_traffic_record_needs_a_matching_hash(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (tmp_path / "k.cu").write_text("__global__ void k() {}\n")
    sha = bench.sources_sha256(["k.cu"])
    prof = tmp_path / "p.md"
    prof.write_text(f"# summary\n\ntraffic-record: kernel=k batch=4 bytes_per_launch=1000 sha256={sha}\n")
    assert bench.traffic_record("p.md", ["k.cu"]) == ((1000.0, 4), None)
    (tmp_path / "k.cu").write_text("__global__ void k() { y(); }\n")
    rec, why = bench.traffic_record("p.md", ["k.cu"])
    assert rec is None and "changed" in why
    assert bench.traffic_record(os.path.join("missing.md"), ["k.cu"])[0] is None
