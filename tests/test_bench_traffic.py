"""The benchmark's `roofline.traffic` comes from the committed ncu summary of
the same workload, and only while the decode code is the code that summary
measured: comment edits keep it, code edits void it (no GPU needed)."""
import bench


def test_code_only_ignores_comments_and_whitespace():
    a = "int f(int x) {  // one\n  return x + 1; /* two\n lines */ }\n"
    b = "int f(int x){return x+1;}"
    assert bench.code_only(a) == bench.code_only(b)
    assert bench.code_only(a) != bench.code_only(a.replace("x + 1", "x + 2"))


def test_committed_profiles_match_the_current_decode_sources():
    assert bench.traffic_record("qwen7b") is not None
    assert bench.traffic_record("longctx") is not None
    assert bench.traffic_record("tiny") is None          # no capture of that workload


def test_traffic_is_voided_by_a_code_change(monkeypatch):
    real = bench.decode_source_sha()
    monkeypatch.setattr(bench, "decode_source_sha", lambda: "0" * 64 if real[0] != "0" else "1" * 64)
    assert bench.traffic_record("qwen7b") is None
