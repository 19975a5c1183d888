"""Host logic of the benchmark on CPU: the traffic table's source key follows the
code, not its comments or layout, and every recorded capture belongs to the
sources as they stand (a stale entry would report counters of other code)."""
import bench


def test_source_key_ignores_comments_and_whitespace_but_not_code():
    a = "int f(int x) {\n    return x + 1;  // one more\n}\n"
    b = "/* header */\nint f(int x)\n{\n  return x + 1;\n}\n"
    c = "int f(int x) {\n    return x + 2;  // one more\n}\n"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)
    assert bench._code_only("x = 1; /* a\n multi-line\n comment */ y = 2;") == "x = 1; y = 2;"


def test_every_traffic_entry_matches_the_current_sources():
    hashes = {k: bench.stage1_source_hash(k) for k in bench.STAGE1_SOURCES}
    names = {w.name for w in bench.workloads().values()}
    for (kernel, workload, h), v in bench.KN1_TRAFFIC.items():
        assert h == hashes[kernel], (kernel, workload)
        assert v > 0 and workload in names, (kernel, workload)


def test_the_default_bench_line_carries_stage1_traffic():
    # the default workload (one request, 16 rows) runs the cluster stage-1
    # kernel; its DRAM counters must be on record for the current sources, or
    # the bench line's roofline.traffic would be null
    wl = bench.workloads()["single_request_B256"]
    key = ("kn1_kernel", wl.name, bench.stage1_source_hash("kn1_kernel"))
    assert bench.KN1_TRAFFIC.get(key, 0) > 0
