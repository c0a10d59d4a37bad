"""bench.py's host bookkeeping, no GPU: the kernel-source hash that keys the
committed ncu traffic figures, and the table of those figures."""
import os

import bench


def test_strip_comments_keeps_code_and_literals():
    src = ('int a = 1; // gone\n'
           '/* gone\n too */ const char* s = "x // kept /* kept */";\n'
           "char q = '\\''; char r = '\"'; const char* t = \"a\\\"b // kept\";  int   b;\n")
    got = bench.strip_comments(src)
    assert "gone" not in got
    assert '"x // kept /* kept */"' in got
    assert "'\\''" in got and "'\"'" in got
    assert '"a\\"b // kept"' in got
    assert got.endswith("int b;")


def test_strip_comments_tells_code_changes_apart():
    base = "x = a + b; // sum\n"
    assert bench.strip_comments(base) == bench.strip_comments("x = a + b;   /* the sum */\n")
    assert bench.strip_comments(base) != bench.strip_comments("x = a - b; // sum\n")
    assert bench.strip_comments("y = a+ +b;") != bench.strip_comments("y = a++b;")


def test_traffic_table_points_at_committed_summaries():
    for workload, (key, traffic, summary) in bench.NCU_TRAFFIC.items():
        assert len(key) == 16 and traffic > 0
        path = os.path.join(bench.ROOT, summary)
        assert os.path.exists(path), summary
        with open(path, encoding="utf-8") as f:
            text = f.read()
        assert f"{traffic:,}" in text, (workload, summary)
        assert key in text, (workload, summary)


def test_traffic_is_reported_only_at_its_hash(monkeypatch):
    workload, (key, traffic, _) = next(iter(bench.NCU_TRAFFIC.items()))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: key)
    assert bench.ncu_traffic(workload) == traffic
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0" * 16)
    assert bench.ncu_traffic(workload) is None
    assert bench.ncu_traffic("no_such_workload") is None
