"""Host-side checks of the benchmark's recorded-measurement logic (no GPU).

`bench.py` reports the decode kernel's DRAM traffic from `profiles/decode_traffic.txt`
only while the kernel sources match the hash recorded with the counters.  The hash
ignores comments, so these tests pin what counts as a change and what does not.
"""
import os

import bench


def test_comment_stripping_keeps_code_and_literals():
    src = ('int a = 1;  // trailing\n'
           '/* block\n comment */ const char* s = "// kept /* kept */";\n'
           "char c = '/'; char d = '\\''; x = y / z; /**/w = 2;")
    assert bench.strip_c_comments(src) == (
        "int a = 1; const char* s = \"// kept /* kept */\"; char c = '/'; "
        "char d = '\\''; x = y / z; w = 2;")


def test_comment_and_whitespace_edits_do_not_change_the_code_text():
    a = "__global__ void k(int* p) {\n    p[0] = 1;   // one\n}\n"
    b = "// header\n__global__ void k(int* p) {\n  /* set */ p[0] = 1;\n\n}\n"
    c = "__global__ void k(int* p) {\n    p[0] = 2;\n}\n"
    assert bench.strip_c_comments(a) == bench.strip_c_comments(b)
    assert bench.strip_c_comments(a) != bench.strip_c_comments(c)


def test_recorded_traffic_needs_matching_hash_and_workload():
    path = os.path.join(bench.ROOT, "profiles", "decode_traffic.txt")
    kv = {}
    with open(path, encoding="utf-8") as f:
        for line in f:
            if "=" in line and not line.startswith("#"):
                k, v = line.split("=", 1)
                kv[k.strip()] = v.strip()
    h = kv["kernel_source_sha256"]
    wl = kv["workload"]
    assert bench.recorded_traffic(h, wl) == float(kv["bytes_per_launch"])
    assert bench.recorded_traffic("0" * 64, wl) is None
    assert bench.recorded_traffic(h, wl + "_other") is None
