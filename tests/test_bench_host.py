"""Host logic of bench.py (no GPU): the kernel-source hash that keys the
committed ncu traffic figures, and the lookup that uses it."""
import re

import bench


def test_comment_edits_leave_the_code_unchanged():
    a = "int f(int x) {  // doubles\n  return 2 * x;  /* plain */\n}\n"
    b = "/* header\n   block */\nint f(int x) {\n\n  return 2 * x;\n}  // end\n"
    assert bench._strip_comments(a) == bench._strip_comments(b)
    assert bench._strip_comments(a) != bench._strip_comments(a.replace("2 * x", "3 * x"))


def test_source_hash_and_traffic_lookup():
    h = bench._csrc_hash()
    assert re.fullmatch(r"[0-9a-f]{16}", h)
    assert bench._traffic("no_such_kernel", bench.MAIN) is None
    assert bench._traffic("dwgu", "no_such_workload") is None
    t = bench._traffic("dwgu", bench.MAIN)  # committed figures, while the hash matches
    assert t is None or t > 0
