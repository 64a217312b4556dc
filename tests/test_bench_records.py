"""Host logic of bench.py that needs no GPU: the source hash that ties a
recorded DRAM-traffic figure to the kernel code it was measured on."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_strip_comments_drops_comments_and_blank_lines_only():
    src = 'int a = 1;  // one\n\n/* two\n   lines */ int b = 2;\nconst char *s = "x // y /* z */";\n'
    assert bench.strip_comments(src) == 'int a = 1;\n  int b = 2;\nconst char *s = "x // y /* z */";'


def test_strip_comments_keeps_character_and_escaped_literals():
    src = "char c = '/'; char d = '*'; const char *e = \"a\\\"//b\"; // gone\n"
    assert bench.strip_comments(src) == "char c = '/'; char d = '*'; const char *e = \"a\\\"//b\";"


def test_comment_edit_keeps_the_hash_and_a_code_edit_changes_it():
    base = "__global__ void k(int *p)\n{\n    p[0] = 1;  // store\n}\n"
    comment_edit = "// a kernel\n__global__ void k(int *p)\n{\n    p[0] = 1;  /* the store */\n}\n"
    code_edit = "__global__ void k(int *p)\n{\n    p[0] = 2;  // store\n}\n"
    assert bench.strip_comments(base) == bench.strip_comments(comment_edit)
    assert bench.strip_comments(base) != bench.strip_comments(code_edit)


def test_traffic_is_withheld_for_unrecorded_or_changed_code(monkeypatch):
    assert bench.profiled_traffic("no_such_workload", "paged_decode_kernel") is None
    rec = dict(bench.PROFILED_TRAFFIC)
    key = ("decode_b256", "paged_decode_kernel")
    rec[key] = {"sources_sha256": "0" * 64, "bytes": 1}
    monkeypatch.setattr(bench, "PROFILED_TRAFFIC", rec)
    assert bench.profiled_traffic(*key) is None
    rec[key] = {"sources_sha256": bench.kernel_sources_sha("paged_decode_kernel"), "bytes": 7}
    assert bench.profiled_traffic(*key) == 7
