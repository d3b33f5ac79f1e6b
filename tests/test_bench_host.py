"""Host-side helpers of bench.py (no GPU): the source key that decides
whether the recorded DRAM traffic of the search kernel still applies."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_strip_comments_keeps_code_and_literals():
    src = ('int a = 1;  // trailing\n'
           '/* block\n   comment */\n'
           'const char* s = "a // b /* c */";\n'
           "char q = '\"';  /* inline */ int b;\n"
           '\n   \n'
           'x();\n')
    assert bench.strip_comments(src) == ('int a = 1;\n'
                                         'const char* s = "a // b /* c */";\n'
                                         "char q = '\"';   int b;\n"
                                         'x();')


def test_comment_only_edits_keep_the_key_and_code_edits_change_it():
    base = "__global__ void k(int* p) {\n    p[0] = 1;  // store\n}\n"
    reworded = "// a kernel\n__global__ void k(int* p) {\n    p[0] = 1;  /* the store */\n}\n"
    changed = "__global__ void k(int* p) {\n    p[0] = 2;  // store\n}\n"
    assert bench.strip_comments(base) == bench.strip_comments(reworded)
    assert bench.strip_comments(base) != bench.strip_comments(changed)


def test_traffic_record_is_well_formed():
    t = bench.SEARCH_TRAFFIC
    assert set(t) == {"bytes_per_step", "src_sha"}
    assert t["bytes_per_step"] > 0 and len(t["src_sha"]) == 16
    assert bench.src_sha(bench.SEARCH_SOURCES) == bench.src_sha(bench.SEARCH_SOURCES)
