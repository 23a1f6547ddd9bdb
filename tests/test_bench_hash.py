"""The kernel-source hash that ties profiles/dram_traffic.json to the code it
was captured on: comments and whitespace do not change it, code does."""

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_comments_and_whitespace_are_ignored():
    a = "int x = 1; // one\n/* block\n comment */ int y = 2;\n"
    b = "int x = 1;\n\n   int y = 2; // two"
    assert bench._code_only(a) == bench._code_only(b) == "int x = 1; int y = 2;"


def test_literals_are_kept_whole():
    src = 'const char* s = "a // not a comment /* nor this */"; char c = \'/\'; char q = \'"\';'
    assert bench._code_only(src) == src
    esc = 'puts("quote \\" // still inside"); // gone'
    assert bench._code_only(esc) == 'puts("quote \\" // still inside");'


def test_code_changes_change_the_code_text():
    assert bench._code_only("x = a + b;") != bench._code_only("x = a - b;")
    assert bench._code_only("f(1);") != bench._code_only("f(1); g();")


def test_hash_is_stable_and_hex():
    h1, h2 = bench.kernel_source_hash(), bench.kernel_source_hash()
    assert h1 == h2 and len(h1) == 64 and all(c in "0123456789abcdef" for c in h1)
