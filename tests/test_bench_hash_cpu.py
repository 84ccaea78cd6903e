"""The key under which measured DRAM traffic is recorded: the kernel sources'
code without comments or layout (a comment edit keeps a measurement, a code
edit invalidates it)."""

import bench


def test_code_only_drops_comments_and_layout():
    src = 'int a = 1;  // note\n/* block\n comment */ int  b =\n 2;\n'
    assert bench.code_only(src) == "int a = 1; int b = 2;"
    # comment markers inside string and character literals are code
    assert bench.code_only('s = "// not a comment"; c = \'/\';') == 's = "// not a comment"; c = \'/\';'
    assert bench.code_only("x = '\\''; // q") == "x = '\\'';"


def test_comment_edit_keeps_code_edit_changes_the_key():
    a = "__global__ void k(int* p) { p[0] = 1; }  // one\n"
    b = "// the kernel\n__global__ void k(int* p) {\n  p[0] = 1;\n}\n"
    c = "__global__ void k(int* p) { p[0] = 2; }\n"
    assert bench.code_only(a) == bench.code_only(b)
    assert bench.code_only(a) != bench.code_only(c)

