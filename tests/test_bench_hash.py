"""The benchmark's kernel-source hash, which keys the committed ncu traffic
records: it covers the code and leaves comments out, so a comment edit keeps
a record valid while any code change makes the bench report traffic as
unknown (null) until the counters are taken again."""

import bench


def test_code_only_strips_comments_and_blank_lines():
    a = "int x = 1;  // one\n/* block\n comment */\nint y = 2;\n\n"
    b = "int x = 1;\nint y = 2;"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only("int x = 1;") != bench._code_only("int x = 2;")


def test_kernel_hashes_cover_each_kernel():
    quad = bench.kernel_source_hash("partial_quad_kernel")
    pair = bench.kernel_source_hash("partial_pair_kernel")
    assert len(quad) == 16 and len(pair) == 16 and quad != pair
    assert quad == bench.kernel_source_hash()  # the default is the four-SM kernel
