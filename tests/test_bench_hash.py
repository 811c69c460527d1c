"""The source fingerprint that ties bench.py's DRAM-traffic figure to the
kernel sources it was captured from: comments do not count, code does."""
import os

import bench

SRC = """// header comment
#define A 1 /* trailing */
static const char *s = "a // b /* c */";
static const char c = '/';

int f(int x) {   // why
    /* several
       lines */
    return x + A;
}
"""


def test_comments_removed_literals_kept():
    got = bench.code_only(SRC)
    assert "header comment" not in got and "why" not in got and "several" not in got
    assert '"a // b /* c */"' in got and "'/'" in got
    assert "\n\n" not in got


def test_comment_edits_keep_code_edits_change():
    base = bench.code_only(SRC)
    assert bench.code_only(SRC.replace("// why", "// a longer reason\n    // on two lines")) == base
    assert bench.code_only(SRC.replace("/* trailing */", "")) == base
    assert bench.code_only(SRC.replace("return x + A;", "return x - A;")) != base
    assert bench.code_only(SRC.replace('"a // b', '"a // B')) != base
    assert bench.code_only(SRC.replace("#define A 1", "#define A 2")) != base


def test_hashed_sources_exist():
    csrc = os.path.join(bench.ROOT, "quantized_moe_expert_align_gb300", "csrc")
    for name in bench.KERNEL_SOURCES:
        assert os.path.exists(os.path.join(csrc, name)), name
