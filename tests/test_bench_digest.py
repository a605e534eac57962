"""The key of the recorded ncu counters: a digest of the code a kernel is
compiled from, blind to comments and spacing (CPU only)."""
from __future__ import annotations

import os

import bench

CSRC = os.path.join(bench.ROOT, "row_normalization_gb300", "csrc")


def test_code_only_drops_comments_and_keeps_literals():
    src = ('int a = 1;   // one\n/* two\n lines */ const char *s = "x // kept /* kept */";\n'
           "char q = '\"'; asm(\"mov.u32 %0, 1; // kept\");\n")
    assert bench.code_only(src) == (
        'int a = 1; const char *s = "x // kept /* kept */"; char q = \'"\'; '
        'asm("mov.u32 %0, 1; // kept");')


def test_comment_edits_keep_the_code_and_code_edits_change_it():
    with open(os.path.join(CSRC, "qk_norm_rope.cu"), encoding="utf-8") as fh:
        src = fh.read()
    commented = src.replace("\n", "\n// a remark that changes nothing\n", 1) + "\n/* and another */\n"
    respaced = src.replace(";\n", ";\n\n  ")
    assert bench.code_only(commented) == bench.code_only(src)
    assert bench.code_only(respaced) == bench.code_only(src)
    edited = src.replace("constexpr int G = 32 / LPH;", "constexpr int G = 16 / LPH;", 1)
    assert edited != src
    assert bench.code_only(edited) != bench.code_only(src)


def test_each_kernel_family_has_its_own_digest():
    assert bench.kernel_source_digest("rms_persistent_bulk_kernel") != \
        bench.kernel_source_digest("qk_persistent_bulk_kernel")
    assert len(bench.kernel_source_digest("qk_pair_kernel")) == 16
