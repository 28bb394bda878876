"""bench.py's record of which sources each timed kernel is built from: a
committed DRAM-traffic figure is reported only while the code of those files
(comments and layout aside) is unchanged, so every kernel source must belong
to some family."""
import os

import bench

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "paged_kv_cache_153_gb300", "csrc")


def test_every_kernel_source_is_in_a_family():
    listed = set()
    for names in bench.KERNEL_SOURCES.values():
        for name in names:
            assert os.path.isfile(os.path.join(CSRC, name)), name
            listed.add(name)
    kernel_files = {n for n in os.listdir(CSRC) if n.endswith((".cu", ".cuh"))}
    # noalloc.cu is the workspace-free decode entry point, which no bench
    # workload times
    assert kernel_files - listed <= {"noalloc.cu"}, sorted(kernel_files - listed)


def test_digest_depends_only_on_its_family():
    # the workloads map to their families; the digests are stable strings
    assert bench.source_family("mha7b") == "decode"
    assert bench.source_family("prefill") == "prefill"
    assert bench.source_family("int8") == "int8"
    assert bench.source_family("cow") == "cow"
    for fam in bench.KERNEL_SOURCES:
        d = bench.kernel_source_digest(fam)
        assert len(d) == 16 and d == bench.kernel_source_digest(fam)
    assert len({bench.kernel_source_digest(f) for f in bench.KERNEL_SOURCES}) == len(bench.KERNEL_SOURCES)


def test_code_only_drops_comments_and_layout_but_keeps_literals():
    src = 'int a = 1; // note\n/* block\n comment */  int  b = 2;\nasm("x // y; /* z */");\nchar c = \'/\';'
    assert bench.code_only(src) == 'int a = 1; int b = 2; asm("x // y; /* z */"); char c = \'/\';'
    # a comment edit leaves the code as it was; a code edit does not
    assert bench.code_only("x = 1; // one") == bench.code_only("x = 1;   // another\n")
    assert bench.code_only("x = 1;") != bench.code_only("x = 2;")
    assert bench.code_only('s = "a\\"//b";') == 's = "a\\"//b";'
