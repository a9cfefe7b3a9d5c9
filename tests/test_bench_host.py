"""Host-side logic of bench.py that needs no GPU: the kernel-source hash that
ties recorded DRAM counters to the code they were taken on."""

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_code_only_drops_comments_and_blank_lines_but_keeps_literals():
    src = 'int a = 1;  // note\n\n/* block\n comment */ const char* s = "// x /* y */";\n  f(\'/\');\n'
    assert bench._code_only(src) == 'int a = 1;\nconst char* s = "// x /* y */";\nf(\'/\');'


def test_comment_only_edits_keep_the_hash_and_code_edits_change_it():
    base = "__global__ void k(int* p) {\n  p[0] = 1;  // store\n}\n"
    same = "// header\n__global__ void k(int* p) {\n\n  p[0] = 1;  /* store */\n}\n"
    other = "__global__ void k(int* p) {\n  p[0] = 2;\n}\n"
    assert bench._code_only(base) == bench._code_only(same)
    assert bench._code_only(base) != bench._code_only(other)


def test_recorded_traffic_matches_the_current_source():
    # The committed ncu summary carries the code hash it was taken on; bench
    # reports its traffic only while that still matches.
    path = os.path.join(ROOT, "profiles", "fwd_dual_tc_bf16_b4h16n2048d128_traffic.txt")
    fields = dict(line.split(":", 1) for line in open(path) if ":" in line)
    recorded = fields["source_hash"].strip()
    if recorded == bench.source_hash():
        assert bench.recorded_traffic("bf16_b4h16n2048d128") == float(
            fields["dram_bytes_per_launch"])
    else:
        assert bench.recorded_traffic("bf16_b4h16n2048d128") is None
