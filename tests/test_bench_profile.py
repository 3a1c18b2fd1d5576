"""bench.py's link between the committed DRAM counters and the kernel code:
the source hash ignores comments and whitespace (a comment-only edit keeps the
counters attached) and changes with any code edit (a kernel change drops
them)."""

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

CODE = """// a kernel
__device__ int f(int a) {  /* block
   comment */
    return a + 1;  // trailing
}
"""


def test_code_only_ignores_comments_and_whitespace():
    same = CODE.replace("// a kernel", "// another comment, longer").replace("  // trailing", "")
    same = same.replace("/* block\n   comment */", "/* x */").replace("    return", "\treturn")
    assert bench._code_only(CODE) == bench._code_only(same)
    assert bench._code_only(CODE) == "__device__ int f(int a) { return a + 1; }"


def test_code_only_sees_code_edits():
    assert bench._code_only(CODE) != bench._code_only(CODE.replace("a + 1", "a + 2"))
    assert bench._code_only(CODE) != bench._code_only(CODE.replace("int f", "int g"))


def test_dram_summary_attaches_only_to_its_code():
    # the bench line carries the committed traffic exactly when the summary's
    # hash is that of the kernel as it stands, and never for another workload
    import re
    with open(bench.DRAM_PROFILE) as f:
        prof = dict(m.groups() for m in re.finditer(r"^- (\w+): (\S+)\s*$", f.read(), re.M))
    same = prof["kernel_src_sha256"] == bench.kernel_source_hash()
    got = bench.dram_traffic_per_launch("msweep")
    assert got == (float(prof["bytes_per_launch_mean"]) if same else None)
    assert bench.dram_traffic_per_launch("other") is None
