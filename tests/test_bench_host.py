"""The benchmark's host-side bookkeeping on CPU: the source hash that decides
whether a committed DRAM-traffic record still describes the kernel, and the
summary of the end-to-end steps' spacing."""
import json
import os

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

KERNEL = """// header comment
__global__ void k(float* x) {
  /* block
     comment */
  x[threadIdx.x] = 1.0f;  // trailing
}
"""


def _hash(files):
    return bench.kernel_source_hash("k.cu", read=lambda rel: files[os.path.basename(rel)])


def test_comment_and_layout_edits_keep_the_hash():
    base = _hash({"k.cu": KERNEL, "common.cuh": "#define A 1\n"})
    edited = KERNEL.replace("// header comment", "// a different header\n\n// and more").replace(
        "  x[threadIdx.x]", "      x[threadIdx.x]").replace("/* block", "/* another block")
    assert _hash({"k.cu": edited, "common.cuh": "#define A 1   // note\n\n"}) == base


def test_code_edits_change_the_hash():
    base = _hash({"k.cu": KERNEL, "common.cuh": "#define A 1\n"})
    assert _hash({"k.cu": KERNEL.replace("1.0f", "2.0f"), "common.cuh": "#define A 1\n"}) != base
    assert _hash({"k.cu": KERNEL, "common.cuh": "#define A 2\n"}) != base


def test_committed_traffic_records_name_files_that_exist():
    rec = json.load(open(os.path.join(ROOT, "profiles", "traffic.txt")))
    for name, r in rec.items():
        assert os.path.exists(os.path.join(ROOT, "block_sparse_attention_05_gb300", "csrc", r["source"])), name
        assert r["units"] > 0 and r["dram_bytes"] > 0 and r["units_kind"] in ("total_q", "total_k")


def test_step_spacing_flags_a_stalled_step():
    sp = bench.step_spacing([21.0, 21.5, 118.0, 20.8, 21.2])
    assert sp["median"] == 21.2 and sp["min"] == 20.8 and sp["max"] == 118.0
    assert sp["over_2x_median"] == 1
    assert bench.step_spacing([5.0, 5.0, 5.0])["over_2x_median"] == 0
