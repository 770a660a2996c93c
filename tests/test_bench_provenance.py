"""The bench record's provenance and the oracle's determinism (CPU): the
same seeded inputs hash the same, a changed input changes the hash, and the
oracle run twice on the same inputs gives the same bits."""
import numpy as np

import bench
import oracle
import workloads

CFG = workloads.BLOCK_CONFIGS["tiny_stablelm2"]


def test_provenance_hashes_follow_the_inputs():
    x, w = workloads.block_inputs(CFG)
    a = bench._provenance(CFG, x, w)
    b = bench._provenance(CFG, *workloads.block_inputs(CFG))
    assert a["inputs_sha256"] == b["inputs_sha256"] and a["seed"] == CFG.seed
    assert a["sources_sha256"] == b["sources_sha256"] and len(a["sources_sha256"]) == 64
    x2 = x.clone()
    x2[0, 0, 0] = -x2[0, 0, 0] if float(x2[0, 0, 0]) != 0 else 1
    assert bench._provenance(CFG, x2, w)["inputs_sha256"] != a["inputs_sha256"]


def test_oracle_is_deterministic():
    x, w = workloads.block_inputs(CFG)
    y1 = oracle.block_forward(CFG, x, w)["y"]
    y2 = oracle.block_forward(CFG, x, w)["y"]
    assert np.array_equal(y1, y2)


def test_kernel_source_hash_ignores_comments_only(tmp_path, monkeypatch):
    """The hash that ties the recorded ncu traffic to the GEMM's sources is
    blind to comment and blank-line edits and sees any code edit."""
    import os
    src = tmp_path / "k.cu"
    src.write_text("int a = 1;  // first\n\nint b = 2;\n")
    monkeypatch.setitem(bench._KERNEL_SOURCES, "probe", (os.path.relpath(src, os.path.dirname(
        os.path.abspath(bench.__file__))),))
    h0 = bench._sources_sha("probe")
    src.write_text("// a new comment\nint a = 1;  // changed\nint b = 2;\n\n")
    assert bench._sources_sha("probe") == h0
    src.write_text("int a = 1;\nint b = 3;\n")
    assert bench._sources_sha("probe") != h0
