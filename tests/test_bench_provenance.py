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
