"""Layout fixtures taken from the pages (tests/golden), CPU only."""
import json
import os

import numpy as np

from gen.workloads import assemble_bdsv_dense

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_glass_strip_layout_fixture():
    g = json.load(open(os.path.join(GOLDEN, "glass_strip_layout.json")))
    bs, nbr = g["block_size"], g["num_block_rows"]
    strips = np.arange(nbr * bs * 3 * bs, dtype=np.float64).reshape(1, nbr, bs, 3 * bs)
    dense = assemble_bdsv_dense(strips)[0]
    for c in g["cases"]:
        assert dense[c["dense_row"], c["dense_col"]] == c["strip_offset"], c
    for c in g["vector_cases"]:
        assert c["padded_offset"] == bs + c["dense_row"]
