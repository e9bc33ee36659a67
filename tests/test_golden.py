"""Checks against the one figure the pages print for a concrete shape."""
import json
import os

HERE = os.path.dirname(os.path.abspath(__file__))


def test_materialisation_figure_64k():
    """P1 and P2 at 64K context, 32 heads, BF16: 2 * N^2 * H * 2 bytes = 512 GiB.

    This is the quadratic footprint the primitive avoids; the bench reports it
    beside the extra HBM it actually uses."""
    with open(os.path.join(HERE, "golden", "materialisation_64k.json")) as f:
        fx = json.load(f)
    n = fx["context_tokens"]
    total = fx["distributions"] * n * n * fx["heads"] * fx["dtype_bytes"]
    assert total == fx["quoted_gigabytes"] * 2**30
