"""The row samplers of the parity tests keep every tile and expert edge."""
import numpy as np

from parity import group_rows, sample_rows


def test_sample_rows_cover_every_tile_edge():
    rows = sample_rows(8192, 1024, seed=2)
    assert rows.size == 1024
    for t0 in range(0, 8192, 128):
        assert t0 in rows and t0 + 127 in rows
    ragged = sample_rows(300, 64, seed=1)
    assert {0, 127, 128, 255, 256, 299} <= set(ragged.tolist())
    assert sample_rows(100, 1000).tolist() == list(range(100))


def test_group_rows_cover_every_expert_and_tile_edge():
    offsets = np.array([0, 3, 3, 300, 301, 1000])
    rows = set(group_rows(offsets, 64, seed=0).tolist())
    # experts [0,3) [3,300) [300,301) [301,1000); tiles start at each expert's first row
    for r in (0, 2, 3, 130, 131, 258, 259, 299, 300, 301, 428, 429, 999):
        assert r in rows, r
    assert max(rows) < 1000
    assert len(group_rows(offsets, 2000)) == 1000
