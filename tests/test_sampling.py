"""The row sampler the full-size parity tests use: every 128-row query tile
of every chunk and head gets a row, and the rows' lanes cover a whole tile."""
import numpy as np

import synth


def test_tile_rows_cover_every_tile_and_lane():
    heads, n_rows, chunk = 4, 54000, 54000
    rows = synth.tile_rows(heads, n_rows, chunk)
    h, r = rows // n_rows, rows % n_rows
    tiles = set(zip(h.tolist(), (r // 128).tolist()))
    assert tiles == {(a, t) for a in range(heads) for t in range((chunk + 127) // 128)}
    assert set((r % 128).tolist()) == set(range(128))


def test_tile_rows_short_last_tile_and_chunks():
    # 3,600-row chunks end in a 16-row tile: every one of its rows is met
    heads, n_rows, chunk = 24, 14400, 3600
    rows = synth.tile_rows(heads, n_rows, chunk)
    assert rows.max() < heads * n_rows and len(np.unique(rows)) == len(rows)
    r = rows % n_rows
    c, i = r // chunk, r % chunk
    assert len(rows) == heads * (n_rows // chunk) * 29
    assert set((i[i >= 3584] - 3584).tolist()) == set(range(16))
    assert set(c.tolist()) == {0, 1, 2, 3}
