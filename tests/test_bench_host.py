"""Host-side helpers of the benchmark (no GPU): the executed-tile count it
reports for the chunked prefill, read from a plan buffer laid out as the
library writes it."""

import numpy as np
import torch

import bench


def _plan(batch, chunk_len, klo, khi):
    def a256(x):
        return (x + 255) & ~255
    nqt = (chunk_len + 127) // 128
    rows = a256(batch * chunk_len * 4)
    tiles = a256(batch * nqt * 4)
    buf = np.zeros(256 + 2 * rows + 2 * tiles, dtype=np.uint8)
    off = 256 + 2 * rows
    buf[off:off + batch * nqt * 4] = np.asarray(klo, dtype=np.int32).view(np.uint8)
    buf[off + tiles:off + tiles + batch * nqt * 4] = np.asarray(khi, dtype=np.int32).view(np.uint8)
    return torch.from_numpy(buf)


def test_executed_tile_pairs():
    # two sequences, 300 rows per chunk (3 query tiles each)
    klo = [0, 0, 100, 5, 0, 0]
    khi = [128, 129, 356, 6, 0, 0]  # 1, 2, 3 (keys 100..355 span tiles 0..2), 1, empty, empty
    got = bench.executed_tile_pairs(_plan(2, 300, klo, khi), 2, 300)
    assert got == (1 + 2 + 3 + 1) * 128 * 128
