"""Pins of the oracle's scale layouts (oracle.scale_layout), each an
independent property of the target layout rather than its index formula:

  * swizzled (the tiled E8M0 layout of block-scaled MMA operands): the
    rearrangement is a bijection onto the padded buffer, with zeros in the
    padding; every 512-entry tile holds exactly one 128-row x 4-column block;
    tiles follow each other tile-column fastest; every 16-entry line of a
    tile holds the rows j, j+32, j+64, j+96 of its band, each row's 4
    columns contiguous and in order;
  * column-major: numpy's transpose, zero-padded to a multiple of 4 rows.

The GPU test tests/test_gpu_layouts.py pins the swizzled layout once more
against a block-scaled GEMM library consumer.
"""
import numpy as np
import pytest

import oracle


def _ids(M, G):
    """Unique positive ids for every (row, column): id = r * G + g + 1."""
    return (np.arange(M * G, dtype=np.int64) + 1).reshape(M, G)


@pytest.mark.parametrize("M,G", [(1, 1), (128, 4), (200, 130), (300, 9), (7, 192)])
def test_swizzled_is_a_bijection_with_zero_padding(M, G):
    out = oracle.scale_layout("mxfp8", _ids(M, G), "swizzled")
    Mp, Gp = -(-M // 128) * 128, -(-G // 4) * 4
    assert out.shape == (Mp, Gp)
    flat = out.ravel()
    vals = flat[flat != 0]
    assert np.array_equal(np.sort(vals), np.arange(1, M * G + 1))
    assert (flat == 0).sum() == Mp * Gp - M * G


@pytest.mark.parametrize("M,G", [(256, 8), (200, 130), (130, 6)])
def test_swizzled_tiles_and_lines(M, G):
    ids = _ids(M, G)
    flat = oracle.scale_layout("mxfp8", ids, "swizzled").ravel()
    Gp = -(-G // 4) * 4
    tiles_per_band = Gp // 4
    for t in range(flat.size // 512):
        band, tcol = divmod(t, tiles_per_band)        # tile-column fastest
        tile = flat[t * 512:(t + 1) * 512]
        for j in range(32):
            line = tile[j * 16:(j + 1) * 16]
            for k in range(4):                        # rows j, j+32, j+64, j+96 of the band
                r = band * 128 + j + 32 * k
                for c in range(4):                    # the row's 4 columns, contiguous
                    g = tcol * 4 + c
                    want = ids[r, g] if (r < M and g < G) else 0
                    assert line[4 * k + c] == want, (t, j, k, c)


def test_swizzled_keeps_dtype_and_values():
    rng = np.random.default_rng(0)
    s = rng.integers(0, 255, size=(130, 6), dtype=np.uint8)
    out = oracle.scale_layout("mxfp8", s, "swizzled")
    assert out.dtype == np.uint8
    assert np.array_equal(np.sort(out.ravel())[-s.size:], np.sort(s.ravel()))


@pytest.mark.parametrize("M,G", [(1, 1), (5, 32), (8, 3), (4097, 96)])
def test_col_major_is_the_padded_transpose(M, G):
    rng = np.random.default_rng(M)
    s = rng.standard_normal((M, G)).astype(np.float32)
    out = oracle.scale_layout("block128", s, "col_major")
    Mp = -(-M // 4) * 4
    assert out.shape == (G, Mp) and out.dtype == np.float32
    assert np.array_equal(out[:, :M], s.T)
    assert (out[:, M:] == 0).all()


def test_row_is_identity_and_wrong_format_is_refused():
    s = _ids(3, 5)
    assert np.array_equal(oracle.scale_layout("mxfp8", s, "row"), s)
    with pytest.raises(AssertionError):
        oracle.scale_layout("block128", s, "swizzled")
    with pytest.raises(AssertionError):
        oracle.scale_layout("mxfp8", s, "col_major")
