"""Pins of the oracle's 16x16 tile scale (End-to-End 4-Bit Training,
"Block-scaled backward passes": one scale per 16x16 tile from its largest
value, identical when the tensor is transposed): the tile scale against the
1x16 encoder's scales (the block-scale code is monotone in the amax),
equality with 1x16 encoding when every row of a tile holds the tile maximum,
the transposed column encoding, and the pages' underflow figures."""
import numpy as np
import pytest

from nvfp4_block_scaled_02_gb300 import synth


def _x(shape, seed, scale=1.0):
    S, R, Cc = shape
    return synth.outlier_normal(S * R, Cc, seed=seed).reshape(shape)


@pytest.mark.parametrize("fmt", [0, 1])
def test_tile_scale_is_the_largest_row_block_scale(orc, fmt):
    xb = _x((2, 48, 64), seed=1)
    gam, _ = orc.global_amax(xb, 2)
    t = orc.quantize_tile16(xb, gam, scale_fmt=fmt)
    r = orc.quantize(xb, gam, scale_fmt=fmt, scale_max=448.0)
    assert t["status"] == r["status"] == 0
    rs = r["row_scales"].reshape(2, 3, 16, 4)        # [S][tile row][row in tile][tile col]
    want = rs.max(axis=2)                            # code monotone in the amax
    got = t["row_scales"].reshape(2, 3, 16, 4)
    assert np.all(got == want[:, :, None, :])


def test_equal_row_maxima_give_the_1x16_encoding(orc):
    """If every row block of a tile holds the tile's amax, both encodings agree."""
    rng = np.random.default_rng(2)
    x = rng.uniform(-1, 1, (1, 32, 32)).astype(np.float32)
    x[:, :, 0] = 3.0  # the tile maximum in every 1x16 row block (column 0 and 16)
    x[:, :, 16] = -3.0
    xb = orc.f32_to_bf16(x)
    gam, _ = orc.global_amax(xb)
    for rounding in (0, 1):
        t = orc.quantize_tile16(xb, gam, rounding=rounding, seed=4)
        r = orc.quantize(xb, gam, rounding=rounding, seed=4, scale_max=448.0)
        for k in ("row_codes", "row_scales", "row_dq"):
            assert np.array_equal(t[k], r[k]), (rounding, k)


def test_column_encoding_is_the_transposed_row_encoding(orc):
    xb = _x((2, 32, 48), seed=3)
    gam, _ = orc.global_amax(xb, 2)
    t = orc.quantize_tile16(xb, gam, rounding=1, seed=9, step=2)

    def nibbles(codes, R, Cc):
        c = codes.reshape(-1, R, Cc // 2)
        return np.stack([c & 15, c >> 4], axis=-1).reshape(-1, R, Cc)

    rn = nibbles(t["row_codes"], 32, 48)
    cn = nibbles(t["col_codes"], 48, 32)
    assert np.array_equal(cn, rn.transpose(0, 2, 1))
    assert np.array_equal(t["col_dq"], t["row_dq"].transpose(0, 2, 1))
    rs = np.repeat(t["row_scales"], 16, axis=2)      # per element [S][R][C]
    cs = np.repeat(t["col_scales"], 16, axis=2)      # per element [S][C][R]
    assert np.array_equal(cs, rs.transpose(0, 2, 1))


def test_outlier_tile_loses_more_values_than_1x16(orc):
    """The pages' tile with one large outlier: a separate 1x16 scale per row
    group keeps more small values than one 16x16 scale."""
    rng = np.random.default_rng(5)
    x = (rng.uniform(0.5, 1.5, (1, 16, 16)) * rng.choice([-1, 1], (1, 16, 16))).astype(np.float32)
    x[0, 7, 9] = 300.0
    xb = orc.f32_to_bf16(x)
    gam, _ = orc.global_amax(xb)
    t = orc.quantize_tile16(xb, gam)
    r = orc.quantize(xb, gam, scale_max=448.0)

    def nonzero(codes):
        c = codes.reshape(-1)
        return int(np.count_nonzero(c & 7) + np.count_nonzero((c >> 4) & 7))

    n_tile, n_row = nonzero(t["row_codes"]), nonzero(r["row_codes"])
    assert n_row >= 240 and n_tile < n_row  # only the outlier's row group collapses with 1x16


def test_large_row_of_values_survives_only_with_row_groups(orc):
    """The pages' tile with a full row of large values: 1x16 keeps all 256,
    16x1 column blocks and the 16x16 tile flush most small values to zero."""
    rng = np.random.default_rng(6)
    x = rng.uniform(0.5, 1.0, (1, 16, 16)).astype(np.float32)
    x[0, 3, :] = rng.uniform(400, 500, 16)
    xb = orc.f32_to_bf16(x)
    gam, _ = orc.global_amax(xb)
    r = orc.quantize(xb, gam, blocks=3, scale_max=448.0)
    t = orc.quantize_tile16(xb, gam)

    def nonzero(codes):
        c = codes.reshape(-1)
        return int(np.count_nonzero(c & 7) + np.count_nonzero((c >> 4) & 7))

    assert nonzero(r["row_codes"]) == 256
    assert nonzero(r["col_codes"]) < 128 and nonzero(t["row_codes"]) < 128
