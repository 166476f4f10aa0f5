"""Pins of how the oracle lays out its outputs and keys its random draws: the
4/6 bitmap's bit order, and the direction and flat index behind every
stochastic draw (rows 0, columns 1, re-quantisation 2, each at its output
layout's flat index). These are the library's own conventions, stated in its
C ABI header; each whole-tensor entry point is checked against the
block-level functions (themselves pinned against the pages' examples, exact
probabilities and brute force) applied one block at a time with those
conventions, so a wrong direction, index, bit order or outer scale in the
wiring fails here."""
import numpy as np
import pytest


def _bits(words, n):
    b = np.unpackbits(np.ascontiguousarray(words, np.uint32).view(np.uint8), bitorder="little")
    return b[:n]


def _pack(codes16):
    return (codes16[0::2] | (codes16[1::2] << 4)).astype(np.uint8)


def test_choice_bitmap_holds_block_b_in_bit_b_mod_32_of_word_b_div_32(orc):
    rng = np.random.default_rng(40)
    # 2 slices of 3 x 224: 42 blocks per slice, so words span rows and slices
    # end inside a word
    x = orc.f32_to_bf16((rng.standard_normal((2, 3, 224)) *
                         rng.uniform(0.1, 10, (2, 3, 1))).astype(np.float32))
    gam, _ = orc.global_amax(x, 2)
    q = orc.quantize(x, gam, four_over_six=1, dequant=False)
    xf = orc.bf16_to_f32(x).reshape(2, 42, 16)
    for s in range(2):
        g = orc.decode_scale(float(gam[s]), 256.0)
        want = np.array([orc.encode_block(xf[s, b], g, fos=1)["choice"] for b in range(42)])
        assert 0 < want.sum() < 42
        assert np.array_equal(_bits(q["row_choice"][s], 42), want)
        assert not np.any(_bits(q["row_choice"][s], 64)[42:])


def test_row_and_column_draws_use_directions_0_and_1_at_their_layout_index(orc):
    rng = np.random.default_rng(41)
    S, R, C = 2, 32, 48
    x = orc.f32_to_bf16(rng.standard_normal((S, R, C)).astype(np.float32))
    gam, _ = orc.global_amax(x, S)
    q = orc.quantize(x, gam, blocks=3, rounding=1, seed=11, step=4, dequant=False)
    xf = orc.bf16_to_f32(x)
    kw = dict(rounding=1, seed=11, step=4)
    for s in range(S):
        g = orc.decode_scale(float(gam[s]), 448.0)
        for r in (0, 17, R - 1):
            for cb in range(C // 16):
                b = orc.encode_block(xf[s, r, 16 * cb:16 * cb + 16], g, direction=0,
                                     idx0=(s * R + r) * C + 16 * cb, **kw)
                assert np.array_equal(q["row_codes"][s, r, 8 * cb:8 * cb + 8], _pack(b["codes"]))
                assert q["row_scales"][s, r, cb] == b["scale"]
        for c in (0, 29, C - 1):
            for rb in range(R // 16):
                b = orc.encode_block(np.ascontiguousarray(xf[s, 16 * rb:16 * rb + 16, c]), g,
                                     direction=1, idx0=(s * C + c) * R + 16 * rb, **kw)
                assert np.array_equal(q["col_codes"][s, c, 8 * rb:8 * rb + 8], _pack(b["codes"]))
                assert q["col_scales"][s, c, rb] == b["scale"]


def test_row_and_column_draws_differ_on_a_symmetric_matrix(orc):
    rng = np.random.default_rng(43)
    a = rng.standard_normal((32, 32)).astype(np.float32)
    xb = orc.f32_to_bf16(a + a.T)[None]  # both encodings see the same blocks
    gam, _ = orc.global_amax(xb)
    rne = orc.quantize(xb, gam, blocks=3, dequant=False)
    assert np.array_equal(rne["row_codes"], rne["col_codes"])
    sr = orc.quantize(xb, gam, blocks=3, rounding=1, seed=2, dequant=False)
    assert np.array_equal(sr["row_scales"], sr["col_scales"])
    assert not np.array_equal(sr["row_codes"], sr["col_codes"])


@pytest.mark.parametrize("target", [0, 1])
def test_requant_draws_use_direction_2_at_the_output_index(orc, target):
    rng = np.random.default_rng(42)
    S, R, C = 2, 32, 64
    x = orc.f32_to_bf16(rng.standard_normal((S, R, C)).astype(np.float32))
    gam, _ = orc.global_amax(x, S)
    fwd = orc.quantize(x, gam, four_over_six=1, dequant=False)
    xh, _ = orc.dequant(fwd["row_codes"], fwd["row_scales"], gam, four_over_six=1)
    r = orc.requant(fwd["row_codes"], fwd["row_scales"], gam, target=target, rounding=1,
                    seed=5, step=6, src_fos=1, dst_fos=int(target == 1))
    kw = dict(rounding=1, seed=5, step=6, direction=2)
    for s in range(S):
        xt = np.ascontiguousarray(xh[s].T)  # [C][R]
        g = orc.decode_scale(float(gam[s]), 256.0)  # a 4/6 target keeps M = 256
        for c in (0, 33, C - 1):
            if target == 0:
                codes, scales = orc.mx_encode(xt[c], idx0=(s * C + c) * R, **kw)
                assert np.array_equal(r["codes"][s, c], codes)
                assert np.array_equal(r["scales"][s, c], scales)
                continue
            for rb in range(R // 16):
                b = orc.encode_block(xt[c, 16 * rb:16 * rb + 16], g, fos=1,
                                     idx0=(s * C + c) * R + 16 * rb, **kw)
                assert np.array_equal(r["codes"][s, c, 8 * rb:8 * rb + 8], _pack(b["codes"]))
                assert r["scales"][s, c, rb] == b["scale"]
                bit = (c * (R // 16) + rb)
                assert _bits(r["choice"][s], bit + 1)[bit] == b["choice"]


def test_mx_draws_use_directions_0_and_1_at_their_layout_index(orc):
    rng = np.random.default_rng(44)
    R, C = 64, 96
    x = orc.f32_to_bf16(rng.standard_normal((1, R, C)).astype(np.float32))
    q = orc.mx_quantize(x, blocks=3, rounding=1, seed=8, step=9)
    xf = orc.bf16_to_f32(x)[0]
    for r in (0, 40, R - 1):
        codes, scales = orc.mx_encode(xf[r], rounding=1, seed=8, step=9, direction=0, idx0=r * C)
        assert np.array_equal(q["row_codes"][0, r], codes)
        assert np.array_equal(q["row_scales"][0, r], scales)
    for c in (0, 50, C - 1):
        codes, scales = orc.mx_encode(np.ascontiguousarray(xf[:, c]), rounding=1, seed=8, step=9,
                                      direction=1, idx0=c * R)
        assert np.array_equal(q["col_codes"][0, c], codes)
        assert np.array_equal(q["col_scales"][0, c], scales)
