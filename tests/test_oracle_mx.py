"""Pins of the oracle's MXFP8 quantisation of bf16 tensors (End-to-End 4-Bit
Training, quantised-linear-layer figure: bf16 gradients quantised to MXFP8
with stochastic rounding, rows and transposed): RNE codes against PyTorch's
float8_e4m3fn cast (library) at the exponent computed independently in
float64, the column encoding as the row encoding of the transpose,
unbiasedness of stochastic rounding over seeds, and independent row and
column draws."""
import math

import numpy as np
import torch

from nvfp4_block_scaled_02_gb300 import synth


def _exp64(amax: float) -> int:
    """Smallest e with amax <= 448 * 2^e, in float64 (clamped to [-127, 127])."""
    if amax == 0:
        return -127
    e = math.ceil(math.log2(amax / 448.0))
    while amax > 448.0 * 2.0 ** e:
        e += 1
    while e > -127 and amax <= 448.0 * 2.0 ** (e - 1):
        e -= 1
    return max(-127, min(127, e))


def test_rne_codes_are_the_float8_cast_at_the_shared_exponent(orc):
    xb = synth.student_t(16, 256, seed=3).reshape(1, 16, 256)
    out = orc.mx_quantize(xb, blocks=1, rounding=0)
    assert out["status"] == 0
    x = synth.bf16_bits_to_f32(xb[0]).astype(np.float64)
    for r in range(16):
        for b in range(8):
            blk = x[r, 32 * b:32 * b + 32]
            e = _exp64(float(np.abs(blk).max()))
            assert out["row_scales"][0, r, b] == e + 127
            y = torch.from_numpy((blk * 2.0 ** -e).astype(np.float32))
            want = y.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            assert np.array_equal(out["row_codes"][0, r, 32 * b:32 * b + 32], want), (r, b)


def test_column_encoding_is_the_row_encoding_of_the_transpose(orc):
    xb = synth.outlier_normal(64, 96, seed=4).reshape(1, 64, 96)
    col = orc.mx_quantize(xb, blocks=2, rounding=0)
    row_t = orc.mx_quantize(np.ascontiguousarray(xb[0].T)[None], blocks=1, rounding=0)
    assert np.array_equal(col["col_codes"], row_t["row_codes"])
    assert np.array_equal(col["col_scales"], row_t["row_scales"])


def test_stochastic_rounding_is_unbiased(orc):
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((1, 32, 64)) * 0.01).astype(np.float32)
    xb = orc.f32_to_bf16(x)
    xf = synth.bf16_bits_to_f32(xb).astype(np.float64)
    acc = np.zeros_like(xf)
    n = 400
    for seed in range(n):
        q = orc.mx_quantize(xb, blocks=1, rounding=1, seed=seed)
        e = q["row_scales"][0].astype(np.int64) - 127
        v = orc.e4m3_signed_value(q["row_codes"][0]).astype(np.float64)
        acc += v * np.ldexp(1.0, np.repeat(e, 32, axis=1))[None]
    mean = acc / n
    # each draw is one of the value's two grid neighbours, a grid step apart:
    # 1/8 of the value's binade, or 2^(e-9) in the subnormal range of its
    # block, so |mean - x| <= 6 sigma of a step/2 draw
    e = orc.mx_quantize(xb, blocks=1, rounding=0)["row_scales"][0].astype(np.int64) - 127
    sub = np.ldexp(1.0, np.repeat(e, 32, axis=1) - 9)[None]
    step = np.maximum(np.ldexp(1.0, np.floor(np.log2(np.abs(xf) + 1e-30)).astype(int) - 3), sub)
    assert np.all(np.abs(mean - xf) <= 6 * step / (2 * np.sqrt(n)) + 1e-12)


def test_row_and_column_draws_are_independent(orc):
    rng = np.random.default_rng(6)
    a = rng.standard_normal((32, 32)).astype(np.float32)
    xb = orc.f32_to_bf16(a + a.T)[None]  # symmetric: both encodings see the same values
    out = orc.mx_quantize(xb, blocks=3, rounding=1, seed=2)
    assert np.array_equal(out["row_scales"], out["col_scales"])
    assert not np.array_equal(out["row_codes"], out["col_codes"])
