"""Pins of the oracle's status word: every entry point reports a NaN or Inf
in any of its inputs (the non-finite-input bit the C ABI header defines), at
any position of a block, and stays clear on finite inputs. The CUDA path is
compared with these bits in the GPU tests."""
import numpy as np
import pytest

NAN, INF, NINF = 0x7FC0, 0x7F80, 0xFF80  # bf16 patterns


def _x(orc, seed, shape=(4, 64)):
    rng = np.random.default_rng(seed)
    return orc.f32_to_bf16((rng.standard_normal(shape) * 0.1).astype(np.float32))


def _planted(orc, seed, pos, bits, shape=(4, 64)):
    x = _x(orc, seed, shape)
    x.reshape(-1)[pos] = bits
    return x


POSITIONS = [0, 7, 8, 15, 17, 255]  # first, even/odd halves of a block, last


@pytest.mark.parametrize("pos", POSITIONS)
@pytest.mark.parametrize("bits", [NAN, INF, NINF])
def test_every_entry_point_flags_a_nonfinite_input(orc, pos, bits):
    bad = _planted(orc, 1, pos, bits)
    ok = _x(orc, 1)
    s = np.full((4, 4), 0.05, np.float32)
    gam = np.array([1.0], np.float32)
    flag = orc.ST_NONFINITE_INPUT
    cases = {
        "amax": lambda x: orc.global_amax(x)[1],
        "quantize": lambda x: orc.quantize(x, gam)["status"],
        "tile16": lambda x: orc.quantize_tile16(np.tile(x, (4, 1)).reshape(1, 16, 64), gam)["status"],
        "mx": lambda x: orc.mx_quantize(np.tile(x, (8, 1)).reshape(1, 32, 64), blocks=3)["status"],
        "fakequant": lambda x: orc.fakequant_fwd(x, s)[1],
        "fakequant_fp8": lambda x: orc.fakequant_fwd_fp8(x, s, None, 1.0)[1],
        "scale_grad (x)": lambda x: orc.scale_grad_bwd(x, ok, s, s)["status"],
        "scale_grad (dL/dx~)": lambda x: orc.scale_grad_bwd(ok, x, s, s)["status"],
        "mse sweep": lambda x: orc.scale_init_mse(x, 1.0)["status"],
        "export": lambda x: orc.export_scales(x, s, s, 1.0)["status"],
    }
    for name, f in cases.items():
        assert f(bad) & flag, name
        assert not f(ok) & flag, name


def test_dequant_flags_values_that_overflow(orc):
    """De-quantisation reports q * d that is not finite: code 6 at the largest
    scale (448) of a 4/6 encoding (g = gamax / (6 * 256)) with gamax 3e38
    gives 6 * 448 * 1.95e35 > FLT_MAX."""
    codes = np.full((1, 2, 8), 0x77, np.uint8)  # 6.0 in both nibbles
    scales = np.full((1, 2, 1), 0x7E, np.uint8)  # E4M3 448
    _, st = orc.dequant(codes, scales, np.array([3.0e38], np.float32), four_over_six=1)
    assert st & orc.ST_NONFINITE_INPUT
    _, st = orc.dequant(codes, scales, np.array([1.0], np.float32), four_over_six=1)
    assert st == 0
