"""CUDA re-quantisation (End-to-End 4-Bit Training, "Re-quantization with
stochastic rounding") against the oracle, element by element: the MXFP8 codecs
exhaustively (signed E4M3 RNE over every fp32 with |y| < 512, the shared
exponent over every non-negative finite fp32, the stochastic E4M3 rounder over
every 16-bit draw for values in each kind of grid cell), then the whole
de-quantise -> transpose -> re-quantise path for both targets, every rounding,
source and target format and 4/6 mode, on shapes spanning several tiles with
ragged tails, edge cases (zero blocks, saturated source scales, overflowing
outer scale, bad amax), and at the full activation size on sampled columns."""
import concurrent.futures as cf
import multiprocessing as mp

import numpy as np
import pytest
import torch

import nvfp4_block_scaled_02_gb300 as nv
import oracle
from helpers import assert_exact, host_u8, host_u32
from nvfp4_block_scaled_02_gb300 import synth

pytestmark = pytest.mark.gpu

CHUNK = 1 << 26


def _oracle_chunk(args):
    op, lo, hi = args
    import numpy as _np
    import oracle as _o
    x = _np.arange(lo, hi, dtype=_np.uint64).astype(_np.uint32).view(_np.float32)
    return _o.e4m3_rne(x) if op == 4 else _o.mx_shared_exp_bytes(x)


@pytest.fixture(scope="module")
def pool():
    oracle.build()
    ctx = mp.get_context("spawn")
    with cf.ProcessPoolExecutor(max_workers=min(16, mp.cpu_count()), mp_context=ctx) as ex:
        yield ex


def _gpu_chunk(op, lo, hi):
    bits = torch.arange(lo, hi, dtype=torch.int64, device="cuda")
    x = (bits - (bits >= 2 ** 31).to(torch.int64) * 2 ** 32).to(torch.int32).view(torch.float32)
    return nv.nvfp4_codec_probe(op, x).cpu().numpy()


def _sweep(pool, op, ranges):
    tasks = [(op, a, min(a + CHUNK, hi)) for lo, hi in ranges for a in range(lo, hi, CHUNK)]
    for (o, a, b), ref in zip(tasks, pool.map(_oracle_chunk, tasks)):
        assert_exact(_gpu_chunk(o, a, b), ref, f"op {o} on [{a:#x}, {b:#x})")


def test_e4m3_element_rne_all_fp32_below_512(pool):
    """Signed E4M3 RNE (cvt ... e4m3x2 satfinite) for every fp32 with |y| < 512,
    both signs: the MX path feeds |y| <= 448 only; 448..512 checks saturation."""
    _sweep(pool, 4, [(0, 0x44000000), (0x80000000, 0xC4000000)])


def test_e4m3_element_rne_saturates_and_keeps_signed_zero():
    y = torch.tensor([448.0, 464.0, 1e30, float("inf"), -float("inf"), -0.0, -1e-9, 0.0],
                     device="cuda")
    got = nv.nvfp4_codec_probe(4, y).cpu().numpy()
    assert list(got) == list(oracle.e4m3_rne(y.cpu().numpy()))


def test_mx_shared_exponent_all_nonnegative_finite_fp32(pool):
    _sweep(pool, 6, [(0, 0x7F800000)])


def test_e4m3_stochastic_rounder_against_oracle():
    rng = np.random.default_rng(31)
    n = 1 << 22
    y = np.concatenate([
        rng.uniform(-448, 448, n).astype(np.float32),
        (rng.integers(0, 0x43E00001, n, dtype=np.uint32)).view(np.float32),   # [0, 448]
        -(rng.integers(0, 0x3C800000, n, dtype=np.uint32)).view(np.float32),  # subnormal range
        np.array([0.0, -0.0, 448.0, -448.0, 500.0, 2.0 ** -6, 2.0 ** -9, 2.0 ** -10], np.float32),
    ])
    v = rng.integers(0, 1 << 16, y.size, dtype=np.uint32)
    got = nv.nvfp4_codec_probe(5, torch.from_numpy(y).cuda(),
                               torch.from_numpy(v.view(np.int32)).cuda()).cpu().numpy()
    assert_exact(got, oracle.e4m3_sr(y, v), "stochastic E4M3")


def test_e4m3_stochastic_rounder_exhaustive_over_draws():
    """Every 16-bit draw for values in subnormal cells, at the subnormal/normal
    boundary, inside low, middle and top binades and just below 448."""
    cells = np.array([2.0 ** -11, 3.3 * 2.0 ** -9, 0.0154, 2.0 ** -6 * 1.01, 0.07, 1.3, 2.9,
                      17.0, 100.1, 300.0, 447.9, -5.5, -0.002], np.float32)
    y = np.repeat(cells, 65536)
    v = np.tile(np.arange(65536, dtype=np.uint32), cells.size)
    got = nv.nvfp4_codec_probe(5, torch.from_numpy(y).cuda(),
                               torch.from_numpy(v.view(np.int32)).cuda()).cpu().numpy()
    assert_exact(got, oracle.e4m3_sr(y, v), "stochastic E4M3, all draws")


def test_e4m3_stochastic_rounder_kernel_form_exhaustive_over_draws():
    """The unsaturated form the kernels run: every 16-bit draw for values in
    subnormal cells (fp32 subnormals included), at the subnormal/normal
    boundary (where the stand-in pattern hands over to the value's own) and
    across the normal binades, zeros of both signs included."""
    cells = np.array([0.0, -0.0, 1e-45, -3e-41, 2.0 ** -40, 2.0 ** -11, 3.3 * 2.0 ** -9, 0.0154,
                      2.0 ** -6 * (1 - 2.0 ** -24), 2.0 ** -6, 2.0 ** -6 * 1.01, -0.0173,
                      2.0 ** -5 * (1 - 2.0 ** -20), 2.0 ** -5, 0.07, 1.3, 2.9, 17.0, 100.1, 300.0,
                      447.9, 448.0, -5.5, -447.0], np.float32)
    y = np.repeat(cells, 65536)
    v = np.tile(np.arange(65536, dtype=np.uint32), cells.size)
    got = nv.nvfp4_codec_probe(7, torch.from_numpy(y).cuda(),
                               torch.from_numpy(v.view(np.int32)).cuda()).cpu().numpy()
    assert_exact(got, oracle.e4m3_sr(y, v), "stochastic E4M3 (kernel form), all draws")


def test_e4m3_stochastic_rounder_kernel_form_random():
    rng = np.random.default_rng(33)
    n = 1 << 22
    mag = (rng.integers(0, 0x43E00001, n, dtype=np.uint32)).view(np.float32)  # [0, 448]
    y = np.where(rng.integers(0, 2, n) == 1, -mag, mag).astype(np.float32)
    y[::97] = 0.0
    v = rng.integers(0, 1 << 16, y.size, dtype=np.uint32)
    got = nv.nvfp4_codec_probe(7, torch.from_numpy(y).cuda(),
                               torch.from_numpy(v.view(np.int32)).cuda()).cpu().numpy()
    assert_exact(got, oracle.e4m3_sr(y, v), "stochastic E4M3 (kernel form)")


def test_tiny_values_land_in_the_e4m3_subnormal_range():
    """Source blocks whose scale is 2^-16 of the others put values in the E4M3
    2^-9-spaced range of their MX blocks (the rounder's stand-in pattern)."""
    codes, scales, gam = _source((1, 64, 128), seed=30)
    scales = scales.copy()
    scales[0, ::5, ::3] = 0x01  # the smallest E4M3 scale: these values land below 2^-6
    r = oracle.requant(codes, scales, gam, target=0, rounding=1, seed=3)
    vals = np.abs(oracle.e4m3_signed_value(r["codes"]))
    assert ((vals > 0) & (vals < 2.0 ** -6)).any()
    run_both(codes, scales, gam, target=0, rounding=1, seed=3)


# ------------------------------------------------------------ whole path --

def _source(shape, *, fmt=0, fos=0, seed=0, dist="t3", stale=1.0):
    """A forward row encoding written by the oracle: codes, scales, gamax."""
    S, R, Cc = shape
    if dist == "t3":
        xb = synth.student_t(S * R, Cc, seed=seed).reshape(shape)
    else:
        xb = synth.outlier_normal(S * R, Cc, seed=seed).reshape(shape)
    gam, _ = oracle.global_amax(xb, S)
    gam = (gam * np.float32(stale)).astype(np.float32)
    q = oracle.quantize(xb, gam, scale_fmt=fmt, four_over_six=fos, dequant=False)
    return q["row_codes"], q["row_scales"], gam


def _random_source(shape, seed):
    """Arbitrary code and scale bytes (every nibble, negative zeros included)."""
    S, R, Cc = shape
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 256, (S, R, Cc // 2), dtype=np.uint8)
    scales = rng.integers(0, 256, (S, R, Cc // 16), dtype=np.uint8)
    scales[..., ::7] = 0  # some all-zero blocks
    gam = rng.uniform(0.5, 40.0, S).astype(np.float32)
    return codes, scales, gam


def run_both(codes, scales, gam, *, target, rounding=1, seed=5, step=3, src_fmt=0, src_fos=0,
             src_scale_max=0.0, dst_fmt=0, dst_fos=0, dst_rule=0, dst_scale_max=0.0,
             check=True):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    src = nv.Config(scale_fmt=src_fmt, four_over_six=src_fos, scale_max=src_scale_max)
    dst = nv.Config(scale_fmt=dst_fmt, rounding=rounding, four_over_six=dst_fos,
                    four_over_six_rule=dst_rule, scale_max=dst_scale_max, seed=seed, step=step)
    out = nv.nvfp4_requant_transpose(torch.from_numpy(codes).cuda(),
                                     torch.from_numpy(scales).cuda(),
                                     torch.from_numpy(gam).cuda(), src, dst, target, status=st)
    torch.cuda.synchronize()
    ref = oracle.requant(codes, scales, gam, target=target, rounding=rounding, seed=seed,
                         step=step, src_fmt=src_fmt, src_scale_max=src_scale_max,
                         src_fos=src_fos, dst_fmt=dst_fmt, dst_fos=dst_fos, dst_rule=dst_rule,
                         dst_scale_max=dst_scale_max)
    if check:
        what = f"target={target} sr={rounding} src=({src_fmt},{src_fos}) dst=({dst_fmt},{dst_fos})"
        assert int(st.item()) == ref["status"], what
        assert_exact(host_u8(out["codes"]), ref["codes"], what + " codes")
        assert_exact(host_u8(out["scales"]), ref["scales"], what + " scales")
        if target == nv.TARGET_NVFP4 and dst_fos:
            assert_exact(host_u32(out["choice"]), ref["choice"], what + " 4/6 bits")
    return out, ref, int(st.item())


MX_SHAPES = [(1, 64, 128), (2, 96, 144), (1, 32, 16), (3, 160, 400), (1, 256, 1024)]
NV_SHAPES = [(1, 48, 80), (2, 80, 272), (1, 16, 16), (2, 208, 400), (1, 512, 512)]


@pytest.mark.parametrize("rounding", [0, 1])
@pytest.mark.parametrize("src_fmt,src_fos", [(0, 0), (0, 1), (1, 1)])
@pytest.mark.parametrize("shape", MX_SHAPES)
def test_mxfp8_target(shape, src_fmt, src_fos, rounding):
    codes, scales, gam = _source(shape, fmt=src_fmt, fos=src_fos, seed=sum(shape))
    run_both(codes, scales, gam, target=0, rounding=rounding, src_fmt=src_fmt, src_fos=src_fos,
             seed=17, step=2)


@pytest.mark.parametrize("rounding", [0, 1])
@pytest.mark.parametrize("dst_fmt", [0, 1])
@pytest.mark.parametrize("dst_fos", [0, 1])
@pytest.mark.parametrize("shape", NV_SHAPES)
def test_nvfp4_target(shape, dst_fmt, dst_fos, rounding):
    codes, scales, gam = _source(shape, fos=1, seed=3 + sum(shape))
    run_both(codes, scales, gam, target=1, rounding=rounding, src_fos=1, dst_fmt=dst_fmt,
             dst_fos=dst_fos, seed=9, step=1)


@pytest.mark.parametrize("rule", [nv.FOS_MAE, nv.FOS_MAX])
@pytest.mark.parametrize("rounding", [0, 1])
def test_nvfp4_target_alternative_four_over_six_rules(rule, rounding):
    codes, scales, gam = _source((2, 80, 272), fos=1, seed=12)
    run_both(codes, scales, gam, target=1, rounding=rounding, src_fos=1, dst_fos=1,
             dst_rule=rule)


@pytest.mark.parametrize("target", [0, 1])
@pytest.mark.parametrize("src_fmt", [0, 1])
def test_arbitrary_source_bytes(target, src_fmt):
    codes, scales, gam = _random_source((2, 96, 400), seed=40 + src_fmt)
    run_both(codes, scales, gam, target=target, src_fmt=src_fmt, dst_fos=target)


@pytest.mark.parametrize("target", [0, 1])
def test_explicit_scale_maxima(target):
    codes, scales, gam = _source((1, 64, 256), fos=0, seed=8)
    run_both(codes, scales, gam, target=target, src_scale_max=300.0, dst_scale_max=200.0,
             dst_fos=target)


@pytest.mark.parametrize("target", [0, 1])
def test_stale_amax_saturated_source_scales(target):
    """A periodic (stale) amax 8x too small saturates source block scales."""
    codes, scales, gam = _source((1, 96, 272), seed=21, stale=0.125)
    assert (scales == 0x7E).any()
    run_both(codes, scales, gam, target=target, dst_fos=target)


@pytest.mark.parametrize("target", [0, 1])
def test_all_zero_tensor(target):
    shape = (2, 64, 160)
    codes = np.zeros((2, 64, 80), np.uint8)
    scales = np.zeros((2, 64, 10), np.uint8)
    gam = np.zeros(2, np.float32)
    out, ref, st = run_both(codes, scales, gam, target=target, dst_fos=target)
    assert st == 0 and not ref["codes"].any()
    if target == 0:
        assert (ref["scales"] == 0).all()  # e = -127


def test_step_and_seed_change_the_draws():
    codes, scales, gam = _source((1, 64, 128), seed=2)
    a, _, _ = run_both(codes, scales, gam, target=0, seed=1, step=0)
    b, _, _ = run_both(codes, scales, gam, target=0, seed=1, step=1)
    assert (host_u8(a["codes"]) != host_u8(b["codes"])).any()


@pytest.mark.parametrize("target", [0, 1])
def test_bad_amax_is_flagged(target):
    codes, scales, gam = _source((2, 64, 128), seed=4)
    gam[1] = np.float32("nan")
    _, ref, st = run_both(codes, scales, gam, target=target, check=False)
    assert st & nv.DEV_BAD_AMAX and ref["status"] & oracle.ST_BAD_AMAX


@pytest.mark.parametrize("target", [0, 1])
def test_overflowing_dequant_is_flagged(target):
    """g near FLT_MAX / (6 M) with UE5M3 scales: q * d overflows fp32."""
    codes, scales, _ = _random_source((1, 64, 128), seed=6)
    gam = np.array([3.0e38], np.float32)
    _, ref, st = run_both(codes, scales, gam, target=target, src_fmt=1, check=False)
    assert st & nv.DEV_NONFINITE_INPUT and ref["status"] & oracle.ST_NONFINITE_INPUT


# ------------------------------------------------- full activation size --

@pytest.fixture(scope="module")
def activation_source():
    """The activation tensor 8192 x 4096 (0.5 * Student-t(3)), forward-encoded
    by the oracle with 4/6 and E4M3 scales, as the benchmark re-quantises it."""
    return _source((1, 8192, 4096), fos=1, seed=1)


def test_full_size_mxfp8_sampled_columns(activation_source):
    """Stochastic MXFP8 at 8192 x 4096 in the benchmark's launch configuration;
    96 sampled output rows (input columns) re-encoded one by one by the oracle
    from its de-quantised values, with their own flat indices."""
    codes, scales, gam = activation_source
    R, Cc = 8192, 4096
    seed, step = 123, 45
    out = nv.nvfp4_requant_transpose(torch.from_numpy(codes).cuda(),
                                     torch.from_numpy(scales).cuda(),
                                     torch.from_numpy(gam).cuda(), nv.Config(four_over_six=1),
                                     nv.Config(rounding=1, seed=seed, step=step), 0)
    got_c, got_s = host_u8(out["codes"])[0], host_u8(out["scales"])[0]
    xh, st = oracle.dequant(codes, scales, gam, four_over_six=1)
    assert st == 0
    cols = np.random.default_rng(9).choice(Cc, 96, replace=False)
    cols[:2] = (0, Cc - 1)
    for c in cols:
        wc, ws = oracle.mx_encode(xh[0, :, c], rounding=1, seed=seed, step=step, direction=2,
                                  idx0=int(c) * R)
        assert_exact(got_c[c], wc, f"column {c} codes")
        assert_exact(got_s[c], ws, f"column {c} scales")


def test_full_size_nvfp4_target(activation_source):
    codes, scales, gam = activation_source
    run_both(codes, scales, gam, target=1, rounding=1, src_fos=1, dst_fos=1, seed=77, step=6)
