"""Device codecs against the oracle, exhaustively over fp32 inputs: the E2M1
round-to-nearest-even conversion (Blackwell cvt ... e2m1x2), the E4M3 (cvt ...
e4m3x2) and UE5M3 (software) block-scale encoders, the stochastic E2M1 rounder,
and the Philox4x32-10 draw stream. NaN inputs are excluded: the path never feeds
NaN to an encoder (non-finite data is flagged instead)."""
import concurrent.futures as cf
import multiprocessing as mp

import numpy as np
import pytest
import torch

import nvfp4_block_scaled_02_gb300 as nv
from helpers import assert_exact

pytestmark = pytest.mark.gpu

CHUNK = 1 << 26


def _oracle_chunk(args):
    op, lo, hi = args
    import numpy as _np
    import oracle as _o
    x = _np.arange(lo, hi, dtype=_np.uint64).astype(_np.uint32).view(_np.float32)
    if op == 0:
        return _o.e2m1_rne(x)
    return _o.scale_encode(op - 1, x)


@pytest.fixture(scope="module")
def pool():
    import oracle
    oracle.build()
    ctx = mp.get_context("spawn")
    with cf.ProcessPoolExecutor(max_workers=min(16, mp.cpu_count()), mp_context=ctx) as ex:
        yield ex


def _gpu_chunk(op, lo, hi):
    bits = torch.arange(lo, hi, dtype=torch.int64, device="cuda")
    x = (bits - (bits >= 2 ** 31).to(torch.int64) * 2 ** 32).to(torch.int32).view(torch.float32)
    return nv.nvfp4_codec_probe(op, x).cpu().numpy()


def _sweep(pool, op, lo, hi):
    tasks = [(op, a, min(a + CHUNK, hi)) for a in range(lo, hi, CHUNK)]
    for (o, a, b), ref in zip(tasks, pool.map(_oracle_chunk, tasks)):
        got = _gpu_chunk(o, a, b)
        x = np.arange(a, b, dtype=np.uint64).astype(np.uint32)
        keep = (x & 0x7FFFFFFF) <= 0x7F800000  # not NaN
        assert_exact(got[keep], ref[keep], f"op {o} on [{a:#x}, {b:#x})")


def test_e2m1_rne_all_fp32(pool):
    _sweep(pool, 0, 0, 1 << 32)


def test_e4m3_encoder_all_nonnegative_fp32(pool):
    _sweep(pool, 1, 0, 0x7F800001)


def test_ue5m3_encoder_all_nonnegative_fp32(pool):
    _sweep(pool, 2, 0, 0x7F800001)


def test_e2m1_pairs_pack_even_element_low():
    import oracle
    y = torch.tensor([0.5, 6.0, -1.0, 3.0], device="cuda")
    got = nv.nvfp4_codec_probe(0, y).cpu().numpy()
    assert list(got) == list(oracle.e2m1_rne(y.cpu().numpy()))


def test_stochastic_rounder_against_oracle():
    import oracle
    rng = np.random.default_rng(21)
    n = 1 << 22
    y = np.concatenate([
        rng.uniform(-7, 7, n).astype(np.float32),
        (rng.integers(0, 0x40E00000, n, dtype=np.uint32)).view(np.float32),  # [0, 7)
        np.repeat(np.array([0.25, 2.25, 5.0, 1.0, 0.0, -0.0, 6.0, 1e-30, 5.9999995], np.float32),
                  4096),
    ])
    v = rng.integers(0, 1 << 16, y.size, dtype=np.uint32)
    v[-9 * 4096:] = np.tile(np.arange(4096, dtype=np.uint32) * 16, 9)
    got = nv.nvfp4_codec_probe(3, torch.from_numpy(y).cuda(),
                               torch.from_numpy(v.view(np.int32)).cuda()).cpu().numpy()
    assert_exact(got, oracle.e2m1_sr(y, v), "stochastic E2M1")


def test_stochastic_rounder_exhaustive_over_bits_for_grid_cells():
    """Every 16-bit draw for values across each grid cell."""
    import oracle
    cells = np.array([0.1, 0.3, 0.75, 1.2, 1.74, 2.5, 3.3, 4.0, 4.5, 5.0, 5.99], np.float32)
    y = np.repeat(cells, 65536)
    v = np.tile(np.arange(65536, dtype=np.uint32), cells.size)
    got = nv.nvfp4_codec_probe(3, torch.from_numpy(y).cuda(),
                               torch.from_numpy(v.view(np.int32)).cuda()).cpu().numpy()
    assert_exact(got, oracle.e2m1_sr(y, v), "stochastic E2M1, all draws")


@pytest.mark.parametrize("seed,step,direction,idx0", [
    (0, 0, 0, 0), (1234, 7, 1, 8 * 12345 + 3), (0xFFFFFFFF, 31, 0, (1 << 35) + 5),
    (3, 16, 1, (1 << 40) - 100)])
def test_draw_stream_matches_oracle(seed, step, direction, idx0):
    import oracle
    n = 1 << 16
    got = nv.nvfp4_sr_bits(seed, step, direction, idx0, n).cpu().numpy().view(np.uint32)
    assert_exact(got, oracle.sr_bits(seed, step, direction, idx0, n), "random bits")
