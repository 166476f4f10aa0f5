"""Parity at the benchmark's full sizes, in the configurations bench.py times:
the whole tensor goes through the CUDA path in one call, and sampled rows,
blocks or experts are checked against the oracle. Blocks are independent
given their slice's global amax, so the oracle can encode a sample of rows on
its own; stochastic rounding draws its bits from the flat index, so sampled
stochastic blocks are re-encoded one by one at their own indices."""
import numpy as np
import pytest
import torch

import nvfp4_block_scaled_02_gb300 as nv
import oracle
from helpers import assert_close_bf16, assert_close_f32, assert_exact, dev_bits, host_u16, host_u8
from nvfp4_block_scaled_02_gb300 import synth

pytestmark = pytest.mark.gpu


def _rows(n, k, seed):
    r = np.random.default_rng(seed).choice(n, k, replace=False)
    r[:2] = (0, n - 1)
    return np.sort(r)


def test_activation_8192x4096_amax_and_row_four_over_six():
    """The default workload: per-tensor amax, then 1x16 row blocks with E4M3
    scales, RNE, Four-Over-Six and the dequantised output."""
    R, Cc = 8192, 4096
    xb = synth.student_t(R, Cc, seed=1)
    x = dev_bits(xb)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    amax = nv.nvfp4_amax(x, status=st)
    out = nv.nvfp4_quantize(x, amax, nv.Config(four_over_six=1), status=st)["row"]
    ref_amax, _ = oracle.global_amax(xb)
    assert_exact(amax.cpu().numpy().view(np.uint32), ref_amax.view(np.uint32), "amax")
    rows = _rows(R, 24, 1)
    ref = oracle.quantize(xb[rows], ref_amax, four_over_six=1)
    assert int(st.item()) == ref["status"] == 0
    assert_exact(host_u8(out["codes"]).reshape(R, Cc // 2)[rows], ref["row_codes"], "codes")
    assert_exact(host_u8(out["scales"]).reshape(R, Cc // 16)[rows], ref["row_scales"], "scales")
    words = Cc // 16 // 32  # 4/6 bitmap words per row
    choice = out["choice"].cpu().numpy().view(np.uint32).reshape(R, words)[rows]
    assert_exact(choice, ref["row_choice"], "4/6 choices")
    assert_close_bf16(host_u16(out["dequant"]).reshape(R, Cc)[rows], ref["row_dq"], "dequant")


def test_gradient_16384x4096_stochastic_ue5m3_stale_amax():
    """The gradient workload on a refresh-free step: step 5 of the drifting
    stream quantised with step 0's amax (periodic scaling), UE5M3 scales,
    stochastic rounding keyed on (seed 3, step 5); sampled blocks re-encoded
    at their flat indices."""
    R, Cc, t = 16384, 4096, 5
    gen = synth.DriftingGradient(R, Cc, seed=3)
    x0 = dev_bits(gen.step(0))
    stale = nv.nvfp4_amax(x0)
    del x0
    xb = gen.step(t)
    cfg = nv.Config(scale_fmt=1, rounding=1, scale_max=448.0, seed=3, step=t)
    out = nv.nvfp4_quantize(dev_bits(xb), stale, cfg, dequant=False)["row"]
    codes = host_u8(out["codes"]).reshape(-1, 8)
    scales = host_u8(out["scales"]).reshape(-1)
    g = oracle.decode_scale(float(stale.item()), 448.0)
    xf = synth.bf16_bits_to_f32(xb).reshape(-1, 16)
    blocks = np.concatenate([[0, 1, xf.shape[0] - 1],
                             np.random.default_rng(7).choice(xf.shape[0], 3000, replace=False)])
    for b in blocks:
        r = oracle.encode_block(xf[b], g, fmt=1, rounding=1, seed=3, step=t, direction=0,
                                idx0=int(b) * 16)
        want = (r["codes"][0::2] | (r["codes"][1::2] << 4)).astype(np.uint8)
        assert_exact(codes[b], want, f"codes of block {b}")
        assert int(scales[b]) == r["scale"], f"scale of block {b}"


def test_scale_learning_14336x4096_forward_and_backward():
    """The scale-learning step: fake-quant forward and STE backward with dual
    scales (equal at initialisation, as benchmarked), dL/dx written; sampled
    rows against the oracle."""
    R, Cc = 14336, 4096
    wb, gb, s = synth.scale_learning(R, Cc, seed=2)
    w, g, sp = dev_bits(wb), dev_bits(gb), torch.from_numpy(s).cuda()
    so = sp.clone()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    xq = nv.nvfp4_fakequant_fwd(w, sp, so, status=st)
    res = nv.nvfp4_scale_grad_bwd(w, g, sp, so, status=st)
    assert int(st.item()) == 0
    rows = _rows(R, 16, 2)
    want_q, wst = oracle.fakequant_fwd(wb[rows], s[rows], s[rows])
    assert wst == 0
    assert_close_bf16(host_u16(xq).reshape(R, Cc)[rows], want_q, "x~")
    want = oracle.scale_grad_bwd(wb[rows], gb[rows], s[rows], s[rows])
    assert_close_f32(res["gs_pre"].cpu().numpy()[rows], want["gs_pre"], "dL/ds_pre")
    assert_close_f32(res["gs_post"].cpu().numpy()[rows], want["gs_post"], "dL/ds_post")
    assert_close_bf16(host_u16(res["gx"]).reshape(R, Cc)[rows], want["gx"], "dL/dx")


def test_moe_64x2048x7168_dual_four_over_six_sampled_experts():
    """The MoE workload: per-expert amax for all 64 experts, then both
    encodings (rows and the transpose) with 4/6 and both dequants in one
    launch; three experts compared whole with the oracle."""
    E, R, Cc = 64, 2048, 7168
    xb = synth.moe_experts(E, R, Cc, seed=4)
    x = dev_bits(xb)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    amax = nv.nvfp4_amax(x, status=st)
    out = nv.nvfp4_quantize(x, amax, nv.Config(blocks=3, four_over_six=1), status=st)
    assert int(st.item()) == 0
    ref_amax, _ = oracle.global_amax(xb, E)
    assert_exact(amax.cpu().numpy().view(np.uint32), ref_amax.view(np.uint32), "amaxes")
    for e in (0, 37, E - 1):
        ref = oracle.quantize(xb[e:e + 1], ref_amax[e:e + 1], blocks=3, four_over_six=1)
        for side in ("row", "col"):
            o = out[side]
            assert_exact(host_u8(o["codes"][e]), ref[side + "_codes"], f"{side} codes, expert {e}")
            assert_exact(host_u8(o["scales"][e]), ref[side + "_scales"], f"{side} scales, expert {e}")
            assert_exact(o["choice"][e].cpu().numpy().view(np.uint32), ref[side + "_choice"],
                         f"{side} 4/6 choices, expert {e}")
            assert_close_bf16(host_u16(o["dequant"][e]), ref[side + "_dq"],
                              f"{side} dequant, expert {e}")


def _bits(words, start, n):
    """Bits start .. start + n - 1 of a little-endian 4/6 choice bitmap."""
    b = np.unpackbits(np.ascontiguousarray(words).view(np.uint8), bitorder="little")
    return b[start:start + n]


def test_more_than_two_to_the_31_elements():
    """524304 x 4096 values (2^31 + 65536): 64-bit index arithmetic in amax and
    the dual encoding (rows and columns, 4/6), checked on the rows past index
    2^31 and on sampled columns (each the row encoding of a 524304-value
    column). The input is generated on the device in seeded chunks."""
    R, Cc = (1 << 19) + 16, 4096
    x = torch.empty((R, Cc), dtype=torch.bfloat16, device="cuda")
    gen = torch.Generator(device="cuda").manual_seed(31)
    step = 1 << 16
    for a in range(0, R, step):
        b = min(R, a + step)
        x[a:b] = torch.randn((b - a, Cc), generator=gen, device="cuda").to(torch.bfloat16)
    x[R - 3, 7] = 9.5  # the tensor's amax sits past index 2^31
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    amax = nv.nvfp4_amax(x, status=st)
    assert float(amax.item()) == float(x.abs().max().item()) == 9.5
    out = nv.nvfp4_quantize(x, amax, nv.Config(blocks=3, four_over_six=1), status=st,
                            dequant=False)
    assert int(st.item()) == 0
    gam = amax.cpu().numpy()
    ref = oracle.quantize(host_u16(x[R - 16:]), gam, four_over_six=1, dequant=False)
    row = out["row"]
    assert_exact(host_u8(row["codes"][0, R - 16:]), ref["row_codes"], "row codes")
    assert_exact(host_u8(row["scales"][0, R - 16:]), ref["row_scales"], "row scales")
    nb = 16 * Cc // 16  # 4/6 bits of the last 16 rows
    assert_exact(_bits(row["choice"][0].cpu().numpy(), (R - 16) * Cc // 16, nb),
                 _bits(ref["row_choice"], 0, nb), "row 4/6 choices")
    col = out["col"]
    cwords = col["choice"][0].cpu().numpy()
    for c in (0, 1777, Cc - 1):
        ref = oracle.quantize(host_u16(x[:, c].contiguous()).reshape(1, 1, R), gam,
                              four_over_six=1, dequant=False)
        assert_exact(host_u8(col["codes"][0, c]), ref["row_codes"], f"column {c} codes")
        assert_exact(host_u8(col["scales"][0, c]), ref["row_scales"], f"column {c} scales")
        assert_exact(_bits(cwords, c * (R // 16), R // 16), _bits(ref["row_choice"], 0, R // 16),
                     f"column {c} 4/6 choices")
    del out, row, col
    # row-only stochastic rounding: the random bits are keyed on flat indices past 2^31
    cfg = nv.Config(rounding=1, scale_max=448.0, seed=5, step=2)
    sr = nv.nvfp4_quantize(x, amax, cfg, status=st, dequant=False)["row"]
    assert int(st.item()) == 0
    g = oracle.decode_scale(float(amax.item()), 448.0)
    nblk = R * Cc // 16
    blocks = np.concatenate([[0, nblk - 1], (1 << 27) + np.arange(4),
                             np.random.default_rng(8).choice(nblk, 400, replace=False)])
    codes = sr["codes"].view(-1, 8)
    scales = sr["scales"].view(-1)
    xf = x.view(-1, 16)
    for b in blocks:
        b = int(b)
        r = oracle.encode_block(xf[b].float().cpu().numpy(), g, rounding=1, seed=5, step=2,
                                direction=0, idx0=b * 16)
        want = (r["codes"][0::2] | (r["codes"][1::2] << 4)).astype(np.uint8)
        assert_exact(host_u8(codes[b]), want, f"codes of block {b}")
        assert int(scales[b].item()) == r["scale"], f"scale of block {b}"
