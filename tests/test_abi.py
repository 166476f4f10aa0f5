"""The C-ABI library builds, loads, exports every function include/nvfp4.h
declares, and rejects bad arguments synchronously -- all without a GPU (the
validation runs before any CUDA call, so nothing here launches a kernel)."""
import ctypes as C
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "nvfp4.h")


@pytest.fixture(scope="module")
def L():
    import nvfp4_block_scaled_02_gb300 as nv
    nv.build()
    return nv.lib()


def _declared():
    text = open(HEADER).read()
    return re.findall(r"NVFP4_API\s+[\w\s\*]+?\b(nvfp4_\w+)\s*\(", text)


def test_header_declares_the_boundary():
    names = set(_declared())
    assert {"nvfp4_amax", "nvfp4_quantize", "nvfp4_fakequant_fwd",
            "nvfp4_scale_grad_bwd"} <= names


def test_every_declared_symbol_is_exported(L):
    for name in _declared():
        assert hasattr(L, name), name


def test_library_links_no_oracle_and_no_cpu_path():
    """The product library and the oracle share nothing: no oracle symbol is in
    the CUDA library and the package source never imports the oracle."""
    import nvfp4_block_scaled_02_gb300 as nv
    lib = nv.lib()
    for sym in ("orc_quantize", "orc_e2m1_rne", "orc_philox4x32_10"):
        assert not hasattr(lib, sym)
    pkg = os.path.dirname(nv.__file__)
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in src and "from oracle" not in src, f
                assert "nvfp4_oracle" not in src, f


def _cfg(**kw):
    import nvfp4_block_scaled_02_gb300 as nv
    c = nv.Config(**kw).c()
    return c


FAKE = 0x100000  # a 16-byte aligned, never dereferenced address


def _out(codes=FAKE, scales=FAKE, choice=FAKE, dq=FAKE):
    import nvfp4_block_scaled_02_gb300 as nv
    return nv._Out(codes, scales, choice, dq)


def q(L, cfg, x=FAKE, S=1, R=16, Cc=32, amax=FAKE, row=None, col=None, status=None):
    return L.nvfp4_quantize(C.byref(cfg) if cfg is not None else None, x, S, R, Cc, amax,
                            C.byref(row) if row is not None else None,
                            C.byref(col) if col is not None else None, status, None)


def test_quantize_argument_errors(L):
    assert q(L, None) == 1
    for bad in (dict(blocks=0), dict(blocks=5), dict(scale_fmt=2), dict(rounding=3),
                dict(four_over_six=2), dict(scale_max=-1.0), dict(scale_max=float("nan")),
                dict(four_over_six_rule=3), dict(four_over_six_rule=-1)):
        assert q(L, _cfg(**bad), row=_out(), col=_out()) == 4, bad
    assert q(L, _cfg(blocks=1), Cc=24, row=_out()) == 2      # cols % 16 for row blocks
    assert q(L, _cfg(blocks=2), R=24, col=_out()) == 2       # rows % 16 for column blocks
    assert q(L, _cfg(blocks=3), R=24, row=_out(), col=_out()) == 2
    assert q(L, _cfg(blocks=1), R=-1, row=_out()) == 2
    assert q(L, _cfg(blocks=1), x=0, row=_out()) == 1
    assert q(L, _cfg(blocks=1), amax=0, row=_out()) == 1
    assert q(L, _cfg(blocks=1), row=None) == 1
    assert q(L, _cfg(blocks=2), col=None) == 1
    assert q(L, _cfg(blocks=1, four_over_six=1), row=_out(choice=0)) == 1
    assert q(L, _cfg(blocks=1), x=FAKE + 2, row=_out()) == 3
    assert q(L, _cfg(blocks=1), row=_out(codes=FAKE + 4)) == 3
    assert q(L, _cfg(blocks=1), row=_out(dq=FAKE + 8)) == 3
    assert q(L, _cfg(blocks=1), amax=FAKE + 1, row=_out()) == 3


def test_tile16_argument_errors(L):
    t = _cfg(blocks=4)
    assert q(L, _cfg(blocks=5), row=_out(), col=_out()) == 4
    assert q(L, _cfg(blocks=4, four_over_six=1), row=_out(), col=_out()) == 4
    assert q(L, t, R=24, row=_out(), col=_out()) == 2       # rows % 16
    assert q(L, t, Cc=24, row=_out(), col=_out()) == 2      # cols % 16
    assert q(L, t, row=None, col=_out()) == 1               # row encoding required
    assert q(L, t, x=0, row=_out(), col=_out()) == 1
    assert q(L, t, row=_out(), col=_out(dq=0)) == 1          # dequant for both or neither
    assert q(L, t, row=_out(codes=FAKE + 4), col=_out()) == 3
    assert q(L, t, x=0, S=0, amax=0, row=None, col=None) == 0


def test_empty_inputs_enqueue_nothing(L):
    for S, R, Cc in ((0, 16, 32), (1, 0, 32), (1, 16, 0)):
        assert q(L, _cfg(blocks=3), x=0, S=S, R=R, Cc=Cc, amax=0, row=None, col=None) == 0
    assert L.nvfp4_amax(None, 0, 4, 4, None, None, None) == 0
    assert L.nvfp4_fakequant_fwd(None, 0, 16, None, None, None, None, None) == 0
    assert L.nvfp4_scale_grad_bwd(None, None, 4, 0, None, None, None, None, None, None,
                                  None) == 0


def test_per_token_argument_errors(L):
    pt = L.nvfp4_quantize_per_token
    assert pt(None, FAKE, 4, 32, FAKE, C.byref(_out()), None, None) == 1
    assert pt(C.byref(_cfg(blocks=3)), FAKE, 4, 32, FAKE, C.byref(_out()), None, None) == 4
    assert pt(C.byref(_cfg()), FAKE, 4, 24, FAKE, C.byref(_out()), None, None) == 2
    assert pt(C.byref(_cfg()), FAKE, 4, 32, None, C.byref(_out()), None, None) == 1
    assert pt(C.byref(_cfg()), FAKE, 4, 32, FAKE, None, None, None) == 1
    assert pt(C.byref(_cfg()), FAKE + 2, 4, 32, FAKE, C.byref(_out()), None, None) == 3
    assert pt(C.byref(_cfg()), None, 0, 32, None, None, None, None) == 0


def rq(L, src, dst, target=0, codes=FAKE, scales=FAKE, S=1, R=32, Cc=32, amax=FAKE, out=None,
       status=None):
    return L.nvfp4_requant_transpose(C.byref(src) if src is not None else None,
                                     C.byref(dst) if dst is not None else None, target, codes,
                                     scales, S, R, Cc, amax,
                                     C.byref(out) if out is not None else None, status, None)


def test_requant_argument_errors(L):
    s, d = _cfg(), _cfg(rounding=1)
    ok = _out(dq=0)
    assert rq(L, None, d, out=ok) == 1
    assert rq(L, s, None, out=ok) == 1
    assert rq(L, s, d, target=2, out=ok) == 4
    for bad in (dict(scale_fmt=2), dict(four_over_six=2), dict(scale_max=-1.0)):
        assert rq(L, _cfg(**bad), d, out=ok) == 4, bad
    assert rq(L, s, _cfg(rounding=2), out=ok) == 4
    # target-side format fields matter only for the NVFP4 target
    assert rq(L, s, _cfg(scale_fmt=5), target=1, out=ok) == 4
    assert rq(L, s, _cfg(four_over_six_rule=3), target=1, out=ok) == 4
    assert rq(L, s, d, R=16, out=ok) == 2                # MXFP8 needs rows % 32
    assert rq(L, s, d, target=1, R=8, out=ok) == 2       # NVFP4 needs rows % 16
    assert rq(L, s, d, Cc=24, out=ok) == 2               # the source needs cols % 16
    assert rq(L, s, d, S=-1, out=ok) == 2
    assert rq(L, s, d, codes=0, out=ok) == 1
    assert rq(L, s, d, scales=0, out=ok) == 1
    assert rq(L, s, d, amax=0, out=ok) == 1
    assert rq(L, s, d, out=None) == 1
    assert rq(L, s, d, out=_out(codes=0, dq=0)) == 1
    assert rq(L, s, _cfg(four_over_six=1), target=1, out=_out(choice=0, dq=0)) == 1
    assert rq(L, s, d, out=_out()) == 4                  # dequant output not offered
    assert rq(L, s, d, codes=FAKE + 8, out=ok) == 3
    assert rq(L, s, d, out=_out(scales=FAKE + 1, dq=0)) == 3
    assert rq(L, s, d, amax=FAKE + 2, out=ok) == 3
    for S, R, Cc in ((0, 32, 32), (1, 0, 32), (1, 32, 0)):
        assert rq(L, s, d, codes=0, scales=0, S=S, R=R, Cc=Cc, amax=0, out=None) == 0


def mx(L, cfg, x=FAKE, S=1, R=32, Cc=64, row=None, col=None, status=None):
    return L.nvfp4_mx_quantize(C.byref(cfg) if cfg is not None else None, x, S, R, Cc,
                               C.byref(row) if row is not None else None,
                               C.byref(col) if col is not None else None, status, None)


def test_mx_quantize_argument_errors(L):
    ok = _out(choice=0, dq=0)
    assert mx(L, None, row=ok, col=ok) == 1
    for bad in (dict(blocks=0), dict(blocks=4), dict(rounding=2), dict(rounding=-1)):
        assert mx(L, _cfg(**bad), row=ok, col=ok) == 4, bad
    assert mx(L, _cfg(blocks=1), Cc=48, row=ok) == 2       # rows need cols % 32
    assert mx(L, _cfg(blocks=2), R=16, col=ok) == 2        # columns need rows % 32
    assert mx(L, _cfg(blocks=3), R=48, row=ok, col=ok) == 2
    assert mx(L, _cfg(blocks=3), S=-1, row=ok, col=ok) == 2
    assert mx(L, _cfg(blocks=1), x=0, row=ok) == 1
    assert mx(L, _cfg(blocks=1), row=None) == 1
    assert mx(L, _cfg(blocks=2), col=None) == 1
    assert mx(L, _cfg(blocks=3), row=ok, col=_out(scales=0, choice=0, dq=0)) == 1
    assert mx(L, _cfg(blocks=1), row=_out(choice=0)) == 4  # dequant output not offered
    assert mx(L, _cfg(blocks=1), x=FAKE + 2, row=ok) == 3
    assert mx(L, _cfg(blocks=1), row=_out(codes=FAKE + 8, choice=0, dq=0)) == 3
    assert mx(L, _cfg(blocks=2), col=_out(codes=FAKE + 4, choice=0, dq=0)) == 3
    assert mx(L, _cfg(blocks=1), row=_out(scales=FAKE + 1, choice=0, dq=0)) == 3
    assert mx(L, _cfg(blocks=1), row=ok, status=FAKE + 2) == 3
    # a column-only call does not need cols % 32 (nor a row output)
    assert mx(L, _cfg(blocks=2), Cc=40, col=ok, x=FAKE + 2) == 3
    for S, R, Cc in ((0, 32, 32), (1, 0, 32), (1, 32, 0)):
        assert mx(L, _cfg(blocks=3), x=0, S=S, R=R, Cc=Cc) == 0


def test_fp8_scale_learning_argument_errors(L):
    fq = L.nvfp4_fakequant_fwd_fp8scale
    assert fq(FAKE, 4, 32, FAKE, None, None, FAKE, None, None) == 1       # no global amax
    assert fq(FAKE, 4, 24, FAKE, None, FAKE, FAKE, None, None) == 2
    assert fq(FAKE, 4, 32, FAKE, None, FAKE + 2, FAKE, None, None) == 3
    assert fq(FAKE, 4, 32, FAKE, None, FAKE, None, None, None) == 1
    assert fq(None, 0, 32, None, None, None, None, None, None) == 0
    bwd = L.nvfp4_scale_grad_bwd_fp8scale
    assert bwd(FAKE, FAKE, 4, 32, FAKE, FAKE, None, FAKE, FAKE, FAKE, None, None) == 1
    assert bwd(FAKE, FAKE, 4, 32, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None) == 1
    assert bwd(FAKE, FAKE, 4, 32, FAKE, None, FAKE, FAKE, FAKE, FAKE, None, None) == 1
    init = L.nvfp4_scale_init_mse
    assert init(FAKE, 4, 32, FAKE, None, None, None, None) == 1           # no output
    assert init(FAKE, 4, 24, FAKE, FAKE, None, None, None) == 2
    assert init(FAKE, 4, 32, None, FAKE, None, None, None) == 1
    assert init(FAKE + 8, 4, 32, FAKE, FAKE, None, None, None) == 3
    assert init(FAKE, 4, 32, FAKE, None, FAKE + 2, None, None) == 3
    assert init(None, 4, 0, None, None, None, None, None) == 0
    ex = L.nvfp4_export_scales
    assert ex(FAKE, 4, 32, FAKE, None, FAKE, None, None, None) == 1
    assert ex(FAKE, 4, 32, FAKE, None, FAKE, C.byref(_out(scales=0, dq=0)), None, None) == 1
    assert ex(FAKE, 4, 32, FAKE, None, FAKE, C.byref(_out()), None, None) == 4   # dequant
    assert ex(FAKE, 4, 32, FAKE, None, FAKE, C.byref(_out(codes=FAKE + 4, dq=0)), None,
              None) == 3
    assert ex(FAKE, 4, 32, FAKE, None, None, C.byref(_out(dq=0)), None, None) == 1


def test_amax_ws_argument_errors(L):
    ws = L.nvfp4_amax_ws
    assert L.nvfp4_amax_ws_bytes(3) == 24 and L.nvfp4_amax_ws_bytes(0) == 0
    assert ws(FAKE, 2, 4, 4, FAKE, None, 16, None, None) == 1        # no workspace
    assert ws(FAKE, 2, 4, 4, FAKE, FAKE, 15, None, None) == 2        # workspace too small
    assert ws(FAKE, 2, 4, 4, None, FAKE, 16, None, None) == 1        # no output
    assert ws(None, 2, 4, 4, FAKE, FAKE, 16, None, None) == 1        # no input
    assert ws(FAKE, -1, 4, 4, FAKE, FAKE, 16, None, None) == 2
    assert ws(FAKE + 2, 2, 4, 4, FAKE, FAKE, 16, None, None) == 3    # misaligned x
    assert ws(FAKE, 2, 4, 4, FAKE, FAKE + 2, 16, None, None) == 3    # misaligned workspace
    assert ws(None, 0, 4, 4, None, None, 0, None, None) == 0         # empty: nothing enqueued


def test_amax_noalloc_argument_errors(L):
    na = L.nvfp4_amax_noalloc
    assert na(FAKE, 4097, 4, 4, FAKE, None, None) == 2      # above the fixed scratch's limit
    assert na(FAKE, -1, 4, 4, FAKE, None, None) == 2
    assert na(FAKE, 2, 4, 4, None, None, None) == 1
    assert na(None, 2, 4, 4, FAKE, None, None) == 1
    assert na(FAKE + 2, 2, 4, 4, FAKE, None, None) == 3
    assert na(None, 0, 4, 4, None, None, None) == 0         # empty: nothing enqueued


def test_amax_argument_errors(L):
    assert L.nvfp4_amax(FAKE, -1, 4, 4, FAKE, None, None) == 2
    assert L.nvfp4_amax(FAKE, 1, 4, 4, None, None, None) == 1
    assert L.nvfp4_amax(None, 1, 4, 4, FAKE, None, None) == 1
    assert L.nvfp4_amax(FAKE + 2, 1, 4, 4, FAKE, None, None) == 3


def test_ste_argument_errors(L):
    assert L.nvfp4_fakequant_fwd(FAKE, 4, 24, FAKE, None, FAKE, None, None) == 2
    assert L.nvfp4_fakequant_fwd(FAKE, 4, 32, None, None, FAKE, None, None) == 1
    assert L.nvfp4_fakequant_fwd(FAKE, 4, 32, FAKE, None, None, None, None) == 1
    assert L.nvfp4_fakequant_fwd(FAKE + 8, 4, 32, FAKE, None, FAKE, None, None) == 3
    bwd = L.nvfp4_scale_grad_bwd
    assert bwd(FAKE, FAKE, 4, 24, FAKE, FAKE, FAKE, FAKE, FAKE, None, None) == 2
    assert bwd(FAKE, FAKE, 4, 32, FAKE, FAKE, FAKE, FAKE, None, None, None) == 1  # dual, no gs_post
    assert bwd(FAKE, FAKE, 4, 32, FAKE, None, FAKE, FAKE, FAKE, None, None) == 1  # tied + gs_post
    assert bwd(FAKE, FAKE, 4, 32, FAKE, None, FAKE, None, None, None, None) == 1  # no gs_pre
    assert bwd(FAKE, None, 4, 32, FAKE, None, FAKE, FAKE, None, None, None) == 1
    assert bwd(FAKE, FAKE + 4, 4, 32, FAKE, None, FAKE, FAKE, None, None, None) == 3


def test_diagnostics_argument_errors(L):
    assert L.nvfp4_codec_probe(8, FAKE, None, 4, FAKE, None) == 4
    assert L.nvfp4_codec_probe(7, FAKE, None, 4, FAKE, None) == 1
    assert L.nvfp4_codec_probe(3, FAKE, None, 4, FAKE, None) == 1
    assert L.nvfp4_codec_probe(0, FAKE, None, -1, FAKE, None) == 2
    assert L.nvfp4_sr_bits(0, 0, 0, 0, 4, None, None) == 1


def test_status_strings(L):
    for code in (0, 1, 2, 3, 4, 6):
        assert L.nvfp4_status_string(code)
    assert L.nvfp4_status_string(99) == b"unknown status"


def test_binding_refuses_cpu_tensors():
    import torch
    import nvfp4_block_scaled_02_gb300 as nv
    x = torch.zeros((16, 32), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        nv.nvfp4_amax(x)


def test_sizes_whose_element_count_overflows_are_shape_errors(L):
    """A dimension or element count above 2^60 - 1 (byte offsets of up to 8
    bytes per element would no longer fit in int64) is refused before any
    pointer is read, including products that would wrap around to a small
    or negative count."""
    big = 1 << 40
    assert q(L, _cfg(blocks=1), R=big, Cc=big, row=_out()) == 2          # 2^80 elements
    assert q(L, _cfg(blocks=3), S=1 << 21, R=1 << 20, Cc=1 << 20, row=_out(), col=_out()) == 2
    assert q(L, _cfg(blocks=4), R=big, Cc=big, row=_out(), col=_out()) == 2
    assert q(L, _cfg(blocks=1), S=1 << 62, R=0, row=_out()) == 2        # one dimension alone
    assert L.nvfp4_amax(FAKE, 1, 1 << 32, 1 << 32, FAKE, None, None) == 2  # 2^64 wraps to 0
    assert L.nvfp4_amax(FAKE, 1 << 61, 0, 4, FAKE, None, None) == 2
    pt = L.nvfp4_quantize_per_token
    assert pt(C.byref(_cfg()), FAKE, big, big, FAKE, C.byref(_out()), None, None) == 2
    assert L.nvfp4_fakequant_fwd(FAKE, big, big, FAKE, None, FAKE, None, None) == 2
    assert L.nvfp4_codec_probe(0, FAKE, None, 1 << 61, FAKE, None) == 2
    assert L.nvfp4_sr_bits(0, 0, 0, 0, 1 << 61, FAKE, None) == 2
    # the largest accepted count still gets past the shape check (to the null check)
    assert L.nvfp4_amax(None, 1, 1 << 30, (1 << 30) - 1, FAKE, None, None) == 1
    assert L.nvfp4_amax(None, 1, 1 << 30, 1 << 30, FAKE, None, None) == 2   # 2^60
