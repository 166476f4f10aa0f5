"""CPU oracle for NVFP4 block-scaled quantisation and the scale-learning STE.

TEST INFRASTRUCTURE, not product code. Only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import this package. The CUDA
library never loads it and shares no code with it.

The arithmetic lives in ``nvfp4_oracle.c`` (plain single-threaded C, fp32
round-to-nearest, no contraction); this module only compiles it with gcc and
marshals numpy arrays through ctypes. A second build of the same source with
OpenMP (``set_threads(n)``, n > 1) runs its independent loops on n host
threads, only to time the oracle on all cores; it returns the same bytes.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nvfp4_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_LIB_OMP = os.path.join(_HERE, "liboracle_omp.so")
_lock = threading.Lock()
_lib = None
_lib_omp = None
_threads = 1

ST_NONFINITE_INPUT = 1
ST_BAD_SCALE = 2
ST_BAD_AMAX = 4

CFLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def _compile(out: str, extra: list) -> None:
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, *extra, _SRC, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, out)


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/liboracle.so`` (one thread) and
    ``oracle/liboracle_omp.so`` (the same source with OpenMP, used only to
    time the oracle on all host cores); skipped when up to date."""
    for out, extra in ((_LIB, []), (_LIB_OMP, ["-fopenmp"])):
        if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(_SRC):
            _compile(out, extra)
    return _LIB


def set_threads(n: int) -> int:
    """Run the following oracle calls on n host threads: 1 selects the
    single-threaded build, more the OpenMP build of the same source. Returns
    the thread count in use."""
    global _threads
    with _lock:
        _threads = max(1, int(n))
    return lib().orc_set_threads(_threads) if _threads > 1 else 1


def threads() -> int:
    return _threads


def lib() -> C.CDLL:
    global _lib, _lib_omp
    with _lock:
        if _lib is None:
            build()
            _lib = C.CDLL(_LIB)
            _declare(_lib)
        if _threads > 1 and _lib_omp is None:
            _lib_omp = C.CDLL(_LIB_OMP)
            _declare(_lib_omp)
        return _lib_omp if _threads > 1 else _lib


_u8p = C.POINTER(C.c_uint8)
_u16p = C.POINTER(C.c_uint16)
_u32p = C.POINTER(C.c_uint32)
_f32p = C.POINTER(C.c_float)
_i64 = C.c_int64


def _declare(L):
    L.orc_set_threads.restype = C.c_int
    L.orc_set_threads.argtypes = [C.c_int]
    L.orc_bf16_to_f32.restype = C.c_float
    L.orc_bf16_to_f32.argtypes = [C.c_uint16]
    L.orc_f32_to_bf16.restype = C.c_uint16
    L.orc_f32_to_bf16.argtypes = [C.c_float]
    L.orc_f32_to_bf16_array.argtypes = [_f32p, _i64, _u16p]
    for name in ("orc_e2m1_value", "orc_e4m3_value", "orc_ue5m3_value"):
        getattr(L, name).restype = C.c_float
        getattr(L, name).argtypes = [C.c_uint8]
    L.orc_scale_value.restype = C.c_float
    L.orc_scale_value.argtypes = [C.c_int, C.c_uint8]
    L.orc_e2m1_rne.restype = C.c_uint8
    L.orc_e2m1_rne.argtypes = [C.c_float]
    L.orc_scale_encode.restype = C.c_uint8
    L.orc_scale_encode.argtypes = [C.c_int, C.c_float]
    L.orc_e2m1_sr.restype = C.c_uint8
    L.orc_e2m1_sr.argtypes = [C.c_float, C.c_uint32]
    L.orc_philox4x32_10.argtypes = [_u32p, _u32p, _u32p]
    L.orc_sr_bits.restype = C.c_uint32
    L.orc_sr_bits.argtypes = [C.c_uint32, C.c_uint32, C.c_uint32, C.c_uint64]
    L.orc_e2m1_rne_array.argtypes = [_f32p, _i64, _u8p]
    L.orc_scale_encode_array.argtypes = [C.c_int, _f32p, _i64, _u8p]
    L.orc_e2m1_sr_array.argtypes = [_f32p, _u32p, _i64, _u8p]
    L.orc_sr_bits_array.argtypes = [C.c_uint32, C.c_uint32, C.c_uint32, C.c_uint64, _i64, _u32p]
    L.orc_encode_block.argtypes = [_f32p, C.c_float, C.c_int, C.c_int, C.c_int, C.c_int,
                                   C.c_uint32, C.c_uint32, C.c_uint32, C.c_uint64,
                                   _u8p, _u8p, _u8p, _u16p, _f32p, _f32p]
    L.orc_global_amax.restype = C.c_int
    L.orc_global_amax.argtypes = [_u16p, _i64, _i64, _f32p]
    L.orc_decode_scale.restype = C.c_float
    L.orc_decode_scale.argtypes = [C.c_float, C.c_float]
    L.orc_quantize.restype = C.c_int
    L.orc_quantize.argtypes = [C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, C.c_float,
                               C.c_uint32, C.c_uint32, _u16p, _i64, _i64, _i64, _f32p,
                               _u8p, _u8p, _u32p, _u16p, _u8p, _u8p, _u32p, _u16p]
    L.orc_e4m3_sr.restype = C.c_uint8
    L.orc_e4m3_sr.argtypes = [C.c_float, C.c_uint32]
    L.orc_e4m3_rne.restype = C.c_uint8
    L.orc_e4m3_rne.argtypes = [C.c_float]
    L.orc_e4m3_signed_value.restype = C.c_float
    L.orc_e4m3_signed_value.argtypes = [C.c_uint8]
    L.orc_mx_shared_exp.restype = C.c_int
    L.orc_mx_shared_exp.argtypes = [C.c_float]
    L.orc_mx_encode.argtypes = [_f32p, _i64, C.c_int, C.c_uint32, C.c_uint32, C.c_uint32,
                                C.c_uint64, _u8p, _u8p]
    L.orc_dequant.restype = C.c_int
    L.orc_dequant.argtypes = [C.c_int, C.c_float, C.c_int, _u8p, _u8p, _i64, _i64, _i64, _f32p,
                              _f32p]
    L.orc_requant.restype = C.c_int
    L.orc_requant.argtypes = [C.c_int, C.c_float, C.c_int, _u8p, _u8p, _i64, _i64, _i64, _f32p,
                              C.c_int, C.c_int, C.c_uint32, C.c_uint32, C.c_int, C.c_int,
                              C.c_int, C.c_float, _u8p, _u8p, _u32p]
    L.orc_e4m3_rne_array.argtypes = [_f32p, _i64, _u8p]
    L.orc_e4m3_sr_array.argtypes = [_f32p, _u32p, _i64, _u8p]
    L.orc_mx_shared_exp_array.argtypes = [_f32p, _i64, _u8p]
    L.orc_mx_quantize.restype = C.c_int
    L.orc_mx_quantize.argtypes = [C.c_int, C.c_int, C.c_uint32, C.c_uint32, _u16p, _i64, _i64,
                                  _i64, _u8p, _u8p, _u8p, _u8p]
    L.orc_quantize_tile16.restype = C.c_int
    L.orc_quantize_tile16.argtypes = [C.c_int, C.c_int, C.c_float, C.c_uint32, C.c_uint32, _u16p,
                                      _i64, _i64, _i64, _f32p, _u8p, _u8p, _u16p, _u8p, _u8p,
                                      _u16p]
    L.orc_fakequant_fwd_fp8.restype = C.c_int
    L.orc_fakequant_fwd_fp8.argtypes = [_u16p, _i64, _i64, _f32p, _f32p, C.c_float, _u16p]
    L.orc_scale_grad_bwd_fp8.restype = C.c_int
    L.orc_scale_grad_bwd_fp8.argtypes = [_u16p, _u16p, _i64, _i64, _f32p, _f32p, C.c_float,
                                         _u16p, _f32p, _f32p]
    L.orc_scale_init_mse.restype = C.c_int
    L.orc_scale_init_mse.argtypes = [_u16p, _i64, _i64, C.c_float, _u8p, _f32p, _f32p]
    L.orc_export_scales.restype = C.c_int
    L.orc_export_scales.argtypes = [_u16p, _i64, _i64, _f32p, _f32p, C.c_float, _u8p, _u8p]
    L.orc_fakequant_fwd.restype = C.c_int
    L.orc_fakequant_fwd.argtypes = [_u16p, _i64, _i64, _f32p, _f32p, _u16p]
    L.orc_scale_grad_bwd.restype = C.c_int
    L.orc_scale_grad_bwd.argtypes = [_u16p, _u16p, _i64, _i64, _f32p, _f32p, _u16p,
                                     _f32p, _f32p]


def _c(a, dtype) -> np.ndarray:
    """C-contiguous array of dtype that keeps the shape (0-d included)."""
    a = np.asarray(a, dtype=dtype)
    return a if a.flags["C_CONTIGUOUS"] else np.ascontiguousarray(a)


def _p(a, ptype):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ptype)


# ---------------------------------------------------------------- codecs --

def bf16_to_f32(h) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    return (h.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(f) -> np.ndarray:
    f = _c(f, np.float32)
    out = np.empty(f.shape, np.uint16)
    lib().orc_f32_to_bf16_array(_p(f, _f32p), f.size, _p(out, _u16p))
    return out


def e2m1_value(codes) -> np.ndarray:
    L = lib()
    c = np.asarray(codes, dtype=np.uint8)
    return np.array([L.orc_e2m1_value(int(v)) for v in c.ravel()], np.float32).reshape(c.shape)


def scale_value(fmt: int, codes) -> np.ndarray:
    L = lib()
    c = np.asarray(codes, dtype=np.uint8)
    return np.array([L.orc_scale_value(fmt, int(v)) for v in c.ravel()], np.float32).reshape(c.shape)


def e2m1_rne(y) -> np.ndarray:
    y = _c(y, np.float32)
    out = np.empty(y.shape, np.uint8)
    lib().orc_e2m1_rne_array(_p(y, _f32p), y.size, _p(out, _u8p))
    return out


def scale_encode(fmt: int, t) -> np.ndarray:
    t = _c(t, np.float32)
    out = np.empty(t.shape, np.uint8)
    lib().orc_scale_encode_array(int(fmt), _p(t, _f32p), t.size, _p(out, _u8p))
    return out


def e2m1_sr(y, v16) -> np.ndarray:
    y = _c(y, np.float32)
    v = np.ascontiguousarray(np.broadcast_to(np.asarray(v16, np.uint32), y.shape))
    out = np.empty(y.shape, np.uint8)
    lib().orc_e2m1_sr_array(_p(y, _f32p), _p(v, _u32p), y.size, _p(out, _u8p))
    return out


def philox(ctr, key) -> np.ndarray:
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.empty(4, np.uint32)
    lib().orc_philox4x32_10(_p(c, _u32p), _p(k, _u32p), _p(out, _u32p))
    return out


def sr_bits(seed: int, step: int, direction: int, idx0: int, n: int) -> np.ndarray:
    out = np.empty(n, np.uint32)
    lib().orc_sr_bits_array(seed, step, direction, idx0, n, _p(out, _u32p))
    return out


# ---------------------------------------------------------- block level --

def encode_block(x16, g: float, fmt: int = 0, rounding: int = 0, fos: int = 0,
                 seed: int = 0, step: int = 0, direction: int = 0, idx0: int = 0,
                 rule: int = 0) -> dict:
    x = np.ascontiguousarray(x16, dtype=np.float32)
    assert x.shape == (16,)
    codes = np.empty(16, np.uint8)
    scale = np.empty(1, np.uint8)
    choice = np.empty(1, np.uint8)
    dq = np.empty(16, np.uint16)
    dqf = np.empty(16, np.float32)
    sse = np.empty(2, np.float32)
    lib().orc_encode_block(_p(x, _f32p), g, fmt, rounding, fos, rule, seed, step, direction, idx0,
                           _p(codes, _u8p), _p(scale, _u8p), _p(choice, _u8p),
                           _p(dq, _u16p), _p(dqf, _f32p), _p(sse, _f32p))
    return dict(codes=codes, scale=int(scale[0]), choice=int(choice[0]), dq=dq, dqf=dqf,
                sse6=float(sse[0]), sse4=float(sse[1]))


def decode_scale(gamax: float, M: float) -> float:
    """The per-slice decode scale g = gamax / (6 M) (1 for a zero or bad amax)."""
    return float(lib().orc_decode_scale(float(gamax), float(M)))


# ----------------------------------------------------------- whole path --

def global_amax(x_bf16: np.ndarray, slices: int = 1):
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16).reshape(-1)
    n = x.size // slices if slices else 0
    out = np.zeros(max(slices, 1), np.float32)[:slices]
    st = lib().orc_global_amax(_p(x, _u16p), slices, n, _p(out, _f32p))
    return out, st


def quantize(x_bf16: np.ndarray, gamax: np.ndarray, *, blocks: int = 1, scale_fmt: int = 0,
             rounding: int = 0, four_over_six: int = 0, scale_max: float = 0.0,
             seed: int = 0, step: int = 0, dequant: bool = True, rule: int = 0) -> dict:
    """x_bf16: uint16 array shaped [S, R, C] (or [R, C]); gamax: float32 [S]."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    if x.ndim == 2:
        x = x[None]
    S, R, Cc = x.shape
    gam = np.ascontiguousarray(gamax, dtype=np.float32).reshape(-1)
    assert gam.size == S
    out = {}
    B = R * Cc // 16
    W = (B + 31) // 32

    def alloc(tag, mr, mc):
        out[tag + "codes"] = np.zeros((S, mr, mc // 2), np.uint8)
        out[tag + "scales"] = np.zeros((S, mr, mc // 16), np.uint8)
        out[tag + "choice"] = np.zeros((S, W), np.uint32)
        out[tag + "dq"] = np.zeros((S, mr, mc), np.uint16) if dequant else None

    if blocks & 1:
        alloc("row_", R, Cc)
    if blocks & 2:
        alloc("col_", Cc, R)
    g = out.get
    st = lib().orc_quantize(blocks, scale_fmt, rounding, four_over_six, rule, scale_max, seed, step,
                            _p(x, _u16p), S, R, Cc, _p(gam, _f32p),
                            _p(g("row_codes"), _u8p), _p(g("row_scales"), _u8p),
                            _p(g("row_choice"), _u32p), _p(g("row_dq"), _u16p),
                            _p(g("col_codes"), _u8p), _p(g("col_scales"), _u8p),
                            _p(g("col_choice"), _u32p), _p(g("col_dq"), _u16p))
    out["status"] = st
    return out


def mx_quantize(x_bf16: np.ndarray, *, blocks: int = 3, rounding: int = 1, seed: int = 0,
                step: int = 0) -> dict:
    """MXFP8 encodings of a bf16 [S, R, C] tensor: rows (blocks of 32 along C,
    codes [S, R, C], E8M0 scales [S, R, C/32]) and/or columns (the row encoding
    of the transpose, codes [S, C, R], scales [S, C, R/32])."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    if x.ndim == 2:
        x = x[None]
    S, R, Cc = x.shape
    out = {"row_codes": np.zeros((S, R, Cc), np.uint8) if blocks & 1 else None,
           "row_scales": np.zeros((S, R, Cc // 32), np.uint8) if blocks & 1 else None,
           "col_codes": np.zeros((S, Cc, R), np.uint8) if blocks & 2 else None,
           "col_scales": np.zeros((S, Cc, R // 32), np.uint8) if blocks & 2 else None}
    g = out.get
    out["status"] = lib().orc_mx_quantize(
        blocks, rounding, seed, step, _p(x, _u16p), S, R, Cc, _p(g("row_codes"), _u8p),
        _p(g("row_scales"), _u8p), _p(g("col_codes"), _u8p), _p(g("col_scales"), _u8p))
    return out


def quantize_tile16(x_bf16: np.ndarray, gamax: np.ndarray, *, scale_fmt: int = 0,
                    rounding: int = 0, scale_max: float = 0.0, seed: int = 0, step: int = 0,
                    dequant: bool = True) -> dict:
    """One scale per 16x16 tile: the row encoding of x [S, R, C] and its exact
    transpose as the column encoding (keys as quantize())."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    if x.ndim == 2:
        x = x[None]
    S, R, Cc = x.shape
    gam = np.ascontiguousarray(gamax, dtype=np.float32).reshape(-1)
    out = {"row_codes": np.zeros((S, R, Cc // 2), np.uint8),
           "row_scales": np.zeros((S, R, Cc // 16), np.uint8),
           "row_dq": np.zeros((S, R, Cc), np.uint16),
           "col_codes": np.zeros((S, Cc, R // 2), np.uint8),
           "col_scales": np.zeros((S, Cc, R // 16), np.uint8),
           "col_dq": np.zeros((S, Cc, R), np.uint16)}
    g = out.get
    out["status"] = lib().orc_quantize_tile16(
        scale_fmt, rounding, scale_max, seed, step, _p(x, _u16p), S, R, Cc, _p(gam, _f32p),
        _p(g("row_codes"), _u8p), _p(g("row_scales"), _u8p), _p(g("row_dq"), _u16p),
        _p(g("col_codes"), _u8p), _p(g("col_scales"), _u8p), _p(g("col_dq"), _u16p))
    if not dequant:
        out["row_dq"] = out["col_dq"] = None
    return out


def fakequant_fwd(x_bf16, s_pre, s_post=None):
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    R, Cc = x.shape
    sp = np.ascontiguousarray(s_pre, dtype=np.float32)
    so = None if s_post is None else np.ascontiguousarray(s_post, dtype=np.float32)
    xq = np.empty_like(x)
    st = lib().orc_fakequant_fwd(_p(x, _u16p), R, Cc, _p(sp, _f32p), _p(so, _f32p),
                                 _p(xq, _u16p))
    return xq, st


def scale_grad_bwd(x_bf16, gq_bf16, s_pre, s_post=None, want_gx: bool = True):
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    gq = np.ascontiguousarray(gq_bf16, dtype=np.uint16)
    R, Cc = x.shape
    sp = np.ascontiguousarray(s_pre, dtype=np.float32)
    so = None if s_post is None else np.ascontiguousarray(s_post, dtype=np.float32)
    gx = np.empty_like(x) if want_gx else None
    gs_pre = np.empty(sp.shape, np.float32)
    gs_post = None if so is None else np.empty(sp.shape, np.float32)
    st = lib().orc_scale_grad_bwd(_p(x, _u16p), _p(gq, _u16p), R, Cc, _p(sp, _f32p),
                                  _p(so, _f32p), _p(gx, _u16p), _p(gs_pre, _f32p),
                                  _p(gs_post, _f32p))
    return dict(gx=gx, gs_pre=gs_pre, gs_post=gs_post, status=st)


# ------------------------------------------- scale learning, FP8 scales --

def fakequant_fwd_fp8(x_bf16, s_pre, s_post, gamax):
    """Fake quantisation at the FP8-rounded scales (s_post None = tied)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    R, Cc = x.shape
    sp = np.ascontiguousarray(s_pre, dtype=np.float32)
    so = None if s_post is None else np.ascontiguousarray(s_post, dtype=np.float32)
    xq = np.empty_like(x)
    st = lib().orc_fakequant_fwd_fp8(_p(x, _u16p), R, Cc, _p(sp, _f32p), _p(so, _f32p),
                                     float(gamax), _p(xq, _u16p))
    return xq, st


def scale_grad_bwd_fp8(x_bf16, gq_bf16, s_pre, s_post, gamax, want_gx: bool = True):
    """STE backward at the FP8-rounded scales, gradients passed straight through."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    gq = np.ascontiguousarray(gq_bf16, dtype=np.uint16)
    R, Cc = x.shape
    sp = np.ascontiguousarray(s_pre, dtype=np.float32)
    so = None if s_post is None else np.ascontiguousarray(s_post, dtype=np.float32)
    gx = np.empty_like(x) if want_gx else None
    gs_pre = np.empty(sp.shape, np.float32)
    gs_post = None if so is None else np.empty(sp.shape, np.float32)
    st = lib().orc_scale_grad_bwd_fp8(_p(x, _u16p), _p(gq, _u16p), R, Cc, _p(sp, _f32p),
                                      _p(so, _f32p), float(gamax), _p(gx, _u16p),
                                      _p(gs_pre, _f32p), _p(gs_post, _f32p))
    return dict(gx=gx, gs_pre=gs_pre, gs_post=gs_post, status=st)


def scale_init_mse(x_bf16, gamax):
    """MSE scale setting with the FP8 sweep: per block the E4M3 code, its scale
    dec(code) * g and the winning block sum of squared errors."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    R, Cc = x.shape
    codes = np.empty((R, Cc // 16), np.uint8)
    s = np.empty((R, Cc // 16), np.float32)
    sse = np.empty((R, Cc // 16), np.float32)
    st = lib().orc_scale_init_mse(_p(x, _u16p), R, Cc, float(gamax), _p(codes, _u8p),
                                  _p(s, _f32p), _p(sse, _f32p))
    return dict(codes=codes, s=s, sse=sse, status=st)


def export_scales(x_bf16, s_pre, s_post, gamax):
    """NVFP4 row encoding carrying the learned post-scales: codes [R][C/2] and
    E4M3 scale bytes [R][C/16] (s_post None = tied)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    R, Cc = x.shape
    sp = np.ascontiguousarray(s_pre, dtype=np.float32)
    so = None if s_post is None else np.ascontiguousarray(s_post, dtype=np.float32)
    codes = np.empty((R, Cc // 2), np.uint8)
    scales = np.empty((R, Cc // 16), np.uint8)
    st = lib().orc_export_scales(_p(x, _u16p), R, Cc, _p(sp, _f32p), _p(so, _f32p),
                                 float(gamax), _p(codes, _u8p), _p(scales, _u8p))
    return dict(codes=codes, scales=scales, status=st)


# ------------------------------------------------------- re-quantisation --

def e4m3_sr(y, v16) -> np.ndarray:
    """Signed E4M3 codes of y by stochastic rounding with 16-bit draws v16."""
    y = _c(np.asarray(y, np.float32).ravel(), np.float32)
    v = _c(np.broadcast_to(np.asarray(v16, np.uint32), y.shape), np.uint32)
    out = np.empty(y.size, np.uint8)
    lib().orc_e4m3_sr_array(_p(y, _f32p), _p(v, _u32p), y.size, _p(out, _u8p))
    return out


def e4m3_rne(y) -> np.ndarray:
    """Signed E4M3 codes of y, round to nearest even, saturating at 448."""
    y = _c(np.asarray(y, np.float32).ravel(), np.float32)
    out = np.empty(y.size, np.uint8)
    lib().orc_e4m3_rne_array(_p(y, _f32p), y.size, _p(out, _u8p))
    return out


def mx_shared_exp_bytes(amax) -> np.ndarray:
    """E8M0 bytes (e + 127) of the MX shared exponents of the given amaxes."""
    a = _c(np.asarray(amax, np.float32).ravel(), np.float32)
    out = np.empty(a.size, np.uint8)
    lib().orc_mx_shared_exp_array(_p(a, _f32p), a.size, _p(out, _u8p))
    return out


def e4m3_signed_value(codes) -> np.ndarray:
    L = lib()
    c = np.asarray(codes, np.uint8)
    return np.array([L.orc_e4m3_signed_value(int(v)) for v in c.ravel()],
                    np.float32).reshape(c.shape)


def mx_shared_exp(amax: float) -> int:
    return lib().orc_mx_shared_exp(float(amax))


def mx_encode(v, rounding=1, seed=0, step=0, direction=2, idx0=0):
    v = np.ascontiguousarray(v, np.float32).ravel()
    codes = np.empty(v.size, np.uint8)
    scales = np.empty(v.size // 32, np.uint8)
    lib().orc_mx_encode(_p(v, _f32p), v.size, rounding, seed, step, direction, idx0,
                        _p(codes, _u8p), _p(scales, _u8p))
    return codes, scales


def dequant(codes, scales, gamax, *, scale_fmt=0, scale_max=0.0, four_over_six=0):
    """fp32 values of a row encoding: codes [S][R][C/2], scales [S][R][C/16]."""
    codes = np.ascontiguousarray(codes, np.uint8)
    scales = np.ascontiguousarray(scales, np.uint8)
    S, R, half = codes.shape
    out = np.empty((S, R, 2 * half), np.float32)
    gam = np.ascontiguousarray(gamax, np.float32)
    st = lib().orc_dequant(scale_fmt, scale_max, four_over_six, _p(codes, _u8p),
                           _p(scales, _u8p), S, R, 2 * half, _p(gam, _f32p), _p(out, _f32p))
    return out, st


def requant(codes, scales, gamax, *, target=0, rounding=1, seed=0, step=0, src_fmt=0,
            src_scale_max=0.0, src_fos=0, dst_fmt=0, dst_fos=0, dst_rule=0,
            dst_scale_max=0.0) -> dict:
    """De-quantise a row encoding [S][R][C], transpose, re-quantise: target 0 =
    MXFP8 (codes [S][C][R], E8M0 scales [S][C][R/32]), 1 = NVFP4 (codes
    [S][C][R/2], scales [S][C][R/16], bitmap when dst_fos)."""
    codes = np.ascontiguousarray(codes, np.uint8)
    scales = np.ascontiguousarray(scales, np.uint8)
    S, R, half = codes.shape
    Cc = 2 * half
    gam = np.ascontiguousarray(gamax, np.float32)
    if target == 0:
        oc = np.zeros((S, Cc, R), np.uint8)
        os_ = np.zeros((S, Cc, R // 32), np.uint8)
        ch = None
    else:
        oc = np.zeros((S, Cc, R // 2), np.uint8)
        os_ = np.zeros((S, Cc, R // 16), np.uint8)
        ch = np.zeros((S, (R * Cc // 16 + 31) // 32), np.uint32) if dst_fos else None
    st = lib().orc_requant(src_fmt, src_scale_max, src_fos, _p(codes, _u8p), _p(scales, _u8p),
                           S, R, Cc, _p(gam, _f32p), target, rounding, seed, step, dst_fmt,
                           dst_fos, dst_rule, dst_scale_max, _p(oc, _u8p), _p(os_, _u8p),
                           _p(ch, _u32p))
    return dict(codes=oc, scales=os_, choice=ch, status=st)
