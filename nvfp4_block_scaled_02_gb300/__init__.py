"""GB300 (sm_103a) NVFP4 block-scaled quantisation and scale-learning STE.

The compute lives in ``libnvfp4.so`` (hand-written CUDA behind the C ABI of
``include/nvfp4.h``). This module only marshals arguments: it passes device
pointers of torch tensors and the current CUDA stream to the C entry points,
which have the same names. There is no CPU fallback: every call raises if the
library is not built or no CUDA device is present.

    from nvfp4_block_scaled_02_gb300 import nvfp4_amax, nvfp4_quantize, Config
    amax = nvfp4_amax(x)                           # current tensor scaling
    out = nvfp4_quantize(x, amax, Config(four_over_six=1))
"""
from __future__ import annotations

import ctypes as C
import functools
import os
import threading
from dataclasses import dataclass

import torch

__all__ = [
    "Config", "Nvfp4Error", "build", "lib", "nvfp4_amax", "nvfp4_quantize",
    "nvfp4_fakequant_fwd", "nvfp4_scale_grad_bwd", "nvfp4_codec_probe", "nvfp4_sr_bits",
    "nvfp4_quantize_per_token", "nvfp4_requant_transpose", "TARGET_MXFP8", "TARGET_NVFP4",
    "nvfp4_fakequant_fwd_fp8scale", "nvfp4_scale_grad_bwd_fp8scale", "nvfp4_scale_init_mse",
    "nvfp4_export_scales", "nvfp4_mx_quantize", "alloc_mx",
    "alloc_encoding", "alloc_requant", "PeriodicAmax", "BLOCKS_ROW", "BLOCKS_COL", "BLOCKS_BOTH",
    "BLOCKS_TILE16",
    "SCALE_E4M3", "SCALE_UE5M3", "ROUND_RNE", "ROUND_SR", "FOS_MSE", "FOS_MAE", "FOS_MAX",
    "DEV_NONFINITE_INPUT", "DEV_BAD_SCALE", "DEV_BAD_AMAX",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libnvfp4.so")

BLOCKS_ROW, BLOCKS_COL, BLOCKS_BOTH, BLOCKS_TILE16 = 1, 2, 3, 4
FOS_MSE, FOS_MAE, FOS_MAX = 0, 1, 2
SCALE_E4M3, SCALE_UE5M3 = 0, 1
ROUND_RNE, ROUND_SR = 0, 1
DEV_NONFINITE_INPUT, DEV_BAD_SCALE, DEV_BAD_AMAX = 1, 2, 4
TARGET_MXFP8, TARGET_NVFP4 = 0, 1

_STATUS = {0: "ok", 1: "null pointer", 2: "shape", 3: "alignment", 4: "enum", 6: "cuda"}


class Nvfp4Error(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: status {code} ({_STATUS.get(code, '?')})")
        self.code = code


class _Config(C.Structure):
    _fields_ = [("blocks", C.c_int32), ("scale_fmt", C.c_int32), ("rounding", C.c_int32),
                ("four_over_six", C.c_int32), ("scale_max", C.c_float), ("seed", C.c_uint32),
                ("step", C.c_uint32), ("four_over_six_rule", C.c_int32)]


class _Out(C.Structure):
    _fields_ = [("codes", C.c_void_p), ("scales", C.c_void_p), ("choice", C.c_void_p),
                ("dequant", C.c_void_p)]


@dataclass
class Config:
    blocks: int = BLOCKS_ROW
    scale_fmt: int = SCALE_E4M3
    rounding: int = ROUND_RNE
    four_over_six: int = 0
    scale_max: float = 0.0
    seed: int = 0
    step: int = 0
    four_over_six_rule: int = 0  # FOS_MSE, FOS_MAE or FOS_MAX

    def c(self) -> _Config:
        return _Config(self.blocks, self.scale_fmt, self.rounding, self.four_over_six,
                       self.scale_max, self.seed & 0xFFFFFFFF, self.step & 0xFFFFFFFF,
                       self.four_over_six_rule)


_lock = threading.Lock()
_lib = None

_i64, _vp, _u32, _i32 = C.c_int64, C.c_void_p, C.c_uint32, C.c_int32


def build(force: bool = False) -> str:
    """Compile libnvfp4.so for sm_103a (no-op when up to date)."""
    from . import buildlib
    return buildlib.build(force=force)


def lib() -> C.CDLL:
    """The loaded CUDA library. Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build the CUDA library first "
                    "(python -m nvfp4_block_scaled_02_gb300.buildlib)")
            L = C.CDLL(LIB_PATH)
            L.nvfp4_amax.argtypes = [_vp, _i64, _i64, _i64, _vp, _vp, _vp]
            L.nvfp4_amax_ws.argtypes = [_vp, _i64, _i64, _i64, _vp, _vp, C.c_size_t, _vp, _vp]
            L.nvfp4_amax_noalloc.argtypes = [_vp, _i64, _i64, _i64, _vp, _vp, _vp]
            L.nvfp4_amax_ws_bytes.argtypes = [_i64]
            L.nvfp4_amax_ws_bytes.restype = C.c_size_t
            L.nvfp4_quantize.argtypes = [C.POINTER(_Config), _vp, _i64, _i64, _i64, _vp,
                                         C.POINTER(_Out), C.POINTER(_Out), _vp, _vp]
            L.nvfp4_quantize_per_token.argtypes = [C.POINTER(_Config), _vp, _i64, _i64, _vp,
                                                   C.POINTER(_Out), _vp, _vp]
            L.nvfp4_fakequant_fwd.argtypes = [_vp, _i64, _i64, _vp, _vp, _vp, _vp, _vp]
            L.nvfp4_scale_grad_bwd.argtypes = [_vp, _vp, _i64, _i64, _vp, _vp, _vp, _vp, _vp,
                                               _vp, _vp]
            L.nvfp4_requant_transpose.argtypes = [C.POINTER(_Config), C.POINTER(_Config), _i32,
                                                  _vp, _vp, _i64, _i64, _i64, _vp,
                                                  C.POINTER(_Out), _vp, _vp]
            L.nvfp4_fakequant_fwd_fp8scale.argtypes = [_vp, _i64, _i64, _vp, _vp, _vp, _vp, _vp,
                                                       _vp]
            L.nvfp4_scale_grad_bwd_fp8scale.argtypes = [_vp, _vp, _i64, _i64, _vp, _vp, _vp, _vp,
                                                        _vp, _vp, _vp, _vp]
            L.nvfp4_scale_init_mse.argtypes = [_vp, _i64, _i64, _vp, _vp, _vp, _vp, _vp]
            L.nvfp4_export_scales.argtypes = [_vp, _i64, _i64, _vp, _vp, _vp, C.POINTER(_Out),
                                              _vp, _vp]
            L.nvfp4_mx_quantize.argtypes = [C.POINTER(_Config), _vp, _i64, _i64, _i64,
                                            C.POINTER(_Out), C.POINTER(_Out), _vp, _vp]
            L.nvfp4_codec_probe.argtypes = [_i32, _vp, _vp, _i64, _vp, _vp]
            L.nvfp4_sr_bits.argtypes = [_u32, _u32, _u32, C.c_uint64, _i64, _vp, _vp]
            L.nvfp4_status_string.restype = C.c_char_p
            L.nvfp4_status_string.argtypes = [C.c_int]
            for name in ("nvfp4_amax", "nvfp4_amax_ws", "nvfp4_amax_noalloc", "nvfp4_quantize", "nvfp4_quantize_per_token",
                         "nvfp4_requant_transpose", "nvfp4_fakequant_fwd",
                         "nvfp4_fakequant_fwd_fp8scale", "nvfp4_scale_grad_bwd_fp8scale",
                         "nvfp4_scale_init_mse", "nvfp4_export_scales", "nvfp4_mx_quantize",
                         "nvfp4_scale_grad_bwd", "nvfp4_codec_probe", "nvfp4_sr_bits"):
                getattr(L, name).restype = C.c_int
            _lib = L
    return _lib


# ------------------------------------------------------------- marshalling --

def _dev(t: torch.Tensor | None, name: str) -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (this library has no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"{name} is on {t.device} but the call runs on "
                         f"cuda:{torch.cuda.current_device()}: every buffer of a call must "
                         "be on one device")
    return t.data_ptr()


def _on_input_device(fn):
    """Run an entry point with the device of its first tensor argument
    current: the library launches on the current CUDA device and sizes its
    grids for that device's SM count."""
    @functools.wraps(fn)
    def wrapper(*args, **kwargs):
        dev = next((a.device for a in args if isinstance(a, torch.Tensor)), None)
        if dev is None or dev.type != "cuda":
            return fn(*args, **kwargs)
        with torch.cuda.device(dev):
            return fn(*args, **kwargs)
    return wrapper


def _bf16(t: torch.Tensor, name: str) -> int:
    if t.dtype not in (torch.bfloat16, torch.int16, torch.uint16):
        raise TypeError(f"{name} must hold bf16 data, got {t.dtype}")
    return _dev(t, name)


_KINDS = {"bf16": (torch.bfloat16, torch.int16, torch.uint16), "f32": (torch.float32,),
          "u8": (torch.uint8, torch.int8), "i32": (torch.int32, torch.uint32)}


def _need(t: torch.Tensor | None, name: str, n: int, kind: str) -> None:
    """Refuse a buffer the kernels would read or write past: wrong element
    type, or fewer than n elements (the ABI takes raw pointers and cannot
    check sizes itself)."""
    if t is None:
        return
    if t.dtype not in _KINDS[kind]:
        raise TypeError(f"{name} must hold {kind} data, got {t.dtype}")
    if t.numel() < n:
        raise ValueError(f"{name} holds {t.numel()} elements; the call needs {n}")


def _need_enc(enc: dict | None, name: str, s: int, r: int, c: int, four_over_six: bool) -> None:
    """An NVFP4 encoding of s x r x c values (blocks of 16 along c)."""
    if enc is None:
        return
    _need(enc["codes"], name + " codes", s * r * c // 2, "u8")
    _need(enc["scales"], name + " scales", s * r * c // 16, "u8")
    if four_over_six:
        if enc.get("choice") is None:
            raise ValueError(f"{name} needs a choice bitmap under Four-Over-Six")
        _need(enc["choice"], name + " choice", s * ((r * c // 16 + 31) // 32), "i32")
    _need(enc.get("dequant"), name + " dequant", s * r * c, "bf16")


def _stream(device: torch.device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _check(fn: str, code: int) -> None:
    if code != 0:
        raise Nvfp4Error(fn, code)


def _shape3(x: torch.Tensor):
    if x.dim() == 2:
        return 1, x.shape[0], x.shape[1]
    if x.dim() == 3:
        return x.shape[0], x.shape[1], x.shape[2]
    raise ValueError("x must be [rows, cols] or [slices, rows, cols]")


# ---------------------------------------------------------------- entries --

@_on_input_device
def nvfp4_amax(x: torch.Tensor, amax: torch.Tensor | None = None,
               status: torch.Tensor | None = None) -> torch.Tensor:
    """Per-slice max |x| of a bf16 [rows, cols] or [slices, rows, cols] tensor."""
    S, R, Cc = _shape3(x)
    _need(amax, "amax", S, "f32")
    _need(status, "status", 1, "i32")
    if amax is None:
        amax = torch.empty(S, dtype=torch.float32, device=x.device)
    _check("nvfp4_amax", lib().nvfp4_amax(_bf16(x, "x"), S, R, Cc, _dev(amax, "amax"),
                                          _dev(status, "status"), _stream(x.device)))
    return amax


def amax_workspace(slices: int, device) -> torch.Tensor:
    """A zeroed workspace for nvfp4_amax_ws (two 32-bit words per slice); every
    call leaves it zero, so it is allocated and cleared once."""
    return torch.zeros(max(2 * int(slices), 1), dtype=torch.int32, device=device)


@_on_input_device
def nvfp4_amax_ws(x: torch.Tensor, workspace: torch.Tensor, amax: torch.Tensor | None = None,
                  status: torch.Tensor | None = None) -> torch.Tensor:
    """nvfp4_amax in one kernel launch, with a caller-owned zeroed workspace
    (amax_workspace) that serves one call at a time."""
    S, R, Cc = _shape3(x)
    _need(amax, "amax", S, "f32")
    _need(status, "status", 1, "i32")
    _need(workspace, "workspace", 2 * S, "i32")
    if amax is None:
        amax = torch.empty(S, dtype=torch.float32, device=x.device)
    _check("nvfp4_amax_ws", lib().nvfp4_amax_ws(
        _bf16(x, "x"), S, R, Cc, _dev(amax, "amax"), _dev(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _dev(status, "status"), _stream(x.device)))
    return amax


AMAX_NOALLOC_MAX_SLICES = 4096


@_on_input_device
def nvfp4_amax_noalloc(x: torch.Tensor, amax: torch.Tensor | None = None,
                       status: torch.Tensor | None = None) -> torch.Tensor:
    """The one-launch amax for callers that cannot allocate device memory: the
    library's own fixed scratch array stands in for the workspace (at most
    AMAX_NOALLOC_MAX_SLICES slices; calls that overlap on the GPU race on it)."""
    S, R, Cc = _shape3(x)
    _need(amax, "amax", S, "f32")
    _need(status, "status", 1, "i32")
    if amax is None:
        amax = torch.empty(S, dtype=torch.float32, device=x.device)
    _check("nvfp4_amax_noalloc", lib().nvfp4_amax_noalloc(
        _bf16(x, "x"), S, R, Cc, _dev(amax, "amax"), _dev(status, "status"), _stream(x.device)))
    return amax


def alloc_encoding(slices: int, rows: int, cols: int, device, four_over_six: bool,
                   dequant: bool = True) -> dict:
    """Output tensors of one encoding of a [slices, rows, cols] input, for blocks
    of 16 along `cols` (pass the transposed dims for the column encoding)."""
    nb = rows * cols // 16
    w = (nb + 31) // 32
    return {
        "codes": torch.empty((slices, rows, cols // 2), dtype=torch.uint8, device=device),
        "scales": torch.empty((slices, rows, cols // 16), dtype=torch.uint8, device=device),
        "choice": (torch.empty((slices, w), dtype=torch.int32, device=device)
                   if four_over_six else None),
        "dequant": (torch.empty((slices, rows, cols), dtype=torch.bfloat16, device=device)
                    if dequant else None),
    }


def _out(enc: dict | None) -> _Out | None:
    if enc is None:
        return None
    return _Out(_dev(enc["codes"], "codes"), _dev(enc["scales"], "scales"),
                _dev(enc.get("choice"), "choice"), _dev(enc.get("dequant"), "dequant"))


@_on_input_device
def nvfp4_quantize(x: torch.Tensor, global_amax: torch.Tensor, cfg: Config | None = None,
                   row: dict | None = None, col: dict | None = None,
                   status: torch.Tensor | None = None, dequant: bool = True) -> dict:
    """NVFP4-encode a bf16 tensor. Returns {"row": {...}, "col": {...}} with the
    encodings the config asks for (allocated here unless passed in)."""
    cfg = cfg or Config()
    S, R, Cc = _shape3(x)
    fos = bool(cfg.four_over_six)
    _need(global_amax, "global_amax", S, "f32")
    _need(status, "status", 1, "i32")
    if cfg.blocks == BLOCKS_TILE16:
        _need_enc(row, "row", S, R, Cc, False)
        _need_enc(col, "col", S, Cc, R, False)
        # one scale per 16x16 tile: the row encoding and its transpose
        row = row if row is not None else alloc_encoding(S, R, Cc, x.device, False, dequant)
        col = col if col is not None else alloc_encoding(S, Cc, R, x.device, False, dequant)
        ro, co, c = _out(row), _out(col), cfg.c()
        _check("nvfp4_quantize", lib().nvfp4_quantize(
            C.byref(c), _bf16(x, "x"), S, R, Cc, _dev(global_amax, "global_amax"), C.byref(ro),
            C.byref(co), _dev(status, "status"), _stream(x.device)))
        return {"row": row, "col": col}
    _need_enc(row if cfg.blocks & 1 else None, "row", S, R, Cc, fos)
    _need_enc(col if cfg.blocks & 2 else None, "col", S, Cc, R, fos)
    if cfg.blocks & 1 and row is None:
        row = alloc_encoding(S, R, Cc, x.device, fos, dequant)
    if cfg.blocks & 2 and col is None:
        col = alloc_encoding(S, Cc, R, x.device, fos, dequant)
    ro, co = _out(row if cfg.blocks & 1 else None), _out(col if cfg.blocks & 2 else None)
    c = cfg.c()
    _check("nvfp4_quantize", lib().nvfp4_quantize(
        C.byref(c), _bf16(x, "x"), S, R, Cc, _dev(global_amax, "global_amax"),
        C.byref(ro) if ro is not None else None, C.byref(co) if co is not None else None,
        _dev(status, "status"), _stream(x.device)))
    return {"row": row if cfg.blocks & 1 else None, "col": col if cfg.blocks & 2 else None}


@_on_input_device
def nvfp4_quantize_per_token(x: torch.Tensor, cfg: Config | None = None, out: dict | None = None,
                             row_amax: torch.Tensor | None = None,
                             status: torch.Tensor | None = None, dequant: bool = True) -> dict:
    """Per-token NVFP4 encoding of a bf16 [rows, cols] tensor (one outer scale per
    row, from the row's own amax, in one pass). Returns the row encoding plus
    "row_amax" (fp32 [rows])."""
    cfg = cfg or Config()
    if x.dim() != 2:
        raise ValueError("x must be [rows, cols]")
    R, Cc = x.shape
    _need_enc(out, "out", R, 1, Cc, bool(cfg.four_over_six))
    _need(row_amax, "row_amax", R, "f32")
    _need(status, "status", 1, "i32")
    if out is None:
        out = alloc_encoding(R, 1, Cc, x.device, bool(cfg.four_over_six), dequant)
    if row_amax is None:
        row_amax = torch.empty(R, dtype=torch.float32, device=x.device)
    o = _out(out)
    c = cfg.c()
    _check("nvfp4_quantize_per_token", lib().nvfp4_quantize_per_token(
        C.byref(c), _bf16(x, "x"), R, Cc, _dev(row_amax, "row_amax"), C.byref(o),
        _dev(status, "status"), _stream(x.device)))
    out = dict(out)
    out["row_amax"] = row_amax
    return out


def alloc_requant(slices: int, rows: int, cols: int, device, target: int,
                  four_over_six: bool = False) -> dict:
    """Outputs of nvfp4_requant_transpose for a [slices, rows, cols] source:
    the transposed [slices, cols, rows] tensor in MXFP8 or NVFP4."""
    if target == TARGET_MXFP8:
        return {"codes": torch.empty((slices, cols, rows), dtype=torch.uint8, device=device),
                "scales": torch.empty((slices, cols, rows // 32), dtype=torch.uint8,
                                      device=device),
                "choice": None}
    return alloc_encoding(slices, cols, rows, device, four_over_six, dequant=False)


@_on_input_device
def nvfp4_requant_transpose(codes: torch.Tensor, scales: torch.Tensor,
                            global_amax: torch.Tensor, src: Config | None = None,
                            dst: Config | None = None, target: int = TARGET_MXFP8,
                            out: dict | None = None,
                            status: torch.Tensor | None = None) -> dict:
    """Re-quantise a row encoding (codes [S, R, C/2], scales [S, R, C/16], as
    nvfp4_quantize wrote them under `src`) to the transposed [S, C, R] tensor in
    MXFP8 (target 0) or NVFP4 (target 1, config `dst`), rounding per `dst`."""
    src = src or Config()
    dst = dst or Config(rounding=ROUND_SR)
    if codes.dim() == 2:
        S, (R, half) = 1, codes.shape
    elif codes.dim() == 3:
        S, R, half = codes.shape
    else:
        raise ValueError("codes must be [rows, cols/2] or [slices, rows, cols/2]")
    if codes.dtype != torch.uint8 or scales.dtype != torch.uint8:
        raise TypeError("codes and scales must be uint8")
    Cc = 2 * half
    if scales.numel() != S * R * (Cc // 16):
        raise ValueError("scales must hold one byte per 16 values")
    _need(global_amax, "global_amax", S, "f32")
    _need(status, "status", 1, "i32")
    if out is not None:
        per = 1 if target == TARGET_MXFP8 else 2  # values per code byte
        _need(out["codes"], "out codes", S * R * Cc // per, "u8")
        _need(out["scales"], "out scales", S * R * Cc // (32 if target == TARGET_MXFP8 else 16), "u8")
        if target == TARGET_NVFP4 and dst.four_over_six:
            if out.get("choice") is None:
                raise ValueError("out needs a choice bitmap under Four-Over-Six")
            _need(out["choice"], "out choice", S * ((R * Cc // 16 + 31) // 32), "i32")
    if out is None:
        out = alloc_requant(S, R, Cc, codes.device, target,
                            bool(dst.four_over_six) and target == TARGET_NVFP4)
    o = _Out(_dev(out["codes"], "codes"), _dev(out["scales"], "scales"),
             _dev(out.get("choice"), "choice"), None)
    cs, cd = src.c(), dst.c()
    _check("nvfp4_requant_transpose", lib().nvfp4_requant_transpose(
        C.byref(cs), C.byref(cd), target, _dev(codes, "codes"), _dev(scales, "scales"), S, R, Cc,
        _dev(global_amax, "global_amax"), C.byref(o), _dev(status, "status"),
        _stream(codes.device)))
    return out


def alloc_mx(slices: int, rows: int, cols: int, device) -> dict:
    """Output tensors of one MXFP8 encoding of a [slices, rows, cols] input, for
    blocks of 32 along `cols` (pass the transposed dims for the columns)."""
    return {"codes": torch.empty((slices, rows, cols), dtype=torch.uint8, device=device),
            "scales": torch.empty((slices, rows, cols // 32), dtype=torch.uint8, device=device)}


@_on_input_device
def nvfp4_mx_quantize(x: torch.Tensor, cfg: Config | None = None, row: dict | None = None,
                      col: dict | None = None, status: torch.Tensor | None = None) -> dict:
    """MXFP8-encode a bf16 tensor (E8M0 scale per 32 values, E4M3 elements):
    rows and/or the transpose per cfg.blocks, RNE or stochastic per
    cfg.rounding. Returns {"row": {...}, "col": {...}} (allocated here unless
    passed in)."""
    cfg = cfg or Config(blocks=BLOCKS_BOTH, rounding=ROUND_SR)
    S, R, Cc = _shape3(x)
    for enc, name, on in ((row, "row", cfg.blocks & 1), (col, "col", cfg.blocks & 2)):
        if on and enc is not None:
            _need(enc["codes"], name + " codes", S * R * Cc, "u8")
            _need(enc["scales"], name + " scales", S * R * Cc // 32, "u8")
    _need(status, "status", 1, "i32")
    if cfg.blocks & 1 and row is None:
        row = alloc_mx(S, R, Cc, x.device)
    if cfg.blocks & 2 and col is None:
        col = alloc_mx(S, Cc, R, x.device)
    ro = _Out(_dev(row["codes"], "codes"), _dev(row["scales"], "scales"), None, None) \
        if cfg.blocks & 1 else None
    co = _Out(_dev(col["codes"], "codes"), _dev(col["scales"], "scales"), None, None) \
        if cfg.blocks & 2 else None
    c = cfg.c()
    _check("nvfp4_mx_quantize", lib().nvfp4_mx_quantize(
        C.byref(c), _bf16(x, "x"), S, R, Cc, C.byref(ro) if ro is not None else None,
        C.byref(co) if co is not None else None, _dev(status, "status"), _stream(x.device)))
    return {"row": row if cfg.blocks & 1 else None, "col": col if cfg.blocks & 2 else None}


@_on_input_device
def nvfp4_fakequant_fwd(x: torch.Tensor, s_pre: torch.Tensor, s_post: torch.Tensor | None = None,
                        out: torch.Tensor | None = None,
                        status: torch.Tensor | None = None) -> torch.Tensor:
    R, Cc = x.shape
    nb = R * Cc // 16
    _need(s_pre, "s_pre", nb, "f32")
    _need(s_post, "s_post", nb, "f32")
    _need(status, "status", 1, "i32")
    _need(out, "out", R * Cc, "bf16")
    out = torch.empty_like(x) if out is None else out
    _check("nvfp4_fakequant_fwd", lib().nvfp4_fakequant_fwd(
        _bf16(x, "x"), R, Cc, _dev(s_pre, "s_pre"), _dev(s_post, "s_post"), _bf16(out, "out"),
        _dev(status, "status"), _stream(x.device)))
    return out


@_on_input_device
def nvfp4_scale_grad_bwd(x: torch.Tensor, gq: torch.Tensor, s_pre: torch.Tensor,
                         s_post: torch.Tensor | None = None, want_gx: bool = True,
                         gx: torch.Tensor | None = None, gs_pre: torch.Tensor | None = None,
                         gs_post: torch.Tensor | None = None,
                         status: torch.Tensor | None = None) -> dict:
    R, Cc = x.shape
    nb = R * Cc // 16
    _need(s_pre, "s_pre", nb, "f32")
    _need(s_post, "s_post", nb, "f32")
    _need(status, "status", 1, "i32")
    _need(gq, "gq", R * Cc, "bf16")
    _need(gx, "gx", R * Cc, "bf16")
    _need(gs_pre, "gs_pre", nb, "f32")
    _need(gs_post, "gs_post", nb, "f32")
    if want_gx and gx is None:
        gx = torch.empty_like(x)
    gs_pre = torch.empty_like(s_pre) if gs_pre is None else gs_pre
    if s_post is not None and gs_post is None:
        gs_post = torch.empty_like(s_post)
    _check("nvfp4_scale_grad_bwd", lib().nvfp4_scale_grad_bwd(
        _bf16(x, "x"), _bf16(gq, "gq"), R, Cc, _dev(s_pre, "s_pre"), _dev(s_post, "s_post"),
        _dev(gx if want_gx else None, "gx"), _dev(gs_pre, "gs_pre"),
        _dev(gs_post if s_post is not None else None, "gs_post"), _dev(status, "status"),
        _stream(x.device)))
    return {"gx": gx if want_gx else None, "gs_pre": gs_pre,
            "gs_post": gs_post if s_post is not None else None}


@_on_input_device
def nvfp4_fakequant_fwd_fp8scale(x: torch.Tensor, s_pre: torch.Tensor,
                                 s_post: torch.Tensor | None, global_amax: torch.Tensor,
                                 out: torch.Tensor | None = None,
                                 status: torch.Tensor | None = None) -> torch.Tensor:
    """Fake quantisation at FP8-rounded block scales (global_amax: fp32 [1])."""
    R, Cc = x.shape
    nb = R * Cc // 16
    _need(s_pre, "s_pre", nb, "f32")
    _need(s_post, "s_post", nb, "f32")
    _need(status, "status", 1, "i32")
    _need(global_amax, "global_amax", 1, "f32")
    _need(out, "out", R * Cc, "bf16")
    out = torch.empty_like(x) if out is None else out
    _check("nvfp4_fakequant_fwd_fp8scale", lib().nvfp4_fakequant_fwd_fp8scale(
        _bf16(x, "x"), R, Cc, _dev(s_pre, "s_pre"), _dev(s_post, "s_post"),
        _dev(global_amax, "global_amax"), _bf16(out, "out"), _dev(status, "status"),
        _stream(x.device)))
    return out


@_on_input_device
def nvfp4_scale_grad_bwd_fp8scale(x: torch.Tensor, gq: torch.Tensor, s_pre: torch.Tensor,
                                  s_post: torch.Tensor | None, global_amax: torch.Tensor,
                                  want_gx: bool = True,
                                  status: torch.Tensor | None = None) -> dict:
    """STE backward at FP8-rounded block scales, gradients passed straight through."""
    R, Cc = x.shape
    nb = R * Cc // 16
    _need(s_pre, "s_pre", nb, "f32")
    _need(s_post, "s_post", nb, "f32")
    _need(status, "status", 1, "i32")
    _need(gq, "gq", R * Cc, "bf16")
    _need(global_amax, "global_amax", 1, "f32")
    gx = torch.empty_like(x) if want_gx else None
    gs_pre = torch.empty_like(s_pre)
    gs_post = torch.empty_like(s_post) if s_post is not None else None
    _check("nvfp4_scale_grad_bwd_fp8scale", lib().nvfp4_scale_grad_bwd_fp8scale(
        _bf16(x, "x"), _bf16(gq, "gq"), R, Cc, _dev(s_pre, "s_pre"), _dev(s_post, "s_post"),
        _dev(global_amax, "global_amax"), _dev(gx, "gx"), _dev(gs_pre, "gs_pre"),
        _dev(gs_post, "gs_post"), _dev(status, "status"), _stream(x.device)))
    return {"gx": gx, "gs_pre": gs_pre, "gs_post": gs_post}


@_on_input_device
def nvfp4_scale_init_mse(x: torch.Tensor, global_amax: torch.Tensor,
                         status: torch.Tensor | None = None) -> dict:
    """MSE scale setting over every E4M3 scale per 1x16 block: {"codes", "s"}."""
    R, Cc = x.shape
    _need(global_amax, "global_amax", 1, "f32")
    _need(status, "status", 1, "i32")
    codes = torch.empty((R, Cc // 16), dtype=torch.uint8, device=x.device)
    s = torch.empty((R, Cc // 16), dtype=torch.float32, device=x.device)
    _check("nvfp4_scale_init_mse", lib().nvfp4_scale_init_mse(
        _bf16(x, "x"), R, Cc, _dev(global_amax, "global_amax"), _dev(codes, "codes"),
        _dev(s, "s"), _dev(status, "status"), _stream(x.device)))
    return {"codes": codes, "s": s}


@_on_input_device
def nvfp4_export_scales(x: torch.Tensor, s_pre: torch.Tensor, s_post: torch.Tensor | None,
                        global_amax: torch.Tensor, out: dict | None = None,
                        status: torch.Tensor | None = None) -> dict:
    """NVFP4 row encoding carrying learned post-scales: {"codes", "scales"}."""
    R, Cc = x.shape
    nb = R * Cc // 16
    _need(s_pre, "s_pre", nb, "f32")
    _need(s_post, "s_post", nb, "f32")
    _need(status, "status", 1, "i32")
    _need(global_amax, "global_amax", 1, "f32")
    if out is not None:
        _need(out["codes"], "out codes", R * Cc // 2, "u8")
        _need(out["scales"], "out scales", nb, "u8")
    if out is None:
        out = alloc_encoding(1, R, Cc, x.device, False, dequant=False)
    o = _Out(_dev(out["codes"], "codes"), _dev(out["scales"], "scales"), None, None)
    _check("nvfp4_export_scales", lib().nvfp4_export_scales(
        _bf16(x, "x"), R, Cc, _dev(s_pre, "s_pre"), _dev(s_post, "s_post"),
        _dev(global_amax, "global_amax"), C.byref(o), _dev(status, "status"),
        _stream(x.device)))
    return out


@_on_input_device
def nvfp4_codec_probe(op: int, inp: torch.Tensor, aux: torch.Tensor | None = None,
                      out: torch.Tensor | None = None) -> torch.Tensor:
    _need(inp, "in", inp.numel(), "f32")
    _need(aux, "aux", inp.numel(), "i32")
    _need(out, "out", inp.numel(), "u8")
    out = torch.empty(inp.numel(), dtype=torch.uint8, device=inp.device) if out is None else out
    _check("nvfp4_codec_probe", lib().nvfp4_codec_probe(
        op, _dev(inp, "in"), _dev(aux, "aux"), inp.numel(), _dev(out, "out"),
        _stream(inp.device)))
    return out


def nvfp4_sr_bits(seed: int, step: int, direction: int, idx0: int, n: int,
                  device="cuda", out: torch.Tensor | None = None) -> torch.Tensor:
    _need(out, "out", n, "i32")
    out = torch.empty(n, dtype=torch.int32, device=device) if out is None else out
    with torch.cuda.device(out.device):
        _check("nvfp4_sr_bits", lib().nvfp4_sr_bits(seed & 0xFFFFFFFF, step & 0xFFFFFFFF,
                                                    direction, idx0, n, _dev(out, "out"),
                                                    _stream(out.device)))
    return out


class PeriodicAmax:
    """Periodic tensor scaling (UE5M3 blog): the global amax is recomputed on
    steps where step % period == 0 and reused, stale, in between. period = 1 is
    current tensor scaling. The cached amax lives in a caller-visible device
    buffer, so resuming means passing it back."""

    def __init__(self, period: int, slices: int = 1, device="cuda", amax_fn=None,
                 amax: torch.Tensor | None = None):
        if period < 1:
            raise ValueError("period must be >= 1")
        self.period = period
        self.valid = amax is not None
        self.amax = (amax if amax is not None
                     else torch.zeros(slices, dtype=torch.float32, device=device))
        self._fn = amax_fn or (lambda x, out: nvfp4_amax(x, out))
        self.refreshes = 0

    def __call__(self, x: torch.Tensor, step: int) -> torch.Tensor:
        if step % self.period == 0 or not self.valid:
            self.valid = True
            self._fn(x, self.amax)
            self.refreshes += 1
        return self.amax
