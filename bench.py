"""Throughput of the NVFP4 hot path on one or more GB300s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config 1..13] [--impl ours|reference]

A step is one pass of the hot path over one batch of synthetic input already
resident in HBM. The default workload is the largest one: MoE expert weights,
64 experts x 2048 x 7168 bf16 (N(0, 0.02) with 0.01 % x50 outliers), per-expert
global amax, then one pass that writes both the 1x16 row and the 16x1 column
(transposed) NVFP4 encodings with E4M3 scales, RNE, Four-Over-Six, both 4/6
bitmaps and both dequantised tensors. Other --config values time the other
workloads (see WORKLOADS); --config 13 measures the 4/6 overhead of the row
quantiser.

The K steps run as a pass bracketed by CUDA events; passes repeat back to
back until at least --min-seconds of device time have run and the median pass
is reported. One JSON line is printed by rank 0. `value` is algorithmic HBM
bytes / time (GB/s) summed over all ranks; `roofline` relates the dominant
kernel's own CUDA-event time to the measured HBM copy bandwidth (and, where a
committed ncu count exists, to the instruction-issue bound); `e2e` repeats the
metric through the same C ABI with host buffers (pinned host -> device copy of
the input and device -> host copy of every output inside the timed region);
`cpu_baseline` is the plain C oracle on the host cores, one core and all cores
(a baseline, not the target). With --impl reference the oracle itself is the
timed arm.
"""
from __future__ import annotations

import argparse
import ctypes as C
import inspect
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import nvfp4_block_scaled_02_gb300 as nv  # noqa: E402
from nvfp4_block_scaled_02_gb300 import synth  # noqa: E402

METRIC = "NVFP4 quantize/STE-bwd HBM GB/s and Gelem/s; fraction of GB300 HBM peak"
L2_BYTES = 129 * 2 ** 20
FALLBACK_HBM_GBS = 6800.0


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def sm_max_mhz() -> float:
    """The maximum SM clock: the generated peaks file, else 2070 MHz
    (GB300's maximum SM clock)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["sm_max_mhz"])
    except Exception:
        return 2070.0


def alu_peak_tops(sms: int, mhz: float) -> float:
    """ALU roofline of a kernel bound by arithmetic by definition: simple fp32
    operations per second of the whole GPU, SMs x 128 fp32 lanes x the
    maximum SM clock (an fma counted as one operation)."""
    return sms * 128 * mhz * 1e6 / 1e12


def issue_peak_ginst(sms: int, mhz: float) -> float:
    """Instruction issue rate of the whole GPU: every SM has four schedulers,
    each issuing at most one warp instruction per cycle."""
    return sms * 4 * mhz * 1e6 / 1e9



def _e2m1_rne_values(y: np.ndarray) -> np.ndarray:
    """E2M1 round-to-nearest-even of float32 values, as signed fp32 values."""
    a = np.abs(y)
    q = np.select([a <= 0.25, a < 0.75, a <= 1.25, a < 1.75, a <= 2.5, a < 3.5, a <= 5.0],
                  [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0], 6.0).astype(np.float32)
    return np.copysign(q, y)


def _sweep_sse(x: np.ndarray, d: np.ndarray, inv: np.ndarray) -> np.ndarray:
    """Each block's error sum at its own scale d (1/d = inv), in the fixed
    block order (float32 steps, the fma products taken exactly in float64)."""
    f32 = np.float32
    y = (x * inv[:, None].astype(np.float32)).astype(np.float32)
    q = _e2m1_rne_values(y)
    e = (x.astype(np.float64) - q.astype(np.float64) * d[:, None]).astype(np.float32)
    sq = e.astype(np.float64) ** 2
    out = np.zeros(len(x), f32)
    for h in (0, 8):
        acc = [np.zeros(len(x), f32), np.zeros(len(x), f32)]
        for i in range(8):
            acc[i % 2] = (sq[:, h + i] + acc[i % 2]).astype(f32)
        out = (out + (acc[0] + acc[1]).astype(f32)).astype(f32)
    return out


def sweep_candidates_per_block(w_bits: np.ndarray, gamax: float) -> float:
    """Mean number of candidate scales the MSE sweep kernel encodes per 1x16
    block of this input: the amax-derived code c0, the codes below it down to
    the first one the bound rules out against the best sum so far, and the
    codes above it up to the first all-zero code, with the kernel's steps
    replicated in float32 (the fma steps through exact float64 products). A
    work count for the roofline, not a result."""
    f32 = np.float32
    x = (np.asarray(w_bits, np.uint16).astype(np.uint32) << 16).view(np.float32).reshape(-1, 16)
    A = np.abs(x).max(axis=1)
    g = f32(f32(gamax) / f32(2688.0)) if gamax > 0 else f32(1.0)
    vals = torch.arange(127, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    d = (vals * g).astype(np.float32)
    with np.errstate(divide="ignore", over="ignore"):
        inv = np.where(d > 0, np.minimum(f32(1.0) / np.where(d > 0, d, 1), np.finfo(f32).max), 0)
        rden6 = min(f32(1.0) / f32(f32(6.0) * g), np.finfo(f32).max)
    inv = inv.astype(np.float32)
    t = np.minimum((A * f32(rden6)).astype(np.float32), f32(448.0))
    c0 = torch.from_numpy(t).to(torch.float8_e4m3fn).view(torch.uint8).numpy().astype(np.int64)
    c0 = np.clip(c0, 1, 126)
    best = _sweep_sse(x, d[c0], inv[c0])
    T = (A * f32(4.00002)).astype(np.float32)
    c_last = np.maximum(np.minimum(np.searchsorted(d[1:127], T, side="left") + 1, 126), c0)
    down = np.zeros(len(x), np.int64)
    c = c0 - 1
    active = c >= 1
    while np.any(active):  # walk down until the bound rules the code out
        cc = np.where(active, c, 1)
        m = (A.astype(np.float64) - 6.0 * d[cc]).astype(np.float32)
        lb = ((m * m).astype(np.float32) * f32(0.999996185302734375)).astype(np.float32)
        active &= ~((m > 0) & (lb > best))
        sse = _sweep_sse(x, d[cc], inv[cc])
        best = np.where(active & (sse <= best), sse, best)
        down += active
        c = c - 1
        active &= c >= 1
    return float(np.mean(1 + down + (c_last - c0)))


# ------------------------------------------------------------ workloads --

class Kernel:
    """One call of the C ABI, its algorithmic HBM bytes and the number of our
    kernels it launches (a zeroing kernel precedes the OR-ed 4/6 bitmaps of
    the column, dual and re-quantisation kernels; the global amax is one
    launch, nvfp4_amax_ws)."""

    def __init__(self, name, nbytes, fn, launches=1):
        self.name, self.nbytes, self.fn, self.launches = name, nbytes, fn, launches


class Workload:
    name = ""
    elements = 0

    def kernels(self, k: int, bufset: int) -> list:
        raise NotImplementedError


class Activation(Workload):
    """Activations [S x H] = [8192 x 4096]: amax + row quantise with 4/6."""

    def __init__(self, device, rows=8192, cols=4096, fos=1, seed=1, nsets=None, dist="t3"):
        self.rows, self.cols, self.fos = rows, cols, fos
        self.elements = rows * cols
        xb = (synth.student_t(rows, cols, seed=seed) if dist == "t3"
              else synth.outlier_normal(rows, cols, seed=seed))
        self.host_x = xb
        x0 = torch.from_numpy(xb.view(np.int16)).to(device)
        self.cfg = nv.Config(four_over_six=fos)
        out_bytes = self.elements * (0.5 + 1 / 16 + 2) + (self.elements / 16 / 8 if fos else 0)
        per_set = self.elements * 2 + out_bytes
        self.nsets = nsets or max(2, int(np.ceil(2.5 * L2_BYTES / per_set)))
        self.x = [x0] + [x0.clone() for _ in range(self.nsets - 1)]
        self.amax = [torch.empty(1, dtype=torch.float32, device=device) for _ in range(self.nsets)]
        self.out = [nv.alloc_encoding(1, rows, cols, device, bool(fos)) for _ in range(self.nsets)]
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        bpe = Activation.call_bpe(dict(fos=fos, cols=cols))
        self.q_bytes = self.elements * bpe["quantize_row"]
        self.a_bytes = self.elements * bpe["amax"]
        self.working_set = per_set * self.nsets
        self._prep(device)

    @staticmethod
    def call_bpe(kw):
        """Algorithmic HBM bytes per element of each call of a step: the amax
        pass reads x; the quantiser reads x and writes codes (1/2), scale
        bytes (1/16), the 4/6 bitmap (1/128) and the bf16 dequant (2)."""
        return {"amax": 2.0,
                "quantize_row": 2 + 0.5 + 1 / 16 + 2 + (1 / 128 if kw["fos"] else 0)}

    def _prep(self, device):
        L = nv.lib()
        self._c = self.cfg.c()
        self._outs = [nv._out(o) for o in self.out]
        st = torch.cuda.current_stream(device).cuda_stream
        R, Cc = self.rows, self.cols

        ws = nv.amax_workspace(1, self.x[0].device)
        self._ws = ws

        def amax(i):
            return L.nvfp4_amax_ws(self.x[i].data_ptr(), 1, R, Cc, self.amax[i].data_ptr(),
                                   ws.data_ptr(), ws.numel() * 4, self.status.data_ptr(), st)

        def quant(i):
            return L.nvfp4_quantize(C.byref(self._c), self.x[i].data_ptr(), 1, R, Cc,
                                    self.amax[i].data_ptr(), C.byref(self._outs[i]), None,
                                    self.status.data_ptr(), st)
        self._amax, self._quant = amax, quant

    def kernels(self, k, i):
        return [Kernel("amax", self.a_bytes, lambda: self._amax(i)),
                Kernel("quantize_row", self.q_bytes, lambda: self._quant(i))]

    def e2e_io(self, k, i):
        o = self.out[i]
        outs = [o["codes"], o["scales"], o["dequant"]] + ([o["choice"]] if self.fos else [])
        return [self.x[i]], outs

    def cpu_sample(self, budget_s):
        import oracle
        rows = 64
        t0 = time.perf_counter()
        self._cpu_once(oracle, rows)
        per_row = (time.perf_counter() - t0) / rows
        rows = int(min(self.rows, max(64, budget_s / max(per_row, 1e-9))))
        t0 = time.perf_counter()
        self._cpu_once(oracle, rows)
        dt = time.perf_counter() - t0
        return rows * self.cols, dt, f"first {rows} of {self.rows} rows (amax + quantise)"

    def _cpu_once(self, oracle, rows):
        xb = self.host_x[:rows]
        a, _ = oracle.global_amax(xb)
        oracle.quantize(xb, a, four_over_six=self.fos)

    bytes_per_elem = property(lambda self: (self.q_bytes + self.a_bytes) / self.elements)
    dominant = "quantize_row"
    workload = property(lambda self: (
        f"activation {self.rows}x{self.cols} bf16, 0.5*Student-t(nu=3); current scaling "
        f"(amax pass) + 1x16 row blocks, E4M3 scales, RNE, Four-Over-Six "
        f"{'on' if self.fos else 'off'}; outputs codes, scales, "
        f"{'4/6 bitmap, ' if self.fos else ''}dequant"))


class SmallNormal(Activation):
    """1024 x 1024 N(0,1) with 0.1 % x20 outliers, 4/6 off (L2-resident)."""

    def __init__(self, device):
        super().__init__(device, rows=1024, cols=1024, fos=0, seed=0, dist="normal")

    workload = property(lambda self: (
        "1024x1024 bf16 N(0,1), 0.1% x20 outliers; amax + 1x16 row blocks, E4M3, RNE, "
        "4/6 off; outputs codes, scales, dequant"))


class ScaleLearning(Workload):
    """Weight 14336 x 4096: fake-quant forward + STE backward with dual scales."""

    def __init__(self, device, rows=14336, cols=4096, seed=2):
        wb, gb, s = synth.scale_learning(rows, cols, seed=seed)
        self.rows, self.cols = rows, cols
        self.elements = rows * cols
        self.host = (wb, gb, s)
        per_set = self.elements * (2 + 2 + 2 + 2) + self.elements / 16 * 16
        self.nsets = max(2, int(np.ceil(2.5 * L2_BYTES / per_set)))
        w = torch.from_numpy(wb.view(np.int16)).to(device)
        g = torch.from_numpy(gb.view(np.int16)).to(device)
        sp = torch.from_numpy(s).to(device)
        self.sets = []
        for _ in range(self.nsets):
            self.sets.append(dict(w=w.clone(), g=g.clone(), sp=sp.clone(), so=sp.clone(),
                                  xq=torch.empty_like(w), gx=torch.empty_like(w),
                                  gsp=torch.empty_like(sp), gso=torch.empty_like(sp)))
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        bpe = ScaleLearning.call_bpe({})
        self.f_bytes = self.elements * bpe["fakequant_fwd"]
        self.b_bytes = self.elements * bpe["scale_grad_bwd"]
        self.working_set = per_set * self.nsets
        L = nv.lib()
        st = torch.cuda.current_stream(device).cuda_stream
        R, Cc = rows, cols

        def fwd(i):
            d = self.sets[i]
            return L.nvfp4_fakequant_fwd(d["w"].data_ptr(), R, Cc, d["sp"].data_ptr(),
                                         d["so"].data_ptr(), d["xq"].data_ptr(),
                                         self.status.data_ptr(), st)

        def bwd(i):
            d = self.sets[i]
            return L.nvfp4_scale_grad_bwd(d["w"].data_ptr(), d["g"].data_ptr(), R, Cc,
                                          d["sp"].data_ptr(), d["so"].data_ptr(),
                                          d["gx"].data_ptr(), d["gsp"].data_ptr(),
                                          d["gso"].data_ptr(), self.status.data_ptr(), st)
        self._fwd, self._bwd = fwd, bwd

    @staticmethod
    def call_bpe(kw):
        """Forward: x (2), s_pre and s_post (2 x 4 / 16), x~ (2). Backward: x and
        dL/dx~ (2 + 2), both scales (0.5), dL/dx (2), dL/ds_pre and dL/ds_post
        (0.5)."""
        return {"fakequant_fwd": 4.5, "scale_grad_bwd": 7.0}

    def kernels(self, k, i):
        return [Kernel("fakequant_fwd", self.f_bytes, lambda: self._fwd(i)),
                Kernel("scale_grad_bwd", self.b_bytes, lambda: self._bwd(i))]

    def e2e_io(self, k, i):
        d = self.sets[i]
        return [d["w"], d["g"], d["sp"], d["so"]], [d["xq"], d["gx"], d["gsp"], d["gso"]]

    def cpu_sample(self, budget_s):
        import oracle
        wb, gb, s = self.host
        rows = 256
        t0 = time.perf_counter()
        oracle.fakequant_fwd(wb[:rows], s[:rows], s[:rows])
        oracle.scale_grad_bwd(wb[:rows], gb[:rows], s[:rows], s[:rows])
        per_row = (time.perf_counter() - t0) / rows
        rows = int(min(self.rows, max(256, budget_s / max(per_row, 1e-9))))
        t0 = time.perf_counter()
        oracle.fakequant_fwd(wb[:rows], s[:rows], s[:rows])
        oracle.scale_grad_bwd(wb[:rows], gb[:rows], s[:rows], s[:rows])
        return rows * self.cols, time.perf_counter() - t0, \
            f"first {rows} of {self.rows} rows (forward + backward)"

    bytes_per_elem = property(lambda self: (self.f_bytes + self.b_bytes) / self.elements)
    dominant = "scale_grad_bwd"
    workload = property(lambda self: (
        f"scale-learning step on weight {self.rows}x{self.cols} bf16 N(0,0.02), dual fp32 "
        "per-block scales (init amax/6), dL/dx~ N(0,1e-3): fake-quant forward + STE backward "
        "(dL/dx, dL/ds_pre, dL/ds_post)"))


class DriftingGradient(Workload):
    """Gradients 16384 x 4096, UE5M3, stochastic rounding, periodic scaling
    (amax refreshed every 16 steps), rows drifting x1.05 per step."""

    def __init__(self, device, rows=16384, cols=4096, seed=3, period=16, nsteps=32):
        gen = synth.DriftingGradient(rows, cols, seed=seed)
        self.rows, self.cols, self.period = rows, cols, period
        self.elements = rows * cols
        self.host0 = gen.step(0)
        self.x = [torch.from_numpy(gen.step(t).view(np.int16)).to(device) for t in range(nsteps)]
        self.nsets = nsteps
        self.amax = torch.empty(1, dtype=torch.float32, device=device)
        self.out = [nv.alloc_encoding(1, rows, cols, device, False, dequant=False)
                    for _ in range(2)]
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        bpe = self.call_bpe({})
        self.q_bytes = self.elements * bpe["quantize_row_sr"]
        self.a_bytes = self.elements * bpe["amax"]
        self.working_set = self.elements * 2 * nsteps
        L = nv.lib()
        st = torch.cuda.current_stream(device).cuda_stream
        self._outs = [nv._out(o) for o in self.out]
        self._cfgs = [nv.Config(scale_fmt=1, rounding=1, scale_max=448.0, seed=3, step=t).c()
                      for t in range(nsteps)]

        ws = nv.amax_workspace(1, device)
        self._ws = ws

        def amax(t):
            return L.nvfp4_amax_ws(self.x[t].data_ptr(), 1, rows, cols, self.amax.data_ptr(),
                                   ws.data_ptr(), ws.numel() * 4, self.status.data_ptr(), st)

        def quant(t):
            return L.nvfp4_quantize(C.byref(self._cfgs[t]), self.x[t].data_ptr(), 1, rows, cols,
                                    self.amax.data_ptr(), C.byref(self._outs[t % 2]), None,
                                    self.status.data_ptr(), st)
        self._amax, self._quant = amax, quant

    @staticmethod
    def call_bpe(kw):
        """amax on refresh steps (x, 2); every step x (2), codes (1/2), scale
        bytes (1/16); no dequant."""
        return {"amax": 2.0, "quantize_row_sr": 2 + 0.5 + 1 / 16}

    def kernels(self, k, i):
        t = k % self.nsets
        ks = []
        if t % self.period == 0:
            ks.append(Kernel("amax", self.a_bytes, lambda: self._amax(t)))
        ks.append(Kernel("quantize_row_sr", self.q_bytes, lambda: self._quant(t)))
        return ks

    def e2e_io(self, k, i):  # the step picks its own buffers: input t, output t % 2
        t = k % self.nsets
        o = self.out[t % 2]
        return [self.x[t]], [o["codes"], o["scales"]]

    def cpu_sample(self, budget_s):
        import oracle
        rows = 64
        xb = self.host0
        a, _ = oracle.global_amax(xb[:rows])
        t0 = time.perf_counter()
        oracle.quantize(xb[:rows], a, scale_fmt=1, rounding=1, seed=3, step=0, dequant=False)
        per_row = (time.perf_counter() - t0) / rows
        rows = int(min(self.rows, max(64, budget_s / max(per_row, 1e-9))))
        t0 = time.perf_counter()
        oracle.quantize(xb[:rows], a, scale_fmt=1, rounding=1, seed=3, step=0, dequant=False)
        return rows * self.cols, time.perf_counter() - t0, f"first {rows} of {self.rows} rows"

    bytes_per_elem = property(lambda self: (self.q_bytes + self.a_bytes / self.period)
                              / self.elements)
    dominant = "quantize_row_sr"
    workload = property(lambda self: (
        f"gradient {self.rows}x{self.cols} bf16 N(0,1) x per-row lognormal(0,2), drifting "
        f"x1.05/step over {self.nsets} steps; UE5M3 scales, periodic scaling (amax every "
        f"{self.period} steps), stochastic E2M1 rounding (Philox4x32-10, key seed/step); "
        "outputs codes, scales"))


class MoeExperts(Workload):
    """64 experts x 2048 x 7168: per-expert amax + one pass emitting row and
    column NVFP4 encodings with 4/6 and both dequants. The input is larger
    than L2, so the device-timed steps use one buffer set; the end-to-end run
    uses two (e2e_sets), so one step's copies overlap its neighbours'."""

    e2e_sets = 2

    def __init__(self, device, experts=64, rows=2048, cols=7168, seed=4):
        xb = synth.moe_experts(experts, rows, cols, seed=seed)
        self.S, self.rows, self.cols = experts, rows, cols
        self.elements = experts * rows * cols
        self.host_x = xb
        self.device = device
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.cfg = nv.Config(blocks=3, four_over_six=1)
        self._c = self.cfg.c()
        self._ws = nv.amax_workspace(experts, device)
        self._sets = [self._make_set(torch.from_numpy(xb.view(np.int16)).to(device))]
        del xb
        self.x, self.amax = self._sets[0]["x"], self._sets[0]["amax"]
        self.row, self.col = self._sets[0]["row"], self._sets[0]["col"]
        bpe = self.call_bpe({})
        self.d_bytes = self.elements * bpe["quantize_dual"]
        self.a_bytes = self.elements * bpe["amax"]
        self.nsets = 1
        self.working_set = self.elements * (2 + 2 * 4.57)

    def _make_set(self, x):
        """Device buffers of one step (input, per-expert amax, both encodings)
        and its two calls through the C ABI."""
        E, R, Cc = self.S, self.rows, self.cols
        b = {"x": x, "amax": torch.empty(E, dtype=torch.float32, device=self.device),
             "row": nv.alloc_encoding(E, R, Cc, self.device, True),
             "col": nv.alloc_encoding(E, Cc, R, self.device, True)}
        r, cc = nv._out(b["row"]), nv._out(b["col"])
        L = nv.lib()
        st = torch.cuda.current_stream(self.device).cuda_stream
        ws = self._ws

        def amax():
            return L.nvfp4_amax_ws(x.data_ptr(), E, R, Cc, b["amax"].data_ptr(), ws.data_ptr(),
                                   ws.numel() * 4, self.status.data_ptr(), st)

        def dual():
            return L.nvfp4_quantize(C.byref(self._c), x.data_ptr(), E, R, Cc,
                                    b["amax"].data_ptr(), C.byref(r), C.byref(cc),
                                    self.status.data_ptr(), st)
        b["_refs"] = (r, cc)
        b["amax_fn"], b["dual_fn"] = amax, dual
        return b

    def _set(self, i):
        while len(self._sets) <= i:  # the end-to-end run's second set, made on first use
            self._sets.append(self._make_set(torch.empty_like(self.x)))
        return self._sets[i]

    @staticmethod
    def call_bpe(kw):
        """amax reads x (2); the dual pass reads x once (2) and writes, for each
        of the row and column encodings, codes (1/2), scale bytes (1/16), the
        4/6 bitmap (1/128) and the bf16 dequant (2)."""
        return {"amax": 2.0, "quantize_dual": 2 + 2 * (0.5 + 1 / 16 + 1 / 128 + 2)}

    def kernels(self, k, i):
        b = self._set(i)
        return [Kernel("amax", self.a_bytes, b["amax_fn"]),
                Kernel("quantize_dual", self.d_bytes, b["dual_fn"], 3)]

    def e2e_io(self, k, i):
        b = self._set(i)
        names = ("codes", "scales", "choice", "dequant")
        outs = [b["row"][n] for n in names] + [b["col"][n] for n in names]
        return [b["x"]], outs

    def cpu_sample(self, budget_s):
        import oracle
        xb = self.host_x[0]
        rows = 16
        a, _ = oracle.global_amax(xb[:rows])
        t0 = time.perf_counter()
        oracle.quantize(xb[:rows], a, blocks=3, four_over_six=1)
        per_row = (time.perf_counter() - t0) / rows
        rows = int(min(self.rows, max(16, budget_s / max(per_row, 1e-9))))
        rows -= rows % 16
        t0 = time.perf_counter()
        a, _ = oracle.global_amax(xb[:rows])
        oracle.quantize(xb[:rows], a, blocks=3, four_over_six=1)
        return rows * self.cols, time.perf_counter() - t0, \
            f"first {rows} rows of expert 0 (amax + row and column encodings)"

    bytes_per_elem = property(lambda self: (self.d_bytes + self.a_bytes) / self.elements)
    dominant = "quantize_dual"
    workload = property(lambda self: (
        f"MoE expert weights {self.S} x {self.rows}x{self.cols} bf16 N(0,0.02), 0.01% x50 "
        "outliers; per-expert amax + one pass emitting 1x16 row and 16x1 column encodings, "
        "E4M3, RNE, Four-Over-Six on, both dequants"))


class PerTokenActivation(Activation):
    """The activation tensor with per-token outer scales: one kernel computes
    every row's amax and encodes the row (x read from HBM once)."""

    def __init__(self, device):
        super().__init__(device)
        L = nv.lib()
        st = torch.cuda.current_stream(device).cuda_stream
        R, Cc = self.rows, self.cols
        self.row_amax = [torch.empty(R, dtype=torch.float32, device=device)
                         for _ in range(self.nsets)]
        self.out = [nv.alloc_encoding(R, 1, Cc, device, bool(self.fos)) for _ in range(self.nsets)]
        self._touts = [nv._out(o) for o in self.out]
        self.t_bytes = self.elements * PerTokenActivation.call_bpe(dict(cols=Cc))["quantize_per_token"]

        def tok(i):
            return L.nvfp4_quantize_per_token(C.byref(self._c), self.x[i].data_ptr(), R, Cc,
                                              self.row_amax[i].data_ptr(),
                                              C.byref(self._touts[i]), self.status.data_ptr(), st)
        self._tok = tok

    @staticmethod
    def call_bpe(kw):
        """The row quantiser's bytes with 4/6 and dequant, plus the fp32 row
        amax (4 bytes per row of `cols` elements)."""
        return {"quantize_per_token": 2 + 0.5 + 1 / 16 + 1 / 128 + 2 + 4 / kw["cols"]}

    def kernels(self, k, i):
        return [Kernel("quantize_per_token", self.t_bytes, lambda: self._tok(i))]

    def e2e_io(self, k, i):
        o = self.out[i]
        return [self.x[i]], [o["codes"], o["scales"], o["dequant"], o["choice"], self.row_amax[i]]

    def _cpu_once(self, oracle, rows):
        xb = self.host_x[:rows].reshape(rows, 1, self.cols)
        a, _ = oracle.global_amax(xb, rows)
        oracle.quantize(xb, a, four_over_six=self.fos)

    bytes_per_elem = property(lambda self: self.t_bytes / self.elements)
    dominant = "quantize_per_token"
    workload = property(lambda self: (
        f"activation {self.rows}x{self.cols} bf16, 0.5*Student-t(nu=3); per-token outer scales "
        "(row amax and encoding in one pass), 1x16 row blocks, E4M3, RNE, Four-Over-Six on; "
        "outputs codes, scales, 4/6 bitmap, dequant, row amax"))


class RequantActivation(Workload):
    """The activation tensor's forward NVFP4 encoding (4/6 on, written once,
    untimed) re-quantised for the backward pass: de-quantise, transpose,
    stochastic rounding to MXFP8 (E4M3 values, E8M0 scale per 32)."""

    def __init__(self, device, rows=8192, cols=4096, seed=1, target=0):
        self.rows, self.cols, self.target = rows, cols, target
        self.elements = rows * cols
        xb = synth.student_t(rows, cols, seed=seed)
        self.host_x = xb
        x = torch.from_numpy(xb.view(np.int16)).to(device)
        self.gamax = nv.nvfp4_amax(x)
        self.src_cfg = nv.Config(four_over_six=1)
        enc = nv.nvfp4_quantize(x, self.gamax, self.src_cfg, dequant=False)["row"]
        del x
        torch.cuda.synchronize()
        self.dst_cfg = nv.Config(rounding=1, seed=7, step=0, four_over_six=int(target == 1))
        in_bytes = self.elements * (0.5 + 1 / 16)
        out_bytes = self.elements * ((1 + 1 / 32) if target == 0 else (0.5 + 1 / 16 + 1 / 128))
        per_set = in_bytes + out_bytes
        self.nsets = max(2, int(np.ceil(2.5 * L2_BYTES / per_set)))
        self.codes = [enc["codes"]] + [enc["codes"].clone() for _ in range(self.nsets - 1)]
        self.scales = [enc["scales"]] + [enc["scales"].clone() for _ in range(self.nsets - 1)]
        self.out = [nv.alloc_requant(1, rows, cols, device, target, target == 1)
                    for _ in range(self.nsets)]
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.r_bytes = self.elements * sum(self.call_bpe(dict(target=target)).values())
        self.working_set = per_set * self.nsets
        L = nv.lib()
        st = torch.cuda.current_stream(device).cuda_stream
        self._s, self._d = self.src_cfg.c(), self.dst_cfg.c()
        self._outs = [nv._Out(o["codes"].data_ptr(), o["scales"].data_ptr(),
                              o["choice"].data_ptr() if o.get("choice") is not None else None,
                              None) for o in self.out]

        def rq(i):
            return L.nvfp4_requant_transpose(C.byref(self._s), C.byref(self._d), target,
                                             self.codes[i].data_ptr(), self.scales[i].data_ptr(),
                                             1, rows, cols, self.gamax.data_ptr(),
                                             C.byref(self._outs[i]), self.status.data_ptr(), st)
        self._rq = rq
        self.dominant = "requant_mxfp8_sr" if target == 0 else "requant_nvfp4_sr"

    @staticmethod
    def call_bpe(kw):
        """Reads the source codes (1/2) and scale bytes (1/16); writes MXFP8
        codes (1) and E8M0 scales (1/32), or NVFP4 codes (1/2), scale bytes
        (1/16) and the 4/6 bitmap (1/128)."""
        if kw["target"] == 0:
            return {"requant_mxfp8_sr": 0.5 + 1 / 16 + 1 + 1 / 32}
        return {"requant_nvfp4_sr": 0.5 + 1 / 16 + 0.5 + 1 / 16 + 1 / 128}

    def kernels(self, k, i):
        return [Kernel(self.dominant, self.r_bytes, lambda: self._rq(i), 2 if self.target == 1 else 1)]

    def e2e_io(self, k, i):
        o = self.out[i]
        outs = [o["codes"], o["scales"]] + ([o["choice"]] if self.target == 1 else [])
        return [self.codes[i], self.scales[i], self.gamax], outs

    def cpu_sample(self, budget_s):
        import oracle
        rows = 32
        xb = self.host_x
        a, _ = oracle.global_amax(xb)
        q = oracle.quantize(xb[:1024], a, four_over_six=1, dequant=False)

        def once(n):
            t0 = time.perf_counter()
            oracle.requant(q["row_codes"][:, :n], q["row_scales"][:, :n], a, target=self.target,
                           rounding=1, seed=7, src_fos=1, dst_fos=int(self.target == 1))
            return time.perf_counter() - t0
        per_row = once(rows) / rows
        rows = int(min(1024, max(32, budget_s / max(per_row, 1e-9))))
        rows -= rows % 32
        return rows * self.cols, once(rows), \
            f"first {rows} of {self.rows} source rows (de-quantise, transpose, re-quantise)"

    bytes_per_elem = property(lambda self: self.r_bytes / self.elements)
    workload = property(lambda self: (
        f"activation {self.rows}x{self.cols} bf16, 0.5*Student-t(nu=3), forward NVFP4 row "
        "encoding (E4M3 scales, Four-Over-Six) re-quantised for the backward GEMM: de-quantise, "
        "transpose, stochastic rounding to "
        + ("MXFP8 (E4M3, E8M0 scale per 32)" if self.target == 0 else
           "NVFP4 (E4M3 scales, Four-Over-Six)") + "; outputs codes, scales"))


class ScaleLearningFp8(ScaleLearning):
    """Workload 3's scale-learning step with FP8 block scales: fake-quant
    forward and STE backward at the E4M3-rounded dual scales, the gradients
    passed straight through."""

    def __init__(self, device, rows=14336, cols=4096, seed=2):
        super().__init__(device, rows, cols, seed)
        wb = self.host[0]
        gam = float(np.abs(synth.bf16_bits_to_f32(wb)).max())
        self.gamax = torch.tensor([gam * 1.5], dtype=torch.float32, device=device)
        L = nv.lib()
        st = torch.cuda.current_stream(device).cuda_stream
        R, Cc = rows, cols

        def fwd(i):
            d = self.sets[i]
            return L.nvfp4_fakequant_fwd_fp8scale(d["w"].data_ptr(), R, Cc, d["sp"].data_ptr(),
                                                  d["so"].data_ptr(), self.gamax.data_ptr(),
                                                  d["xq"].data_ptr(), self.status.data_ptr(), st)

        def bwd(i):
            d = self.sets[i]
            return L.nvfp4_scale_grad_bwd_fp8scale(
                d["w"].data_ptr(), d["g"].data_ptr(), R, Cc, d["sp"].data_ptr(),
                d["so"].data_ptr(), self.gamax.data_ptr(), d["gx"].data_ptr(),
                d["gsp"].data_ptr(), d["gso"].data_ptr(), self.status.data_ptr(), st)
        self._fwd, self._bwd = fwd, bwd

    @staticmethod
    def call_bpe(kw):
        """As the fp32-scale step (the FP8 outer amax is one float)."""
        return {"fakequant_fwd_fp8": 4.5, "scale_grad_bwd_fp8": 7.0}

    def kernels(self, k, i):
        return [Kernel("fakequant_fwd_fp8", self.f_bytes, lambda: self._fwd(i)),
                Kernel("scale_grad_bwd_fp8", self.b_bytes, lambda: self._bwd(i))]

    def cpu_sample(self, budget_s):
        import oracle
        wb, gb, s = self.host
        gam = float(self.gamax.item())
        rows = 256
        t0 = time.perf_counter()
        oracle.fakequant_fwd_fp8(wb[:rows], s[:rows], s[:rows], gam)
        oracle.scale_grad_bwd_fp8(wb[:rows], gb[:rows], s[:rows], s[:rows], gam)
        per_row = (time.perf_counter() - t0) / rows
        rows = int(min(self.rows, max(256, budget_s / max(per_row, 1e-9))))
        t0 = time.perf_counter()
        oracle.fakequant_fwd_fp8(wb[:rows], s[:rows], s[:rows], gam)
        oracle.scale_grad_bwd_fp8(wb[:rows], gb[:rows], s[:rows], s[:rows], gam)
        return rows * self.cols, time.perf_counter() - t0, \
            f"first {rows} of {self.rows} rows (forward + backward, FP8 scales)"

    dominant = "scale_grad_bwd_fp8"
    workload = property(lambda self: (
        f"scale-learning step on weight {self.rows}x{self.cols} bf16 N(0,0.02) with FP8 "
        "(E4M3) dual block scales in units of 1.5*amax/2688 (init amax/6, jittered): fake-quant "
        "forward + STE backward at the rounded scales, gradients passed straight through"))


class ScaleInitExport(ScaleLearningFp8):
    """MSE scale setting over every E4M3 scale of each block, then the export
    of the (post-)scales to an NVFP4 encoding, on workload 3's weight."""

    def __init__(self, device, rows=14336, cols=4096, seed=2):
        super().__init__(device, rows, cols, seed)
        L = nv.lib()
        st = torch.cuda.current_stream(device).cuda_stream
        R, Cc = rows, cols
        for d in self.sets:
            d["codes"] = torch.empty((R, Cc // 16), dtype=torch.uint8, device=device)
            d["enc"] = nv.alloc_encoding(1, R, Cc, device, False, dequant=False)
            d["eo"] = nv._Out(d["enc"]["codes"].data_ptr(), d["enc"]["scales"].data_ptr(), None,
                              None)
        bpe = self.call_bpe({})
        self.i_bytes = self.elements * bpe["scale_init_mse"]
        self.e_bytes = self.elements * bpe["export_scales"]

        def init(i):
            d = self.sets[i]
            return L.nvfp4_scale_init_mse(d["w"].data_ptr(), R, Cc, self.gamax.data_ptr(),
                                          d["codes"].data_ptr(), d["sp"].data_ptr(),
                                          self.status.data_ptr(), st)

        def export(i):
            d = self.sets[i]
            return L.nvfp4_export_scales(d["w"].data_ptr(), R, Cc, d["sp"].data_ptr(),
                                         d["so"].data_ptr(), self.gamax.data_ptr(),
                                         C.byref(d["eo"]), self.status.data_ptr(), st)
        self._init, self._export = init, export

    @staticmethod
    def call_bpe(kw):
        """Sweep: x (2), scale codes (1/16), fp32 scales (4/16). Export: x (2),
        both fp32 scales (0.5), codes (1/2), scale bytes (1/16)."""
        return {"scale_init_mse": 2 + 1 / 16 + 4 / 16, "export_scales": 2 + 0.5 + 0.5 + 1 / 16}

    def kernels(self, k, i):
        return [Kernel("scale_init_mse", self.i_bytes, lambda: self._init(i)),
                Kernel("export_scales", self.e_bytes, lambda: self._export(i))]

    def e2e_io(self, k, i):
        d = self.sets[i]
        return [d["w"], d["so"]], [d["codes"], d["sp"], d["enc"]["codes"], d["enc"]["scales"]]

    def cpu_sample(self, budget_s):
        import oracle
        wb, _, s = self.host
        gam = float(self.gamax.item())
        rows = 4
        t0 = time.perf_counter()
        oracle.scale_init_mse(wb[:rows], gam)
        per_row = (time.perf_counter() - t0) / rows
        rows = int(min(self.rows, max(4, budget_s / max(per_row, 1e-9))))
        t0 = time.perf_counter()
        oracle.scale_init_mse(wb[:rows], gam)
        oracle.export_scales(wb[:rows], s[:rows], s[:rows], gam)
        return rows * self.cols, time.perf_counter() - t0, \
            f"first {rows} of {self.rows} rows (MSE sweep over 126 E4M3 scales + export)"

    bytes_per_elem = property(lambda self: (self.i_bytes + self.e_bytes) / self.elements)
    # the sweep's arithmetic: per element and evaluated candidate scale one
    # scaling multiply, one E2M1 rounding, one decode, the error fma and the
    # square-accumulate fma; the kernel evaluates only the candidates that can
    # win (counted on this input by sweep_candidates_per_block)
    alu_ops_per_elem = property(lambda self: {"scale_init_mse": round(5 * self.candidates_per_block, 2)})
    dominant = "scale_init_mse"

    @property
    def candidates_per_block(self):
        if not hasattr(self, "_cands"):
            # every 8th row: the same distribution of blocks, an eighth of the host time
            self._cands = round(sweep_candidates_per_block(self.host[0][::8],
                                                           float(self.gamax.item())), 2)
        return self._cands
    workload = property(lambda self: (
        f"weight {self.rows}x{self.cols} bf16 N(0,0.02): MSE scale setting over all 126 E4M3 "
        "scales per 1x16 block (codes + fp32 scales), then export of the post-scales to an "
        "NVFP4 row encoding (codes + E4M3 scale bytes)"))


class TileWeight(Workload):
    """Weight 14336 x 4096: amax + one scale per 16x16 tile, the row encoding
    and its transpose (codes, scales, both dequants) from one read."""

    def __init__(self, device, rows=14336, cols=4096, seed=2):
        wb, _, _ = synth.scale_learning(rows, cols, seed=seed)
        self.rows, self.cols = rows, cols
        self.elements = rows * cols
        self.host_x = wb
        x0 = torch.from_numpy(wb.view(np.int16)).to(device)
        per_set = self.elements * (2 + 2 * (0.5 + 1 / 16 + 2))
        self.nsets = max(2, int(np.ceil(2.5 * L2_BYTES / per_set)))
        self.x = [x0] + [x0.clone() for _ in range(self.nsets - 1)]
        self.amax = [torch.empty(1, dtype=torch.float32, device=device) for _ in range(self.nsets)]
        self.row = [nv.alloc_encoding(1, rows, cols, device, False) for _ in range(self.nsets)]
        self.col = [nv.alloc_encoding(1, cols, rows, device, False) for _ in range(self.nsets)]
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        bpe = self.call_bpe({})
        self.t_bytes = self.elements * bpe["quantize_tile16"]
        self.a_bytes = self.elements * bpe["amax"]
        self.working_set = per_set * self.nsets
        L = nv.lib()
        st = torch.cuda.current_stream(device).cuda_stream
        self._c = nv.Config(blocks=nv.BLOCKS_TILE16).c()
        self._ro = [nv._out(o) for o in self.row]
        self._co = [nv._out(o) for o in self.col]

        ws = nv.amax_workspace(1, device)
        self._ws = ws

        def amax(i):
            return L.nvfp4_amax_ws(self.x[i].data_ptr(), 1, rows, cols, self.amax[i].data_ptr(),
                                   ws.data_ptr(), ws.numel() * 4, self.status.data_ptr(), st)

        def tile(i):
            return L.nvfp4_quantize(C.byref(self._c), self.x[i].data_ptr(), 1, rows, cols,
                                    self.amax[i].data_ptr(), C.byref(self._ro[i]),
                                    C.byref(self._co[i]), self.status.data_ptr(), st)
        self._amax, self._tile = amax, tile

    @staticmethod
    def call_bpe(kw):
        """amax (2); the tile pass reads x (2) and writes, for the row encoding
        and its transpose, codes (1/2), a scale byte per 16 (1/16: a tile's
        scale is stored once per 16-value row block) and the dequant (2)."""
        return {"amax": 2.0, "quantize_tile16": 2 + 2 * (0.5 + 1 / 16 + 2)}

    def kernels(self, k, i):
        return [Kernel("amax", self.a_bytes, lambda: self._amax(i)),
                Kernel("quantize_tile16", self.t_bytes, lambda: self._tile(i))]

    def e2e_io(self, k, i):
        names = ("codes", "scales", "dequant")
        return [self.x[i]], [self.row[i][n] for n in names] + [self.col[i][n] for n in names]

    def cpu_sample(self, budget_s):
        import oracle
        rows = 16
        t0 = time.perf_counter()
        a, _ = oracle.global_amax(self.host_x[:rows])
        oracle.quantize_tile16(self.host_x[:rows], a)
        per_row = (time.perf_counter() - t0) / rows
        rows = int(min(self.rows, max(16, budget_s / max(per_row, 1e-9))))
        rows -= rows % 16
        t0 = time.perf_counter()
        a, _ = oracle.global_amax(self.host_x[:rows])
        oracle.quantize_tile16(self.host_x[:rows], a)
        return rows * self.cols, time.perf_counter() - t0, \
            f"first {rows} of {self.rows} rows (amax + 16x16 tile encoding and transpose)"

    bytes_per_elem = property(lambda self: (self.t_bytes + self.a_bytes) / self.elements)
    dominant = "quantize_tile16"
    workload = property(lambda self: (
        f"weight {self.rows}x{self.cols} bf16 N(0,0.02): amax + one E4M3 scale per 16x16 tile "
        "(RNE), row encoding and its transpose with both dequants from one read"))


class GradientMx(Workload):
    """The 16384 x 4096 gradient quantised to MXFP8 for the backward GEMMs: rows
    (for DGRAD) and the transpose (for WGRAD) from one read, E8M0 scale per 32,
    E4M3 elements by stochastic rounding."""

    def __init__(self, device, rows=16384, cols=4096, seed=3):
        gen = synth.DriftingGradient(rows, cols, seed=seed)
        self.rows, self.cols = rows, cols
        self.elements = rows * cols
        self.m_bytes = self.elements * self.call_bpe({})["mx_quantize_sr"]
        self.nsets = max(2, int(np.ceil(2.5 * L2_BYTES / self.m_bytes)))
        self.host0 = gen.step(0)
        self.x = [torch.from_numpy(gen.step(t).view(np.int16)).to(device)
                  for t in range(self.nsets)]
        self.row = [nv.alloc_mx(1, rows, cols, device) for _ in range(self.nsets)]
        self.col = [nv.alloc_mx(1, cols, rows, device) for _ in range(self.nsets)]
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.working_set = self.m_bytes * self.nsets
        L = nv.lib()
        st = torch.cuda.current_stream(device).cuda_stream
        self._cfgs = [nv.Config(blocks=nv.BLOCKS_BOTH, rounding=1, seed=12, step=t).c()
                      for t in range(64)]
        self._ro = [nv._Out(o["codes"].data_ptr(), o["scales"].data_ptr(), None, None)
                    for o in self.row]
        self._co = [nv._Out(o["codes"].data_ptr(), o["scales"].data_ptr(), None, None)
                    for o in self.col]

        def mx(k, i):
            return L.nvfp4_mx_quantize(C.byref(self._cfgs[k % 64]), self.x[i].data_ptr(), 1, rows,
                                       cols, C.byref(self._ro[i]), C.byref(self._co[i]),
                                       self.status.data_ptr(), st)
        self._mx = mx

    @staticmethod
    def call_bpe(kw):
        """x (2); rows and transpose: E4M3 codes (1) and E8M0 scales (1/32) each."""
        return {"mx_quantize_sr": 2 + 2 * (1 + 1 / 32)}

    def kernels(self, k, i):
        return [Kernel("mx_quantize_sr", self.m_bytes, lambda: self._mx(k, i))]

    def e2e_io(self, k, i):
        return [self.x[i]], [self.row[i]["codes"], self.row[i]["scales"], self.col[i]["codes"],
                             self.col[i]["scales"]]

    def cpu_sample(self, budget_s):
        import oracle
        rows = 32

        def once(n):
            t0 = time.perf_counter()
            oracle.mx_quantize(self.host0[:n], blocks=3, rounding=1, seed=12, step=0)
            return time.perf_counter() - t0
        per_row = once(rows) / rows
        rows = int(min(self.rows, max(32, budget_s / max(per_row, 1e-9))))
        rows -= rows % 32
        return rows * self.cols, once(rows), \
            f"first {rows} of {self.rows} rows (MXFP8 rows and transpose, stochastic rounding)"

    bytes_per_elem = property(lambda self: self.m_bytes / self.elements)
    dominant = "mx_quantize_sr"
    workload = property(lambda self: (
        f"gradient {self.rows}x{self.cols} bf16 N(0,1) x per-row lognormal(0,2) quantised to "
        "MXFP8 for the backward GEMMs: rows and the transpose from one read, E8M0 scale per 32, "
        "E4M3 elements by stochastic rounding (Philox4x32-10, key seed/step); outputs codes, "
        "scales"))


class RequantActivationNvfp4(RequantActivation):
    def __init__(self, device):
        super().__init__(device, target=1)


WORKLOADS = {1: SmallNormal, 2: Activation, 3: ScaleLearning, 4: DriftingGradient,
             5: MoeExperts, 6: PerTokenActivation, 7: RequantActivation,
             8: RequantActivationNvfp4, 9: ScaleLearningFp8, 10: ScaleInitExport,
             11: TileWeight, 12: GradientMx}


# constructor arguments fixed by subclasses whose __init__ takes none
_CTOR_FIXED = {SmallNormal: dict(rows=1024, cols=1024, fos=0),
               RequantActivationNvfp4: dict(target=1)}


def _ctor_args(config, args):
    """The sizes and options the workload of `config` is built with: its
    constructors' defaults, subclass-fixed arguments and the command line's."""
    cls = WORKLOADS[config]
    kw = {}
    for k in reversed(cls.__mro__):
        init = k.__dict__.get("__init__")
        if init is not None and k is not object:
            for name, prm in inspect.signature(init).parameters.items():
                if prm.default is not inspect.Parameter.empty:
                    kw[name] = prm.default
    kw.update(_CTOR_FIXED.get(cls, {}))
    kw.update({5: dict(experts=args.experts), 4: dict(nsteps=args.sr_steps)}.get(config, {}))
    return kw


def describe_workload(config, args):
    """The `workload` text of `config` without building it on a device (the
    reference arm reports the same workload as ours)."""
    cls = WORKLOADS[config]
    kw = _ctor_args(config, args)
    stub = cls.__new__(cls)
    stub.rows, stub.cols = kw.get("rows"), kw.get("cols")
    stub.fos, stub.target = kw.get("fos", 1), kw.get("target", 0)
    stub.nsets, stub.period, stub.S = kw.get("nsteps"), kw.get("period"), kw.get("experts")
    return stub.workload


# Four-Over-Six overhead of the row quantiser: the 4/6 pages' one published
# figure for this path is an overhead below 2 % at S <= 2048 tokens and below
# 15 % at S = 8192 on their Blackwell kernel.
FOS_OVERHEAD = 13
FOS_PAGES = "4/6 overhead < 2 % at S <= 2048 and < 15 % at S = 8192 (Four Over Six, Blackwell)"


def fos_overhead(args, device):
    """Row quantiser on activations [S x 4096] (0.5 * Student-t(3)), S = 2048
    and 8192, with and without the dequantised output, 4/6 off and on: each
    variant timed alone as back-to-back calls over rotating buffer sets larger
    than L2 (median of repeated passes, events at the pass ends only)."""
    import math
    steps = args.steps or 50
    out, tot_b, tot_ms = [], 0.0, 0.0
    for rows in (2048, 8192):
        for dq in (True, False):
            us = {}
            for fos in (0, 1):
                wl = Activation(device, rows=rows, fos=fos)
                if not dq:
                    for o in wl._outs:
                        o.dequant = None
                def call(i, wl=wl):
                    return wl._quant(i)
                for i in range(wl.nsets):  # each set's global amax, once (untimed)
                    if wl._amax(i) != 0:
                        raise nv.Nvfp4Error("amax", 1)
                for k in range(args.warmup):
                    call(k % wl.nsets)
                torch.cuda.synchronize()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                passes, npass = [], None
                while npass is None or len(passes) < npass:
                    torch.cuda.synchronize()
                    a.record()
                    for k in range(steps):
                        rc = call(k % wl.nsets)
                        if rc != 0:
                            raise nv.Nvfp4Error("quantize_row", rc)
                    b.record()
                    torch.cuda.synchronize()
                    passes.append(a.elapsed_time(b))
                    if npass is None:
                        npass = min(max(3, math.ceil(0.25e3 / max(passes[0], 1e-3))), 2000)
                if int(wl.status.item()) != 0:
                    raise RuntimeError("device status set")
                ms = statistics.median(passes) / steps
                bpe = 2 + 0.5 + 1 / 16 + (2 if dq else 0) + (1 / 128 if fos else 0)
                tot_b += bpe * wl.elements
                tot_ms += ms
                us[fos] = 1e3 * ms
                del wl
                torch.cuda.empty_cache()
            out.append({"rows": rows, "cols": 4096, "dequant": dq, "us_4over6_off": round(us[0], 2),
                        "us_4over6_on": round(us[1], 2),
                        "overhead_pct": round(100 * (us[1] / us[0] - 1), 1)})
    return {"metric": METRIC, "value": round(tot_b / (tot_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
            "n_gpus": 1, "steps": steps, "warmup": args.warmup, "higher_is_better": True,
            "dtype": "f32", "data": "synthetic",
            "config": {"workload": "Four-Over-Six overhead of the 1x16 row quantiser (E4M3, "
                                   "RNE) on activations S x 4096, S = 2048 and 8192, with and "
                                   "without dequant output"},
            "fos_overhead": out, "pages": FOS_PAGES}


# --------------------------------------------------------------- clocks --

class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index, period_ms: int = 50):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", f"-lms={period_ms}"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    @staticmethod
    def _when(stamp: str):
        import datetime
        for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
            try:
                return datetime.datetime.strptime(stamp, fmt).timestamp()
            except ValueError:
                pass
        return None

    def stop(self, t0: float | None = None, t1: float | None = None):
        """Median SM clock, maximum clock and throttle reasons of the samples
        taken between host times t0 and t1 (the timed passes); all samples
        when their timestamps cannot be read."""
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            try:
                rows.append((self._when(f[0]), float(f[2]), float(f[3]), f[6:10]))
            except ValueError:
                continue
        inside = [r for r in rows if r[0] is not None and t0 is not None and t0 <= r[0] <= t1]
        window = "timed passes" if inside else "whole run"
        use = inside or rows
        if not use:
            return None
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = {name for r in use for name, v in zip(names, r[3])
                   if v.lower().startswith("active")}
        return {"sm_mhz": statistics.median(r[1] for r in use),
                "sm_max_mhz": max(r[2] for r in use), "reasons": sorted(reasons),
                "samples": len(use), "window": window}


# --------------------------------------------------------------- timing --

def _smi_id(local: int) -> str:
    """nvidia-smi id of the CUDA device (its PCI bus id when torch exposes it)."""
    try:
        p = torch.cuda.get_device_properties(local)
        dom, bus, devn = p.pci_domain_id, p.pci_bus_id, p.pci_device_id
        return f"{dom:08X}:{bus:02X}:{devn:02X}.0"
    except Exception:
        return str(local)


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_steps(wl, k0, K, events=None):
    """Launch K steps. With `events`, one pre-created event is recorded before
    the first kernel and one after every kernel, so the kernels' durations tile
    the timed region; returns [(kernel, start_event, end_event)]."""
    out = []
    j = 0
    if events is not None:
        events[0].record()
    for k in range(k0, k0 + K):
        i = k % wl.nsets
        for kern in wl.kernels(k, i):
            rc = kern.fn()
            if rc != 0:
                raise nv.Nvfp4Error(kern.name, rc)
            if events is not None:
                events[j + 1].record()
                out.append((kern, events[j], events[j + 1]))
                j += 1
    return out


def time_ours(wl, args, world, local):
    """Timed passes over the same K steps, each bracketed by a barrier, a
    device synchronisation and one CUDA event at either end, repeated back to
    back until at least --min-seconds of device time have run, so that the
    clock samples cover the kernels under load; the median pass is the step
    time. A last pass with an event after every call (an event record between
    kernels costs the device about a microsecond and a half) gives the
    per-kernel durations behind the roofline."""
    import math
    run_steps(wl, 0, args.warmup)
    torch.cuda.synchronize()
    nk = sum(len(wl.kernels(k, k % wl.nsets)) for k in range(args.warmup, args.warmup + args.steps))
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    events = [torch.cuda.Event(enable_timing=True) for _ in range(nk + 1)]
    barrier(world)
    torch.cuda.synchronize()
    clocks = ClockSampler(_smi_id(local))
    time.sleep(0.3)  # the sampler's first line
    t0 = time.time()
    wall0 = time.perf_counter()
    passes, npass = [], None
    while npass is None or len(passes) < npass:
        barrier(world)
        torch.cuda.synchronize()
        a.record()
        run_steps(wl, args.warmup, args.steps)
        b.record()
        torch.cuda.synchronize()
        passes.append(a.elapsed_time(b))
        if npass is None:
            want = math.ceil(args.min_seconds * 1e3 / max(passes[0], 1e-3))
            npass = int(max_over_ranks(float(min(max(3, want), args.max_passes)), world))
    wall = time.perf_counter() - wall0
    barrier(world)
    torch.cuda.synchronize()
    evs = run_steps(wl, args.warmup, args.steps, events)
    torch.cuda.synchronize()
    t1 = time.time()
    barrier(world)
    torch.cuda.synchronize()
    clk = clocks.stop(t0, t1)
    per_kernel = {}
    for kern, e0, e1 in evs:
        d = per_kernel.setdefault(kern.name, {"ms": 0.0, "n": 0, "bytes": kern.nbytes,
                                              "launches": kern.launches})
        d["ms"] += e0.elapsed_time(e1)
        d["n"] += 1
    stats = {"passes": len(passes), "device_s": round(sum(passes) / 1e3, 3),
             "median_ms": round(statistics.median(passes), 4), "min_ms": round(min(passes), 4),
             "max_ms": round(max(passes), 4)}
    return statistics.median(passes), stats, per_kernel, clk, wall


def time_e2e(wl, steps, device, sets=None, passes=3):
    """The same metric through the C ABI with host buffers, as a user streaming
    tensors through it would run it: every step copies its inputs from pinned
    host memory to the device (copy-in stream), runs the kernels (the
    workload's stream) and copies every output back to pinned host memory
    (copy-out stream). Step k uses device buffer set k % B (B = `sets`, else
    the workload's e2e_sets, else 2, or 1 when the workload holds a single
    set); events order each buffer's reuse, so
    one step's copies overlap its neighbours' compute and copies. Events
    bracket each pass of `steps` steps on all three streams; the median of
    `passes` passes is the figure (the host and its memory are shared, so one
    pass can catch a transient slowdown). Afterwards the inputs' and
    outputs' copies are timed on the same buffers, each direction by itself
    and both at once, for the host link's rates in the same run. Returns
    (ms, bytes in, bytes out, link)."""
    B = sets or getattr(wl, "e2e_sets", 1 if wl.nsets == 1 else 2)
    ins0, outs0 = wl.e2e_io(0, 0)
    h_in = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in ins0]
    for h, t in zip(h_in, ins0):
        h.copy_(t.cpu())
    h_out = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs0]
             for _ in range(B)]
    bi = sum(t.numel() * t.element_size() for t in ins0)
    bo = sum(t.numel() * t.element_size() for t in outs0)
    comp = torch.cuda.current_stream(device)
    cin, cout = torch.cuda.Stream(device), torch.cuda.Stream(device)
    in_free = [None] * B   # compute of the last step that read set b is done
    out_free = [None] * B  # copy-out of the last step that wrote set b is done

    def step(k):
        b = k % B
        ins, outs = wl.e2e_io(k, b)
        with torch.cuda.stream(cin):
            if in_free[b] is not None:
                cin.wait_event(in_free[b])
            for h, t in zip(h_in, ins):
                t.copy_(h, non_blocking=True)
            e_in = torch.cuda.Event()
            e_in.record(cin)
        comp.wait_event(e_in)
        if out_free[b] is not None:
            comp.wait_event(out_free[b])
        for kern in wl.kernels(k, b):
            rc = kern.fn()
            if rc != 0:
                raise nv.Nvfp4Error(kern.name, rc)
        e_c = torch.cuda.Event()
        e_c.record(comp)
        in_free[b] = e_c
        with torch.cuda.stream(cout):
            cout.wait_event(e_c)
            for h, t in zip(h_out[b], outs):
                h.copy_(t, non_blocking=True)
            e_o = torch.cuda.Event()
            e_o.record(cout)
        out_free[b] = e_o
        return e_o

    for k in range(2):
        step(k)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    pass_ms = []
    for _ in range(max(1, passes)):
        in_free[:] = [None] * B
        out_free[:] = [None] * B
        a.record(comp)
        cin.wait_event(a)
        cout.wait_event(a)
        last = None
        for k in range(steps):
            last = step(k)
        comp.wait_event(last)
        b.record(comp)
        torch.cuda.synchronize()
        pass_ms.append(a.elapsed_time(b))
    ms = statistics.median(pass_ms)
    # the host link's rates at this moment, each direction alone, on the same
    # buffers (best of 3): the bound the e2e figure is read against
    ins, outs = wl.e2e_io(0, 0)

    def copy_ms(pairs):
        best = float("inf")
        for _ in range(3):
            torch.cuda.synchronize()
            a.record(comp)
            for dst, src in pairs:
                dst.copy_(src, non_blocking=True)
            b.record(comp)
            torch.cuda.synchronize()
            best = min(best, a.elapsed_time(b))
        return best
    def both_ms():
        # the inputs in and the outputs out at once, each on its copy stream
        best = float("inf")
        for _ in range(3):
            torch.cuda.synchronize()
            a.record(comp)
            for s_, pairs in ((cin, list(zip(ins, h_in))), (cout, list(zip(h_out[0], outs)))):
                s_.wait_event(a)
                with torch.cuda.stream(s_):
                    for dst, src in pairs:
                        dst.copy_(src, non_blocking=True)
                comp.wait_stream(s_)
            b.record(comp)
            torch.cuda.synchronize()
            best = min(best, a.elapsed_time(b))
        return best
    link = {"copy_in_gbs": round(bi / (copy_ms(list(zip(ins, h_in))) * 1e-3) / 1e9, 1),
            "copy_out_gbs": round(bo / (copy_ms(list(zip(h_out[0], outs))) * 1e-3) / 1e9, 1),
            "copy_both_gbs": round((bi + bo) / (both_ms() * 1e-3) / 1e9, 1),
            "device_sets": B, "passes_ms": [round(t, 3) for t in pass_ms]}
    return ms, bi, bo, link


def link_bound_gbs(step_bytes: float, bytes_in: float, bytes_out: float, link: dict) -> float:
    """The end-to-end figure's ceiling in GB/s of algorithmic bytes: no step
    can take less than its larger copy at that direction's rate, nor less
    than both copies at the rate the two directions reach together."""
    step_s = max(bytes_in / (link["copy_in_gbs"] * 1e9), bytes_out / (link["copy_out_gbs"] * 1e9),
                 (bytes_in + bytes_out) / (link["copy_both_gbs"] * 1e9))
    return step_bytes / step_s / 1e9


def cpu_model() -> str:
    """The host CPU's model name (Linux /proc/cpuinfo; the Arm machines give a
    part number instead)."""
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read()
    except OSError:
        return "unknown"
    for key in ("model name", "Model Name", "Hardware", "CPU part"):
        for line in info.splitlines():
            if line.split(":")[0].strip() == key:
                val = line.split(":", 1)[1].strip()
                return val if key != "CPU part" else f"Arm CPU part {val}"
    return "unknown"


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(wl, budget_s):
    """The oracle on the host: one core (the single-threaded build) and all
    cores (the OpenMP build of the same source), each on a bounded sample of
    the workload; `value` is the all-core leg."""
    import oracle
    legs = []
    for n in (1, host_cores()):
        used = oracle.set_threads(n)
        try:
            e, dt, sample = wl.cpu_sample(budget_s)
        finally:
            oracle.set_threads(1)
        legs.append({"cores": used, "value": round(e * wl.bytes_per_elem / dt / 1e9, 5),
                     "gelem_per_s": round(e / dt / 1e9, 6), "sample": sample})
    best = legs[-1]
    return {"value": best["value"], "unit": "GB/s", "cores": best["cores"], "kind": "oracle",
            "sample": best["sample"], "gelem_per_s": best["gelem_per_s"],
            "cpu_model": cpu_model(), "nproc": host_cores(), "legs": legs}


def reference_arm(args, world, rank):
    """The oracle, as it stands, timed on all host cores (its OpenMP build):
    each step is a bounded sample of the chosen workload, charged with the
    same per-call algorithmic bytes as our arm, reported in our arm's metric
    and unit."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    bpe = WORKLOADS[args.config].call_bpe(_ctor_args(args.config, args))
    desc, sample_text, step = _reference_sample(args)
    cores = oracle.set_threads(host_cores())
    secs, total_e, total_b = 0.0, 0, 0.0
    for k in range(args.warmup + args.steps):
        e, calls, dt = step(k)
        if k >= args.warmup:
            secs += dt
            total_e += e
            total_b += e * sum(bpe[c] for c in calls)
    oracle.set_threads(1)
    value = total_b / secs / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 5), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * secs / max(1, args.steps), 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": describe_workload(args.config, args), "sample": sample_text,
                   "oracle_workload": desc},
        "gelem_per_s": round(total_e / secs / 1e9, 6),
        "cpu_baseline": {"value": round(value, 5), "unit": "GB/s", "cores": cores,
                         "kind": "oracle", "sample": sample_text, "cpu_model": cpu_model(),
                         "nproc": host_cores()},
        "e2e": {"value": round(value, 5), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _timed(fn):
    t0 = time.perf_counter()
    fn()
    return time.perf_counter() - t0


def _reference_sample(args):
    """(workload text, sample text, step) for the reference arm. step(k) runs
    the oracle on the same rows of the workload for step k and returns
    (elements, names of the calls it ran, seconds); the calls' bytes per
    element come from the workload's call_bpe, as in our arm."""
    import oracle
    n = args.ref_rows
    if args.config in (1, 2):
        rows, cols = (1024, 1024) if args.config == 1 else (8192, 4096)
        fos = 0 if args.config == 1 else 1
        xb = (synth.outlier_normal(rows, cols, seed=0) if args.config == 1
              else synth.student_t(rows, cols, seed=1))
        sub = xb[:n]

        def run():
            a, _ = oracle.global_amax(sub)
            oracle.quantize(sub, a, four_over_six=fos)

        def step(k):
            return sub.size, ("amax", "quantize_row"), _timed(run)
        wl = "activation 8192x4096 bf16 0.5*Student-t(3), amax + row 4/6" if args.config == 2 \
            else "1024x1024 bf16 N(0,1) 0.1% x20, amax + row"
        return wl, f"first {sub.shape[0]} rows of {rows} per step", step
    if args.config in (3, 9):
        wb, gb, s = synth.scale_learning(seed=2)
        names = ("fakequant_fwd", "scale_grad_bwd") if args.config == 3 else \
            ("fakequant_fwd_fp8", "scale_grad_bwd_fp8")
        gam = float(np.abs(synth.bf16_bits_to_f32(wb)).max()) * 1.5

        def run():
            if args.config == 3:
                oracle.fakequant_fwd(wb[:n], s[:n], s[:n])
                oracle.scale_grad_bwd(wb[:n], gb[:n], s[:n], s[:n])
            else:
                oracle.fakequant_fwd_fp8(wb[:n], s[:n], s[:n], gam)
                oracle.scale_grad_bwd_fp8(wb[:n], gb[:n], s[:n], s[:n], gam)

        def step(k):
            return n * wb.shape[1], names, _timed(run)
        return ("scale-learning step 14336x4096" + (", FP8 scales" if args.config == 9 else "")), \
            f"first {n} of 14336 rows per step", step
    if args.config == 4:
        gen = synth.DriftingGradient()
        period = _ctor_args(4, args)["period"]
        subs = [gen.step(t)[:n] for t in range(2)]
        amax = [None]

        def step(k):
            sub = subs[k % 2]
            t = time.perf_counter()
            calls = ("quantize_row_sr",)
            if amax[0] is None or k % period == 0:  # periodic tensor scaling
                amax[0], _ = oracle.global_amax(sub)
                calls = ("amax", "quantize_row_sr")
            oracle.quantize(sub, amax[0], scale_fmt=1, rounding=1, seed=3, step=k,
                            dequant=False)
            return sub.size, calls, time.perf_counter() - t
        return "gradient 16384x4096 UE5M3 SR periodic", \
            f"first {n} of 16384 rows per step (amax every {period} steps)", step
    if args.config == 6:
        xb = synth.student_t(8192, 4096, seed=1)
        sub = xb[:n].reshape(-1, 1, 4096)

        def run():
            a, _ = oracle.global_amax(sub, sub.shape[0])
            oracle.quantize(sub, a, four_over_six=1)

        def step(k):
            return sub.size, ("quantize_per_token",), _timed(run)
        return "activation 8192x4096 per-token outer scales, row 4/6", \
            f"first {sub.shape[0]} of 8192 rows per step", step
    if args.config in (7, 8):
        target = args.config - 7
        xb = synth.student_t(8192, 4096, seed=1)
        a, _ = oracle.global_amax(xb)
        m = max(32, (n // 4) - (n // 4) % 32)
        q = oracle.quantize(xb[:m], a, four_over_six=1, dequant=False)
        name = "requant_mxfp8_sr" if target == 0 else "requant_nvfp4_sr"

        def run():
            oracle.requant(q["row_codes"], q["row_scales"], a, target=target, rounding=1,
                           seed=7, src_fos=1, dst_fos=target)

        def step(k):
            return m * 4096, (name,), _timed(run)
        return ("activation 8192x4096 NVFP4 (4/6) re-quantised, transposed, SR to "
                + ("MXFP8" if target == 0 else "NVFP4")), \
            f"first {m} of 8192 source rows per step", step
    if args.config == 11:
        wb, _, _ = synth.scale_learning(seed=2)
        m = max(16, n - n % 16)

        def run():
            a, _ = oracle.global_amax(wb[:m])
            oracle.quantize_tile16(wb[:m], a)

        def step(k):
            return m * wb.shape[1], ("amax", "quantize_tile16"), _timed(run)
        return "weight 14336x4096 16x16 tile scale + transpose", \
            f"first {m} of 14336 rows per step", step
    if args.config == 12:
        xb = synth.DriftingGradient(seed=3).step(0)
        m = max(32, n - n % 32)

        def step(k):
            return m * xb.shape[1], ("mx_quantize_sr",), _timed(
                lambda: oracle.mx_quantize(xb[:m], blocks=3, rounding=1, seed=12, step=k))
        return "gradient 16384x4096 MXFP8 rows + transpose, SR", \
            f"first {m} of 16384 rows per step", step
    if args.config == 10:
        wb, _, s = synth.scale_learning(seed=2)
        gam = float(np.abs(synth.bf16_bits_to_f32(wb)).max()) * 1.5
        m = max(1, n // 64)

        def run():
            oracle.scale_init_mse(wb[:m], gam)
            oracle.export_scales(wb[:m], s[:m], s[:m], gam)

        def step(k):
            return m * wb.shape[1], ("scale_init_mse", "export_scales"), _timed(run)
        return "MSE scale sweep + export 14336x4096", f"first {m} of 14336 rows per step", step
    xb = synth.moe_experts(1, 2048, 7168, seed=4)[0]
    sub = xb[:max(16, n - n % 16)]

    def run():
        a, _ = oracle.global_amax(sub)
        oracle.quantize(sub, a, blocks=3, four_over_six=1)

    def step(k):
        return sub.size, ("amax", "quantize_dual"), _timed(run)
    return "MoE 64x2048x7168 dual 4/6", \
        f"first {sub.shape[0]} rows of one expert per step", step


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=5, choices=sorted(WORKLOADS) + [FOS_OVERHEAD])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--e2e-passes", type=int, default=3,
                    help="timed end-to-end passes; the median is reported")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-rows", type=int, default=512)
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-sets", type=int, default=None,
                    help="device buffer sets the end-to-end run rotates through (default: one "
                         "and the workload's own count, both timed, the faster kept)")
    ap.add_argument("--experts", type=int, default=64, help="MoE workload: number of experts")
    ap.add_argument("--min-seconds", type=float, default=2.0,
                    help="device time the repeated timed passes run for at least")
    ap.add_argument("--max-passes", type=int, default=5000)
    ap.add_argument("--sr-steps", type=int, default=32,
                    help="drifting-gradient workload: distinct step inputs held on the device")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world, rank, local = dist_setup(args) if args.impl == "ours" else (
        int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")), 0)
    if args.impl == "reference":
        if args.config == FOS_OVERHEAD:
            ap.error("--config 13 (the 4/6 overhead) has no reference arm")
        args.steps = args.steps or 3
        reference_arm(args, world, rank)
        return

    device = torch.device("cuda", local)
    nv.build()
    if args.config == FOS_OVERHEAD:
        if rank == 0:
            print(json.dumps(fos_overhead(args, device)), flush=True)
        return
    extra = {5: dict(experts=args.experts), 4: dict(nsteps=args.sr_steps)}.get(args.config, {})
    wl = WORKLOADS[args.config](device, **extra)
    args.steps = args.steps or 20
    pass_ms, pass_stats, per_kernel, clk, wall = time_ours(wl, args, world, local)
    total_ms = max_over_ranks(pass_ms, world)
    units = wl.elements * args.steps * world
    alg_bytes = sum(d["bytes"] * d["n"] for d in per_kernel.values()) * world
    value = alg_bytes / (total_ms * 1e-3) / 1e9
    st = int(wl.status.item())
    if st != 0:
        raise RuntimeError(f"device status {st} during the benchmark")

    peak, peak_kind = measured_peak()
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    mhz = float(clk["sm_max_mhz"]) if clk and clk.get("sm_max_mhz") else sm_max_mhz()
    dom = per_kernel[wl.dominant]
    if len(per_kernel) == 1 and dom["n"] == args.steps:
        # one call per step: the clean passes' events bracket exactly the K calls
        dom_ms, dur_src = total_ms / args.steps, "median pass, one call per step"
    else:
        dom_ms, dur_src = dom["ms"] / dom["n"], "an event after every call"
    achieved = dom["bytes"] / (dom_ms * 1e-3) / 1e9
    traffic = _committed_counts(args.config, wl.dominant, "traffic.json", "bytes")
    alu_ops = getattr(wl, "alu_ops_per_elem", {}).get(wl.dominant)
    elems_per_call = dom["bytes"] / wl.call_bpe(_wl_kw(wl))[wl.dominant]
    kernels = {name: {"calls": d["n"], "kernels_per_call": d["launches"],
                      "avg_us": round(1e3 * d["ms"] / d["n"], 3),
                      "alg_bytes": int(d["bytes"]),
                      "gbs": round(d["bytes"] / (d["ms"] / d["n"] * 1e-3) / 1e9, 1),
                      "frac_of_peak": round(d["bytes"] / (d["ms"] / d["n"] * 1e-3) / 1e9 / peak, 4)}
               for name, d in per_kernel.items()}
    if alu_ops is None:
        roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                    "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                    "kernel": wl.dominant, "peak_source": f"{peak_kind} HBM copy bandwidth",
                    "duration_from": dur_src}
    else:
        alu_peak = alu_peak_tops(sms, mhz)
        alu = alu_ops * elems_per_call / (dom_ms * 1e-3) / 1e12
        roofline = {"bound": "alu", "achieved": round(alu, 2), "peak": round(alu_peak, 2),
                    "unit": "Top/s", "frac": round(alu / alu_peak, 4), "traffic": traffic,
                    "kernel": wl.dominant,
                    "peak_source": f"{sms} SMs x 128 fp32 lanes x {mhz:.0f} MHz (derived)",
                    "ops_per_element": alu_ops, "duration_from": dur_src}
    ipe = _committed_counts(args.config, wl.dominant, "inst.json", "warp_inst_per_elem")
    if ipe is not None:
        # the same kernel against its instruction-issue bound
        rate = ipe * elems_per_call / (dom_ms * 1e-3) / 1e9
        ipeak = issue_peak_ginst(sms, mhz)
        roofline["issue"] = {"warp_inst_per_elem": round(ipe, 4),
                             "thread_inst_per_elem": round(32 * ipe, 2),
                             "achieved": round(rate, 1), "peak": round(ipeak, 1),
                             "unit": "Gwarp-inst/s", "frac": round(rate / ipeak, 4),
                             "peak_source": f"{sms} SMs x 4 schedulers x {mhz:.0f} MHz",
                             "count_from": "ncu smsp__inst_executed.sum of one launch "
                                           "(profiles/inst.json)"}
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": wl.workload, "elements_per_step": wl.elements,
                   "alg_bytes_per_elem": round(wl.bytes_per_elem, 5),
                   "l2": (f"inputs larger than L2: {wl.nsets} rotating input/output sets, "
                          f"{wl.working_set / 2 ** 20:.0f} MiB > {L2_BYTES / 2 ** 20:.0f} MiB L2")},
        "gelem_per_s": round(units / (total_ms * 1e-3) / 1e9, 3),
        "roofline": roofline,
        "kernels": kernels,
        "timing": dict(pass_stats, steps_per_pass=args.steps,
                       rule="median of the timed passes (barrier + synchronize + events around "
                            "each pass of K steps)"),
        "gpu_launches": sum(d["n"] * d["launches"] for d in per_kernel.values()),
        "clocks": clk,
        "host_wall_s": round(wall, 3),
    }
    if rank == 0 and not args.no_e2e:
        per_step_bytes = alg_bytes / world / args.steps
        # the pipeline depth that suits the host: every device-set count the
        # workload offers is timed (or the one asked for) and the fastest kept
        default_sets = getattr(wl, "e2e_sets", 1 if wl.nsets == 1 else 2)
        depths = [args.e2e_sets] if args.e2e_sets else sorted({1, default_sets})
        best, by_sets = None, {}
        for nsets_e2e in depths:
            ms, bi, bo, link = time_e2e(wl, args.e2e_steps, device, nsets_e2e, args.e2e_passes)
            e2e = per_step_bytes * args.e2e_steps / (ms * 1e-3) / 1e9
            by_sets[str(nsets_e2e)] = round(e2e, 2)
            if best is None or e2e > best[0]:
                best = (e2e, bi, bo, link)
        e2e, bi, bo, link = best
        link["bound_gbs"] = round(link_bound_gbs(per_step_bytes, bi, bo, link), 1)
        link["frac_of_bound"] = round(e2e / link["bound_gbs"], 3)
        link["by_device_sets"] = by_sets
        line["e2e"] = {"value": round(e2e, 2), "unit": "GB/s", "h2d_bytes_per_step": int(bi),
                       "d2h_bytes_per_step": int(bo), "host_link": link}
    if rank == 0 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(wl, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# the CUDA sources each timed kernel is built from
_COMMON = ["device.cuh", "encode.cuh", "launch.h"]
KERNEL_SOURCES = {
    "amax": ["amax.cu", "device.cuh", "launch.h"],
    "quantize_row": ["quant_row.cu"] + _COMMON,
    "quantize_row_sr": ["quant_row.cu"] + _COMMON,
    "quantize_dual": ["quant_dual.cu"] + _COMMON,
    "quantize_per_token": ["quant_token.cu"] + _COMMON,
    "fakequant_fwd": ["ste.cu"] + _COMMON,
    "scale_grad_bwd": ["ste.cu"] + _COMMON,
    "requant_mxfp8_sr": ["requant.cu"] + _COMMON,
    "requant_nvfp4_sr": ["requant.cu"] + _COMMON,
    "fakequant_fwd_fp8": ["ste.cu"] + _COMMON,
    "scale_grad_bwd_fp8": ["ste.cu"] + _COMMON,
    "scale_init_mse": ["scale_init.cu"] + _COMMON,
    "export_scales": ["ste.cu"] + _COMMON,
    "quantize_tile16": ["quant_tile16.cu"] + _COMMON,
    "mx_quantize_sr": ["mx_quant.cu", "mx_quant.h"] + _COMMON,
}


def kernel_source_hash(kernel: str | None = None) -> str:
    """sha256 over the CUDA sources of `kernel` (all of csrc/ when None), so
    committed ncu counters can be matched to the code they were taken from."""
    import glob
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "nvfp4_block_scaled_02_gb300", "csrc")
    if kernel is None:
        files = sorted(os.path.basename(f) for f in glob.glob(os.path.join(csrc, "*"))
                       if f.endswith((".cu", ".cuh", ".h")))
    else:
        files = sorted(KERNEL_SOURCES.get(kernel, []))
    for name in files:
        with open(os.path.join(csrc, name), "rb") as fh:
            h.update(name.encode() + b"\0" + fh.read())
    return h.hexdigest()[:16]


def _committed_counts(config: int, kernel: str, fname: str, key: str):
    """A per-launch ncu figure of `kernel` on workload `config` from a
    committed summary under profiles/ (traffic.json: DRAM bytes read + written;
    inst.json: warp instructions per element), or None when absent or taken
    from other sources of that kernel than the ones built now."""
    p = os.path.join(ROOT, "profiles", fname)
    try:
        with open(p) as f:
            d = json.load(f)
        e = d.get("workloads", {}).get(str(config), {}).get(kernel)
        if not e or e.get("source_sha") != kernel_source_hash(kernel):
            return None
        return float(e[key])
    except Exception:
        return None


def _wl_kw(wl) -> dict:
    """The constructor options a workload's call_bpe reads."""
    return {"fos": getattr(wl, "fos", 1), "cols": getattr(wl, "cols", None),
            "target": getattr(wl, "target", 0)}


if __name__ == "__main__":
    main()
