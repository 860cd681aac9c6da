#!/usr/bin/env python
"""Benchmark of the fine-grained FP8 hot path on B300.

One step = one pass of the whole path over one batch of synthetic inputs, the
FP8 training step of a large MoE transformer layer:

  forward of an FP8 linear layer      X bf16 [8192, 7168] -> 1x128 quantize;
                                      W bf16 [7168, 18432] -> 128x128 quantize;
                                      Y = GEMM (1x128 x 128x128 scales) bf16 [8192, 18432]
  data gradient of that layer         dY bf16 [8192, 18432] -> 1x128 quantize;
                                      W -> 128x128 quantize (row-major codes);
                                      dX = GEMM (1x128 x 128x128 scales) bf16 [8192, 7168]
  weight gradient of that layer       Xw bf16 [8192, 7168] ~ N(0, 1e-3^2) with 0.1% elements
                                      x1000 -> 1x128 quantize (dY quantized above);
                                      cached Xwq and dYq -> 1x128 -> 128x1 requantize;
                                      dW = GEMM (128x1 x 128x1 scales) bf16 [7168, 18432]
  SwiGLU recompute of that MLP        cached gate/up bf16 [8192, 2 x 18432] -> silu(g) u, rounded
                                      to bf16 and 1x128-quantized in one pass -> codes [8192, 18432]
  MoE expert forward                  16384 tokens x 8 picks (Zipf 1.1 over 32 experts,
                                      padded to 128 rows) bf16 [~133k, 7168] -> 1x128 quantize;
                                      32 experts W_g [7168, 2048] -> 128x128 quantize;
                                      grouped GEMM -> bf16 [~133k, 2048]

`pow2_mx` repeats the step with power-of-two scales: the *_pow2 quantizers and
the GEMMs whose scales the tensor core applies (no FP32 promotion), timed the
same way, with the error of both paths against the exact product of the
original bf16 inputs on sampled outputs.

`value` is the step's GEMM work (2MNK summed over the four GEMMs, routed rows
for the MoE) divided by the step time, summed over ranks: whole-step TFLOP/s,
quantizers included.  Inputs live in HBM before the timed region; every input
is larger than L2 or is followed by larger traffic.  `e2e` repeats the step
with the inputs copied from pinned host memory and the outputs read back, the
copies of neighbouring steps overlapping the kernels (two buffer sets).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Multi-GPU (torchrun): every rank runs the same step on its own GPU (weak
scaling, no collective on the data path); the time is the max over ranks.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "block-scaled FP8 GEMM TFLOP/s (% FP8 peak); quantizer GB/s (% HBM)"
UNIT = "TFLOP/s"
FP8_OVER_BF16 = 2.0          # nominal dense FP8 / BF16 tensor throughput ratio (4.5 / 2.25 PFLOP/s)
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
L2_BYTES = 126 * 2 ** 20

# workload sizes
T, CIN, COUT = 8192, 7168, 18432
G, MOE_K, MOE_N, TOKENS, TOPK, ZIPF = 32, 7168, 2048, 16384, 8, 1.1


def parse_args():
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=300)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--e2e-steps", type=int, default=6)
    p.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    p.add_argument("--no-cpu-baseline", action="store_true", help="skip timing the CPU oracle")
    p.add_argument("--cpu-seconds", type=float, default=15.0, help="target CPU time of the oracle sample")
    p.add_argument("--no-pow2", action="store_true", help="skip the power-of-two / hardware-scaled leg")
    p.add_argument("--steady-seconds", type=float, default=2.0,
                   help="length of the steady-state leg (clock record under sustained load; 0 skips it)")
    return p.parse_args()


# ------------------------------------------------------------ workload ----

class Workload:
    """Host (numpy) inputs of one step plus the algorithmic work of each kernel."""

    def __init__(self, seed_offset=0):
        s = seed_offset
        self.x, _ = synth.activation(2 + s, T, CIN)                     # 1% channels x100
        self.w = synth.weight(2 + s, CIN, COUT)                         # N(0, 0.02^2)
        self.dy = synth.wgrad_tensor(4 + s, 1, T, COUT)                 # N(0,1e-3^2), 0.1% x1000
        self.xw = synth.wgrad_tensor(4 + s, 0, T, CIN)                  # the weight gradient's X, same recipe
        self.gate_up = synth.swiglu_inputs(6 + s, T, COUT)              # cached gate | up, N(0, 1.7^2)
        moe = synth.moe_inputs(seed=5 + s, G=G, K=MOE_K, N=MOE_N, tokens=TOKENS, topk=TOPK, zipf_s=ZIPF)
        self.moe_x = moe.x
        self.moe_w = moe.w
        self.moe_offsets = moe.offsets
        self.moe_counts = moe.counts
        self.moe_rows = int(moe.offsets[-1])
        self.routed_rows = moe.routed_rows

    def gemm_flops(self):
        return {
            "gemm_fprop": 2.0 * T * COUT * CIN,
            "gemm_dgrad": 2.0 * T * CIN * COUT,
            "gemm_wgrad": 2.0 * CIN * COUT * T,
            "grouped_gemm_moe": 2.0 * self.routed_rows * MOE_N * MOE_K,
        }

    def quant_bytes(self):
        def q(rows, cols):       # bf16 in, e4m3 out, one fp32 scale per 128 elements
            return rows * cols * 3 + rows * cols // 128 * 4

        def rq(rows, cols):      # e4m3 + scales in, e4m3 + scales out
            return 2 * (rows * cols + rows * cols // 128 * 4)
        return {
            "quant_act_x": q(T, CIN),
            "quant_w": q(CIN, COUT) - CIN * COUT // 128 * 4 + (CIN // 128) * (COUT // 128) * 4,
            "quant_w_rowmajor": q(CIN, COUT) - CIN * COUT // 128 * 4 + (CIN // 128) * (COUT // 128) * 4,
            "quant_act_dy": q(T, COUT),
            "quant_act_xw": q(T, CIN),
            "swiglu_quant": T * 2 * COUT * 2 + T * COUT + T * COUT // 128 * 4,
            "requant_x": rq(T, CIN),
            "requant_dy": rq(T, COUT),
            "quant_act_moe": q(self.moe_rows, MOE_K),
            "quant_w_moe": G * (MOE_K * MOE_N * 3 + (MOE_K // 128) * (MOE_N // 128) * 4),
        }

    def describe(self):
        return {
            "workload": "FP8 training step of one MoE transformer layer: linear fwd "
                        "[8192x7168]x[7168x18432] + dgrad (dX [8192x7168], K=18432) + "
                        "wgrad (dW [7168x18432], K=8192 tokens) + "
                        "MoE grouped fwd (32 experts [7168x2048], 16384 tokens x 8, Zipf 1.1)",
            "fprop": {"M": T, "N": COUT, "K": CIN},
            "dgrad": {"M": T, "N": CIN, "K": COUT},
            "wgrad": {"M": CIN, "N": COUT, "K": T},
            "moe": {"experts": G, "N": MOE_N, "K": MOE_K, "routed_rows": self.routed_rows,
                    "padded_rows": self.moe_rows},
            "quantizers": "1x128 act [8192x7168], [8192x18432], [%dx7168]; 128x128 weight "
                          "[7168x18432] (K-major and row-major codes), 32x[7168x2048]; "
                          "1x128->128x1 requant of [8192x7168], "
                          "[8192x18432]" % self.moe_rows,
            "wgrad_inputs": "X [8192x7168] and dY [8192x18432] ~ N(0, 1e-3^2) with Bernoulli(0.001) "
                            "elements x1000, each 1x128-quantized then requantized 128x1 along tokens",
            "swiglu": "cached gate/up [8192, 2x18432] ~ N(0, 1.7^2) -> 1x128 codes [8192, 18432]",
            "l2": "inputs larger than L2 (126 MB); %.1f GB of quantizer traffic per step"
                  % (sum(self.quant_bytes().values()) / 1e9),
            "global_batch": T,
            "parallelism": "replicas",
        }


# -------------------------------------------------------------- device ----

class DeviceStep:
    """Device buffers and the sequence of library calls of one step."""

    KERNELS = ["quant_act_x", "quant_w", "gemm_fprop", "quant_act_dy", "quant_w_rowmajor", "gemm_dgrad",
               "swiglu_quant", "quant_act_xw", "requant_x", "requant_dy", "gemm_wgrad", "quant_act_moe",
               "quant_w_moe", "grouped_gemm_moe"]
    LAUNCHES_PER_STEP = 14      # the 32 expert weights are quantized in one batched launch

    def __init__(self, wl, device):
        import torch
        import fp8_fine_grained_20_b300 as fg
        self.fg = fg
        self.torch = torch
        self.dev = device
        u8, f32, bf = torch.uint8, torch.float32, torch.bfloat16

        def e(shape, dt):
            return torch.empty(shape, dtype=dt, device=device)

        # inputs
        self.x = e((T, CIN), bf)
        self.w = e((CIN, COUT), bf)
        self.dy = e((T, COUT), bf)
        self.xw = e((T, CIN), bf)
        self.gate_up = e((T, 2 * COUT), bf)
        self.moe_x = e((wl.moe_rows, MOE_K), bf)
        self.moe_w = e((G, MOE_K, MOE_N), bf)
        self.moe_off = e((G + 1,), torch.int32)
        # intermediates (scales MN-major: logical [rows, groups] views with stride 1 along rows)
        self.xq, self.sx = e((T, CIN), u8), e((CIN // 128, T), f32).t()
        self.wq, self.sw = e((COUT, CIN), u8), e((CIN // 128, COUT // 128), f32)
        self.wq_rm, self.sw_rm = e((CIN, COUT), u8), e((CIN // 128, COUT // 128), f32)
        self.dyq, self.sdy = e((T, COUT), u8), e((COUT // 128, T), f32).t()
        self.xwq, self.sxw = e((T, CIN), u8), e((CIN // 128, T), f32).t()
        self.hq, self.sh = e((T, COUT), u8), e((COUT // 128, T), f32).t()
        self.xqT, self.sxT = e((CIN, T), u8), e((T // 128, CIN), f32).t()
        self.dyqT, self.sdyT = e((COUT, T), u8), e((T // 128, COUT), f32).t()
        self.mxq, self.smx = e((wl.moe_rows, MOE_K), u8), e((MOE_K // 128, wl.moe_rows), f32).t()
        self.mwq, self.smw = e((G, MOE_N, MOE_K), u8), e((G, MOE_K // 128, MOE_N // 128), f32)
        # outputs
        self.y = e((T, COUT), bf)
        self.dx = e((T, CIN), bf)
        self.dw = e((CIN, COUT), bf)
        self.moe_y = e((wl.moe_rows, MOE_N), bf)
        self.load_inputs(wl)

    def load_inputs(self, wl):
        torch = self.torch

        def bf16(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
        self.x.copy_(bf16(wl.x))
        self.w.copy_(bf16(wl.w))
        self.dy.copy_(bf16(wl.dy))
        self.xw.copy_(bf16(wl.xw))
        self.gate_up.copy_(bf16(wl.gate_up))
        self.moe_x.copy_(bf16(wl.moe_x))
        self.moe_w.copy_(bf16(wl.moe_w))
        self.moe_off.copy_(torch.from_numpy(wl.moe_offsets))
        torch.cuda.synchronize()

    def run(self, stream, ev=None):
        """Launch one step on `stream`.  `ev`, if given, maps kernel name ->
        (start_event, end_event) recorded around that kernel's launches."""
        fg = self.fg

        def rec(name, i):
            if ev is not None:
                ev[name][i].record(stream)

        rec("quant_act_x", 0)
        fg.fp8_quant_act_1x128(self.x, self.xq, self.sx, stream=stream)
        rec("quant_act_x", 1)
        rec("quant_w", 0)
        fg.fp8_quant_w_128x128(self.w, self.wq, self.sw, stream=stream)
        rec("quant_w", 1)
        rec("gemm_fprop", 0)
        fg.fp8_gemm_blockscaled(self.xq, self.sx, self.wq, self.sw, fg.FP8_SB_BLOCK128x128, self.y,
                                stream=stream)
        rec("gemm_fprop", 1)
        rec("quant_act_dy", 0)
        fg.fp8_quant_act_1x128(self.dy, self.dyq, self.sdy, stream=stream)
        rec("quant_act_dy", 1)
        rec("quant_w_rowmajor", 0)
        fg.fp8_quant_w_128x128(self.w, self.wq_rm, self.sw_rm, q_layout=fg.FP8_ROWMAJOR_KN, stream=stream)
        rec("quant_w_rowmajor", 1)
        rec("gemm_dgrad", 0)
        fg.fp8_gemm_blockscaled(self.dyq, self.sdy, self.wq_rm, self.sw_rm.t(), fg.FP8_SB_BLOCK128x128, self.dx,
                                stream=stream)
        rec("gemm_dgrad", 1)
        rec("swiglu_quant", 0)
        fg.fp8_swiglu_quant_1x128(self.gate_up, q=self.hq, s=self.sh, stream=stream)
        rec("swiglu_quant", 1)
        rec("quant_act_xw", 0)
        fg.fp8_quant_act_1x128(self.xw, self.xwq, self.sxw, stream=stream)
        rec("quant_act_xw", 1)
        rec("requant_x", 0)
        fg.fp8_requant_1x128_to_128x1(self.xwq, self.sxw, self.xqT, self.sxT, stream=stream)
        rec("requant_x", 1)
        rec("requant_dy", 0)
        fg.fp8_requant_1x128_to_128x1(self.dyq, self.sdy, self.dyqT, self.sdyT, stream=stream)
        rec("requant_dy", 1)
        rec("gemm_wgrad", 0)
        fg.fp8_gemm_blockscaled(self.xqT, self.sxT, self.dyqT, self.sdyT.t(), fg.FP8_SB_COL128x1, self.dw,
                                stream=stream)
        rec("gemm_wgrad", 1)
        rec("quant_act_moe", 0)
        fg.fp8_quant_act_1x128(self.moe_x, self.mxq, self.smx, stream=stream)
        rec("quant_act_moe", 1)
        rec("quant_w_moe", 0)
        fg.fp8_quant_w_128x128_batched(self.moe_w, self.mwq, self.smw, stream=stream)
        rec("quant_w_moe", 1)
        rec("grouped_gemm_moe", 0)
        fg.fp8_grouped_gemm_blockscaled(self.mxq, self.smx, self.mwq, self.smw, self.moe_off, self.moe_y,
                                        stream=stream)
        rec("grouped_gemm_moe", 1)


    def run_pow2(self, stream, ev=None):
        """The same step with power-of-two scales: the *_pow2 quantizers and the
        GEMMs whose scales the tensor core applies (same buffers and shapes)."""
        fg = self.fg

        def rec(name, i):
            if ev is not None:
                ev[name][i].record(stream)

        def k(name, fn, *a, **kw):
            rec(name, 0)
            fn(*a, **kw)
            rec(name, 1)
        k("quant_act_x", fg.fp8_quant_act_1x128_pow2, self.x, self.xq, self.sx, stream=stream)
        k("quant_w", fg.fp8_quant_w_128x128_pow2, self.w, self.wq, self.sw, stream=stream)
        k("gemm_fprop", fg.fp8_gemm_blockscaled_mx, self.xq, self.sx, self.wq, self.sw, fg.FP8_SB_BLOCK128x128,
          self.y, stream=stream)
        k("quant_act_dy", fg.fp8_quant_act_1x128_pow2, self.dy, self.dyq, self.sdy, stream=stream)
        k("quant_w_rowmajor", fg.fp8_quant_w_128x128_pow2, self.w, self.wq_rm, self.sw_rm,
          q_layout=fg.FP8_ROWMAJOR_KN, stream=stream)
        k("gemm_dgrad", fg.fp8_gemm_blockscaled_mx, self.dyq, self.sdy, self.wq_rm, self.sw_rm.t(),
          fg.FP8_SB_BLOCK128x128, self.dx, stream=stream)
        k("swiglu_quant", fg.fp8_swiglu_quant_1x128, self.gate_up, q=self.hq, s=self.sh, stream=stream)
        k("quant_act_xw", fg.fp8_quant_act_1x128_pow2, self.xw, self.xwq, self.sxw, stream=stream)
        k("requant_x", fg.fp8_requant_1x128_to_128x1_pow2, self.xwq, self.sxw, self.xqT, self.sxT, stream=stream)
        k("requant_dy", fg.fp8_requant_1x128_to_128x1_pow2, self.dyq, self.sdy, self.dyqT, self.sdyT,
          stream=stream)
        k("gemm_wgrad", fg.fp8_gemm_blockscaled_mx, self.xqT, self.sxT, self.dyqT, self.sdyT.t(),
          fg.FP8_SB_COL128x1, self.dw, stream=stream)
        k("quant_act_moe", fg.fp8_quant_act_1x128_pow2, self.moe_x, self.mxq, self.smx, stream=stream)
        k("quant_w_moe", fg.fp8_quant_w_128x128_batched_pow2, self.moe_w, self.mwq, self.smw, stream=stream)
        k("grouped_gemm_moe", fg.fp8_grouped_gemm_blockscaled_mx, self.mxq, self.smx, self.mwq, self.smw,
          self.moe_off, self.moe_y, stream=stream)


# ------------------------------------------------------------- helpers ----

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return {k: float(pk[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# Dense FP8 tensor-core rate per clock of the whole chip: 148 SMs x 8192 FP8
# multiply-adds per SM per clock x 2 flops (4.93 PFLOP/s at the 2032 MHz
# maximum SM clock).  Used only for the clock-scaled context fraction.
NOMINAL_FP8_FLOP_PER_CLK = 148 * 8192 * 2

# Nominal HBM3e bandwidth the quantizers are also quoted against ("about
# 8 TB/s"); the roofline fraction itself uses the measured copy bandwidth.
NOMINAL_HBM_GBS = 8000.0


def choose_fp8_peak(ms_total, clk, burst, sustained):
    """The FP8 roofline denominator: the burst figure (cuBLAS bf16 timed alone,
    x2) for a timed region shorter than one second or one whose median SM
    clock stayed within 5% of the maximum; the sustained figure (a seconds-long
    bf16 loop under the power cap, x2) otherwise.  Returns (peak, rule)."""
    sm, smax = clk.get("sm_mhz"), clk.get("sm_max_mhz")
    if ms_total < 1000.0:
        return burst, "burst: timed region %.2f s < 1 s" % (ms_total / 1e3)
    if sm and smax and sm >= 0.95 * smax:
        return burst, "burst: median SM clock %.0f MHz within 5%% of %.0f" % (sm, smax)
    return sustained, "sustained: timed region %.2f s, median SM clock %s MHz" % (ms_total / 1e3, sm)


def load_tensor_pipe():
    """ncu tensor-pipe activity (% of cycles) of each GEMM from the committed
    profile summary, valid only while the kernel sources are unchanged."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return {}
    if t.get("source_hash") != kernel_source_hash():
        return {}
    return t.get("tensor_pipe_active_pct", {})


def kernel_source_hash():
    h = hashlib.sha256()
    for f in ("ptx.cuh", "quant.cuh", "gemm.cuh", "gemm_mx.cuh", "swiglu.cuh", "fp8fg.cu"):
        with open(os.path.join(ROOT, "fp8_fine_grained_20_b300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def load_traffic():
    """Per-launch DRAM bytes of each kernel from the committed ncu summary, valid
    only while the kernel sources are unchanged since the capture."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return {}
    if t.get("source_hash") != kernel_source_hash():
        return {}
    return t.get("bytes_per_launch", {})


class NvmlClockSampler:
    """Clock / throttle-reason / power samples every 5 ms from a background
    thread through NVML (libnvidia-ml, the library nvidia-smi reads, called
    through ctypes), so that even a timed region of a tenth of a second gets
    tens of samples; only samples whose times fall inside the window given to
    stop() are kept."""
    INTERVAL_S = 0.005
    CLOCK_SM = 1
    REASONS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20, "hw_thermal_slowdown": 0x40}

    def __init__(self, pci_bus_id):
        import ctypes
        self.ct = ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit_v2 failed")
        self.lib = lib
        self.h = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(pci_bus_id.encode()), ctypes.byref(self.h)) != 0:
            if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(0), ctypes.byref(self.h)) != 0:
                raise RuntimeError("no NVML handle for %s" % pci_bus_id)
        v = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(self.h, self.CLOCK_SM, ctypes.byref(v)) != 0:
            raise RuntimeError("nvmlDeviceGetMaxClockInfo failed")
        self.max_mhz = float(v.value)
        self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self.rows = []
        self.stop_flag = None
        self.thread = None

    def _sample(self):
        ct, lib = self.ct, self.lib
        mhz, mw, bits = ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        if (lib.nvmlDeviceGetClockInfo(self.h, self.CLOCK_SM, ct.byref(mhz)) != 0 or
                lib.nvmlDeviceGetPowerUsage(self.h, ct.byref(mw)) != 0 or
                self.reasons_fn(self.h, ct.byref(bits)) != 0):
            return None
        return (time.time(), float(mhz.value), mw.value / 1000.0,
                {n for n, b in self.REASONS.items() if bits.value & b})

    def _run(self):
        while not self.stop_flag.is_set():
            r = self._sample()
            if r is not None:
                self.rows.append(r)
            self.stop_flag.wait(self.INTERVAL_S)

    def start(self):
        import threading
        self.stop_flag = threading.Event()
        self.thread = threading.Thread(target=self._run, daemon=True)
        self.thread.start()

    def stop(self, t0=None, t1=None):
        self.stop_flag.set()
        self.thread.join(timeout=5)
        inside = [r for r in self.rows if t0 is not None and t0 <= r[0] <= t1]
        window = "timed region"
        if not inside:
            inside, window = self.rows, "whole sampling period (no sample inside the timed region)"
        reasons = set()
        for r in inside:
            reasons |= r[3]
        return {"sm_mhz": statistics.median(r[1] for r in inside) if inside else None,
                "sm_max_mhz": self.max_mhz,
                "power_w_median": statistics.median(r[2] for r in inside) if inside else None,
                "samples": len(inside), "window": window, "interval_ms": 1000 * self.INTERVAL_S,
                "source": "nvml", "reasons": sorted(reasons)}


def clock_sampler(pci_bus_id):
    """NVML sampler when the bindings and the device answer, else nvidia-smi."""
    try:
        return NvmlClockSampler(pci_bus_id)
    except Exception as e:   # no bindings, no driver library, no such device
        c = ClockSampler(pci_bus_id)
        c.nvml_error = "%s: %s" % (type(e).__name__, e)
        return c


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples (every 50 ms) while the timed
    region runs; only samples whose timestamps fall inside the window given to
    stop() are kept."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", "fp8fg_clocks_%d_%s.csv" % (os.getpid(), str(gpu_index).replace(":", "_")))

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    @staticmethod
    def _when(stamp):
        import datetime
        for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
            try:
                return datetime.datetime.strptime(stamp, fmt).timestamp()
            except ValueError:
                pass
        return None

    def stop(self, t0=None, t1=None):
        """Summary of the samples taken between wall-clock times t0 and t1
        (all samples if none falls inside)."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    rows.append((self._when(parts[0]), float(parts[2]), float(parts[3]), float(parts[4]),
                                 {n for n, v in zip(names, parts[6:10]) if v.lower().startswith("active")}))
                except ValueError:
                    continue
        try:
            os.remove(self.path)
        except OSError:
            pass
        inside = [r for r in rows if t0 is not None and r[0] is not None and t0 <= r[0] <= t1]
        window = "timed region"
        if not inside:
            inside, window = rows, "whole sampling period (no sample inside the timed region)"
        sm = [r[1] for r in inside]
        reasons = set()
        for r in inside:
            reasons |= r[4]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(r[2] for r in inside) if inside else None,
                "power_w_median": statistics.median(r[3] for r in inside) if inside else None,
                "samples": len(inside), "window": window, "interval_ms": 50, "source": "nvidia-smi",
                "nvml_error": getattr(self, "nvml_error", None), "reasons": sorted(reasons)}


# ------------------------------------------------------- CPU oracle leg ----

def smi_id(torch, local):
    """nvidia-smi selector of this rank's GPU: its PCI bus id when torch knows it."""
    p = torch.cuda.get_device_properties(local)
    try:
        return "%08X:%02X:%02X.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
    except AttributeError:
        return str(local)


def cpu_oracle_sample(wl, frac, threads=1):
    """Run the CPU oracle on a bounded sample of the step: a fraction `frac` of
    every quantizer's groups and of every GEMM's output elements.  Returns
    (seconds, description, extrapolated full-step seconds)."""
    import oracle
    rng = np.random.default_rng(0)
    t_total = 0.0
    parts = []

    def timed(fn):
        t0 = time.perf_counter()
        out = fn()
        return out, time.perf_counter() - t0

    # 1x128 activation quantization: whole rows
    act_elems = {"x": (wl.x, T * CIN), "dy": (wl.dy, T * COUT), "xw": (wl.xw, T * CIN),
                 "moe": (wl.moe_x, wl.moe_rows * MOE_K)}
    est = 0.0
    for name, (arr, n_full) in act_elems.items():
        rows = max(1, int(round(frac * arr.shape[0])))
        (q, s), dt = timed(lambda: oracle.quant_act_1x128(arr[:rows], threads=threads))
        t_total += dt
        est += dt * n_full / (rows * arr.shape[1])
        parts.append("act %s %d rows" % (name, rows))
    # SwiGLU recompute + 1x128 quantization: whole rows
    rows = max(1, int(round(frac * T)))
    (_, dt) = timed(lambda: oracle.quant_act_1x128(
        oracle.swiglu_bf16(wl.gate_up[:rows, :COUT], wl.gate_up[:rows, COUT:], threads=threads), threads=threads))
    t_total += dt
    est += dt * T / rows
    parts.append("swiglu %d rows" % rows)
    # 128x128 weight quantization: one 128-row block strip, a fraction of its columns
    for name, arr, n_full in (("w", wl.w, CIN * COUT), ("w_rowmajor", wl.w, CIN * COUT),
                              ("moe_w", wl.moe_w[0], G * MOE_K * MOE_N)):
        cols = max(128, int(round(frac * arr.size / 128)) // 128 * 128)
        cols = min(cols, arr.shape[1])
        _, dt = timed(lambda: oracle.quant_w_128x128(np.ascontiguousarray(arr[:128, :cols]), threads=threads))
        t_total += dt
        est += dt * n_full / (128 * cols)
        parts.append("weight %s 128x%d" % (name, cols))
    # requantization: one 128-token block x a fraction of the channels
    for name, arr, n_full in (("x", wl.xw, T * CIN), ("dy", wl.dy, T * COUT)):
        q, s = oracle.quant_act_1x128(arr[:128])
        cols = min(arr.shape[1], max(128, int(round(frac * arr.size / 128)) // 128 * 128))
        _, dt = timed(lambda: oracle.requant_1x128_to_128x1(np.ascontiguousarray(q[:, :cols]),
                                                            np.ascontiguousarray(s[:, :cols // 128]),
                                                            threads=threads))
        t_total += dt
        est += dt * n_full / (128 * cols)
        parts.append("requant %s 128x%d" % (name, cols))
    # GEMMs: sampled output elements (operands: oracle-quantized strips)
    xq, xs = oracle.quant_act_1x128(wl.x[:128])
    wq, ws = oracle.quant_w_128x128(np.ascontiguousarray(wl.w[:, :128]))
    wt = np.ascontiguousarray(wq.T)
    depth = {"fprop": CIN, "dgrad": COUT, "wgrad": T, "moe": MOE_K}
    for name, n_out in (("fprop", T * COUT), ("dgrad", T * CIN), ("wgrad", CIN * COUT),
                        ("moe", wl.routed_rows * MOE_N)):
        k = depth[name]
        cnt = max(16, int(round(frac * n_out)))
        ms = rng.integers(0, 128, cnt)
        ns = rng.integers(0, 128, cnt)
        if k == CIN:
            a, sa, b, sb = xq, xs, wt, ws
        else:  # a deeper reduction: tile the 7168-deep strips up to K
            reps = -(-k // CIN)
            a = np.tile(xq, (1, reps))[:, :k]
            sa = np.tile(xs, (1, reps))[:, :k // 128]
            b = np.tile(wt, (1, reps))[:, :k]
            sb = np.tile(ws, (reps, 1))[:k // 128]
        _, dt = timed(lambda: oracle.gemm_blockscaled_sample(a, sa, b, sb, oracle.SB_BLOCK128x128, ms, ns,
                                                             threads=threads))
        t_total += dt
        est += dt * n_out / cnt
        parts.append("%s %d outputs" % (name, cnt))
    return t_total, "; ".join(parts), est


def oracle_threads():
    """Host threads for the oracle: every core the process may use (at most 32)."""
    try:
        n = len(os.sched_getaffinity(0))
    except AttributeError:
        n = os.cpu_count() or 1
    return max(1, min(32, n))


def calibrate_frac(wl, target_seconds, threads=1):
    """Fraction of the step whose oracle run takes about `target_seconds`."""
    probe = 2e-5
    t, _, est = cpu_oracle_sample(wl, probe, threads=threads)
    return min(1.0, max(1e-7, target_seconds / max(est, 1e-9))), est


# --------------------------------------------------------------- main ----

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value, world, device):
    """The largest of every rank's `value` (a time in ms); `value` itself when
    running alone.  All ranks must call it; the reduction runs on `device`
    (the rank's GPU under NCCL, the CPU under gloo)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_reference(args, world, rank):
    """The CPU oracle as the reference arm: rank 0 only, bounded samples."""
    if rank != 0:
        return
    wl = Workload()
    flops = sum(wl.gemm_flops().values())
    per_step = max(0.05, min(args.cpu_seconds, 150.0 / max(1, args.steps + args.warmup)))
    threads = oracle_threads()
    frac, est_full = calibrate_frac(wl, per_step, threads)
    for _ in range(args.warmup):
        cpu_oracle_sample(wl, frac, threads=threads)
    samples, ests = [], []
    desc = ""
    for _ in range(args.steps):
        t, desc, est = cpu_oracle_sample(wl, frac, threads=threads)
        samples.append(t)
        ests.append(est)
    est_step = statistics.mean(ests)
    value = flops / est_step / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": statistics.mean(samples) * 1e3,
        "extrapolated_ms_per_full_step": est_step * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": wl.describe(),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": "fraction %.3g of each kernel's work per step: %s; ms_per_step is the "
                                   "measured time of that sample, value the step's GEMM work over the "
                                   "sample time scaled to the whole step" % (frac, desc)},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")

    import torch
    import torch.distributed as dist
    import fp8_fine_grained_20_b300 as fg

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=device)
    fg.capi()

    wl = Workload(seed_offset=0)
    step = DeviceStep(wl, device)
    stream = torch.cuda.Stream(device=device)
    flops = wl.gemm_flops()
    qbytes = wl.quant_bytes()
    total_flops = sum(flops.values())

    # warm-up
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step.run(stream)
    torch.cuda.synchronize()
    if fg.fp8_get_device_status(reset=True) != 0:
        raise SystemExit("device status set during warm-up")

    # timed region: K steps, per-kernel events inside, clocks sampled alongside
    evs = [{k: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for k in DeviceStep.KERNELS} for _ in range(args.steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    clocks = clock_sampler(smi_id(torch, local))
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    wall0 = time.time()
    with torch.cuda.stream(stream):
        t0.record(stream)
        for i in range(args.steps):
            step.run(stream, evs[i])
        t1.record(stream)
    torch.cuda.synchronize()
    wall1 = time.time()
    clk = clocks.stop(wall0, wall1)
    if world > 1:
        dist.barrier()
    ms_total = max_over_ranks(t0.elapsed_time(t1), world, device)
    status = fg.fp8_get_device_status(reset=True)
    ms_step = ms_total / args.steps
    value = world * total_flops / (ms_step * 1e-3) / 1e12

    per_kernel_ms = {k: statistics.mean(evs[i][k][0].elapsed_time(evs[i][k][1]) for i in range(args.steps))
                     for k in DeviceStep.KERNELS}
    peaks, peak_src = load_peaks()
    fp8_peak_sustained = peaks["bf16_tflops_sustained"] * FP8_OVER_BF16
    fp8_peak_burst = peaks["bf16_tflops"] * FP8_OVER_BF16
    fp8_peak, peak_rule = choose_fp8_peak(ms_total, clk, fp8_peak_burst, fp8_peak_sustained)
    sm_mhz = clk.get("sm_mhz")
    fp8_nominal = NOMINAL_FP8_FLOP_PER_CLK * sm_mhz * 1e6 / 1e12 if sm_mhz else None
    hbm = peaks["hbm_gbs"]
    traffic = load_traffic()
    pipes = load_tensor_pipe()
    kernels = {}
    for k, ms in per_kernel_ms.items():
        d = {"ms": ms, "launches_per_step": 1}
        if sm_mhz:
            d["kcycles_at_median_clock"] = ms * sm_mhz
        if k in flops:
            tf = flops[k] / (ms * 1e-3) / 1e12
            d.update({"tflops": tf, "frac_fp8": tf / fp8_peak, "frac_fp8_burst": tf / fp8_peak_burst,
                      "frac_fp8_sustained": tf / fp8_peak_sustained})
            if fp8_nominal:
                d["frac_fp8_nominal_at_clock"] = tf / fp8_nominal
            if k in pipes:
                d["ncu_tensor_pipe_active_pct"] = pipes[k]
        else:
            gbs = qbytes[k] / (ms * 1e-3) / 1e9
            d.update({"gbs": gbs, "frac_hbm": gbs / hbm, "frac_hbm_nominal": gbs / NOMINAL_HBM_GBS,
                      "bytes": qbytes[k]})
        kernels[k] = d
    dom = max(per_kernel_ms, key=per_kernel_ms.get)
    if dom in flops:
        ach = flops[dom] / (per_kernel_ms[dom] * 1e-3) / 1e12
        roofline = {"kernel": dom, "bound": "tensor", "achieved": ach, "peak": fp8_peak, "unit": "TFLOP/s",
                    "frac": ach / fp8_peak, "traffic": traffic.get(dom),
                    "peak_source": "%s bf16 x %.0f (nominal FP8/BF16 ratio), %s" % (peak_src, FP8_OVER_BF16,
                                                                                   peak_rule),
                    "frac_nominal_at_clock": (ach / fp8_nominal) if fp8_nominal else None,
                    # ncu sm__pipe_tensor_cycles_active of the same kernel, as a fraction
                    "frac_tensor_pipe": (pipes[dom] / 100.0) if dom in pipes else None}
    else:
        ach = qbytes[dom] / (per_kernel_ms[dom] * 1e-3) / 1e9
        roofline = {"kernel": dom, "bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s",
                    "frac": ach / hbm, "traffic": traffic.get(dom), "peak_source": peak_src + " copy"}
    if roofline["traffic"] is not None:
        roofline["traffic"] = float(roofline["traffic"])

    # steady state: the same step back to back for a few seconds, with tens of
    # clock samples (context for the short timed region above)
    steady = None
    if args.steady_seconds > 0:
        steady = run_steady(args, step, stream, smi_id(torch, local), ms_step, world)

    # the same step with power-of-two scales and tensor-core-applied scaling
    pow2 = None
    if not args.no_pow2:
        pow2 = run_pow2_leg(args, wl, step, stream, flops, qbytes, fp8_peak, hbm, world, device,
                            smi_id(torch, local))

    # end-to-end: pinned host inputs -> device -> step -> outputs back to pinned host
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, wl, step, stream, total_flops, world, device)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        threads = oracle_threads()
        frac, _ = calibrate_frac(wl, args.cpu_seconds, threads)
        secs, desc, est = cpu_oracle_sample(wl, frac, threads=threads)
        cpu = {"value": total_flops / est / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": "fraction %.3g of every kernel's work (%s), %.1f s measured, extrapolated to the "
                         "whole step" % (frac, desc, secs)}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "e4m3", "data": "synthetic", "config": wl.describe(),
            "roofline": roofline, "kernels": kernels,
            "quantizers_gbs": sum(qbytes.values()) / (sum(per_kernel_ms[k] for k in qbytes) * 1e-3) / 1e9,
            "gemms_tflops": total_flops / (sum(per_kernel_ms[k] for k in flops) * 1e-3) / 1e12,
            "fp8_peak_tflops": {"used": fp8_peak, "rule": peak_rule, "sustained": fp8_peak_sustained,
                                "burst": fp8_peak_burst, "nominal_at_median_clock": fp8_nominal,
                                "source": peak_src},
            "hbm_peak_gbs": hbm, "hbm_nominal_gbs": NOMINAL_HBM_GBS,
            "cpu_baseline": cpu, "e2e": e2e, "steady_state": steady, "pow2_mx": pow2,
            "gpu_launches": DeviceStep.LAUNCHES_PER_STEP * args.steps,
            "clocks": clk, "device_status": status,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def path_errors(wl, step, stream, n=2048):
    """Error of the FP8 forward and weight-gradient outputs against the exact
    (FP64) product of the ORIGINAL bf16 inputs, on n sampled outputs each,
    for the promoting path (scales amax/448) and the power-of-two path:
    relative Frobenius error and the largest error relative to rms(exact)."""
    import torch
    rng = np.random.default_rng(99)
    ms, ns = rng.integers(0, T, n), rng.integers(0, COUT, n)
    cs, os_ = rng.integers(0, CIN, n), rng.integers(0, COUT, n)
    f64 = lambda b: synth.f32_from_bf16_bits(b).astype(np.float64)   # noqa: E731
    exact_y = np.einsum("ik,ki->i", f64(wl.x[ms]), f64(wl.w[:, ns]))
    exact_dw = np.einsum("ti,ti->i", f64(wl.xw[:, cs]), f64(wl.dy[:, os_]))
    tm, tn = torch.from_numpy(ms).cuda(), torch.from_numpy(ns).cuda()
    tc, to = torch.from_numpy(cs).cuda(), torch.from_numpy(os_).cuda()

    def errs(got, ref):
        d = got - ref
        rms = np.sqrt(np.mean(ref ** 2))
        return {"rel_frobenius": float(np.linalg.norm(d) / np.linalg.norm(ref)),
                "max_abs_over_rms": float(np.max(np.abs(d)) / rms)}
    out = {}
    for name, run in (("amax_over_448_promoting", step.run), ("power_of_two_mx", step.run_pow2)):
        with torch.cuda.stream(stream):
            run(stream)
        torch.cuda.synchronize()
        y = step.y[tm, tn].double().cpu().numpy()
        dw = step.dw[tc, to].double().cpu().numpy()
        out[name] = {"forward": errs(y, exact_y), "weight_gradient": errs(dw, exact_dw)}
    out["sample"] = "%d forward and %d weight-gradient outputs against FP64 products of the bf16 inputs" % (n, n)
    return out


def run_pow2_leg(args, wl, step, stream, flops, qbytes, fp8_peak, hbm, world, device, gpu):
    """Time the power-of-two step exactly as the main step is timed (warm-up,
    args.steps steps between events, per-kernel events, clocks sampled through
    its own timed region) and compare the two paths' errors."""
    import torch
    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            step.run_pow2(stream)
    torch.cuda.synchronize()
    evs = [{k: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for k in DeviceStep.KERNELS} for _ in range(args.steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    clocks = clock_sampler(gpu)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    wall0 = time.time()
    with torch.cuda.stream(stream):
        t0.record(stream)
        for i in range(args.steps):
            step.run_pow2(stream, evs[i])
        t1.record(stream)
    torch.cuda.synchronize()
    wall1 = time.time()
    clk = clocks.stop(wall0, wall1)
    ms_step = max_over_ranks(t0.elapsed_time(t1), world, device) / args.steps
    kernels = {}
    for k in DeviceStep.KERNELS:
        ms = statistics.mean(evs[i][k][0].elapsed_time(evs[i][k][1]) for i in range(args.steps))
        d = {"ms": ms}
        if k in flops:
            tf = flops[k] / (ms * 1e-3) / 1e12
            d.update({"tflops": tf, "frac_fp8": tf / fp8_peak})
        else:
            gbs = qbytes[k] / (ms * 1e-3) / 1e9
            d.update({"gbs": gbs, "frac_hbm": gbs / hbm, "frac_hbm_nominal": gbs / NOMINAL_HBM_GBS})
        kernels[k] = d
    status = step.fg.fp8_get_device_status(reset=True)
    return {"ms_per_step": ms_step, "value": world * sum(flops.values()) / (ms_step * 1e-3) / 1e12,
            "unit": UNIT, "kernels": kernels, "device_status": status, "clocks": clk,
            "errors_vs_exact_bf16_product": path_errors(wl, step, stream),
            "note": "same step, *_pow2 quantizers and the hardware block-scaled GEMMs (scales applied by "
                    "the tensor core, no FP32 promotion); not the headline"}


def run_steady(args, step, stream, gpu, ms_step, world):
    """Run the step back to back for about args.steady_seconds with an event
    pair around every step, sampling clocks (every 5 ms through NVML, else
    every 50 ms through nvidia-smi).  Returns the median, minimum and
    last-quarter step times and the clock record of that run."""
    import torch
    n = max(10, int(args.steady_seconds * 1e3 / max(ms_step, 1e-3)))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    clocks = clock_sampler(gpu)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    wall0 = time.time()
    with torch.cuda.stream(stream):
        for i in range(n):
            evs[i][0].record(stream)
            step.run(stream)
            evs[i][1].record(stream)
    torch.cuda.synchronize()
    wall1 = time.time()
    clk = clocks.stop(wall0, wall1)
    ms = [a.elapsed_time(b) for a, b in evs]
    return {"steps": n, "seconds": wall1 - wall0, "ms_per_step_median": statistics.median(ms),
            "ms_per_step_min": min(ms), "ms_per_step_last_quarter": statistics.median(ms[3 * n // 4:]),
            "clocks": clk, "note": "not the timed region; per-rank figures, rank 0 printed" if world > 1 else
            "not the timed region"}


def run_e2e(args, wl, step, stream, total_flops, world, device):
    """The step through the public API with host buffers: every step copies
    its bf16 inputs from pinned host memory and its four bf16 outputs back.
    Two device buffer sets alternate, so the host-to-device copies of step
    i + 1 (copy stream), the kernels of step i (compute stream) and the
    device-to-host copies of step i - 1 (a third stream) overlap; events keep
    each buffer set's copies and kernels in order.  All copies of all steps
    are inside the timed region."""
    import torch

    def pinned(a, dtype=None):
        t = torch.from_numpy(np.ascontiguousarray(a))
        if dtype is not None:
            t = t.view(dtype)
        return t.pin_memory()
    h_in = [pinned(wl.x.view(np.int16), torch.bfloat16), pinned(wl.w.view(np.int16), torch.bfloat16),
            pinned(wl.dy.view(np.int16), torch.bfloat16), pinned(wl.xw.view(np.int16), torch.bfloat16),
            pinned(wl.gate_up.view(np.int16), torch.bfloat16), pinned(wl.moe_x.view(np.int16), torch.bfloat16),
            pinned(wl.moe_w.view(np.int16), torch.bfloat16), pinned(wl.moe_offsets)]
    sets = [step, DeviceStep(wl, device)]

    def dev_in(st):
        return [st.x, st.w, st.dy, st.xw, st.gate_up, st.moe_x, st.moe_w, st.moe_off]

    def dev_out(st):
        return [st.y, st.dx, st.dw, st.moe_y]
    h_out = [[torch.empty(d.shape, dtype=d.dtype).pin_memory() for d in dev_out(st)] for st in sets]
    h2d = sum(h.numel() * h.element_size() for h in h_in)
    d2h = sum(h.numel() * h.element_size() for h in h_out[0])
    s_h2d = torch.cuda.Stream(device=device)
    s_d2h = torch.cuda.Stream(device=device)
    ev = [{k: torch.cuda.Event() for k in ("h2d", "compute", "d2h")} for _ in sets]

    def one(i):
        j = i % 2
        st, e = sets[j], ev[j]
        if i >= 2:
            s_h2d.wait_event(e["compute"])          # the kernels of step i - 2 no longer read these inputs
        with torch.cuda.stream(s_h2d):
            for h, d in zip(h_in, dev_in(st)):
                d.copy_(h, non_blocking=True)
        e["h2d"].record(s_h2d)
        stream.wait_event(e["h2d"])
        if i >= 2:
            stream.wait_event(e["d2h"])             # step i - 2's outputs are on the host
        st.run(stream)
        e["compute"].record(stream)
        s_d2h.wait_event(e["compute"])
        with torch.cuda.stream(s_d2h):
            for d, h in zip(dev_out(st), h_out[j]):
                h.copy_(d, non_blocking=True)
        e["d2h"].record(s_d2h)

    for i in range(2):                               # warm-up of both buffer sets
        one(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    e0.record(s_h2d)
    for i in range(args.e2e_steps):
        one(i)
    stream.wait_event(ev[(args.e2e_steps - 1) % 2]["d2h"])
    stream.wait_event(ev[args.e2e_steps % 2]["d2h"])
    e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1), world, device)
    ms_step = ms / args.e2e_steps
    del sets[1]
    torch.cuda.empty_cache()
    # restore the device-resident inputs used by later legs
    step.load_inputs(wl)
    return {"value": world * total_flops / (ms_step * 1e-3) / 1e12, "unit": UNIT, "ms_per_step": ms_step,
            "steps": args.e2e_steps, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "overlap": "two device buffer sets; host-to-device, kernels and device-to-host on three streams"}


if __name__ == "__main__":
    main()
