"""Benchmark of the W4A4 MoE expert-MLP hot path on GB300.

One step = one pass of the whole path over one batch of the skewed-load
Qwen3-30B-A3B-shaped layer (32768 tokens, hidden 2048, 128 experts top-8,
intermediate 768, Zipf(1.2) expert load with empty experts):

  weight quant (W_gate_up along K; W_down along K and along N, the dgrad
  layout with the same global scales, from one read)
  -> permute + per-token amax + NVFP4 quant of x
  -> grouped gate_up GEMM -> weighted SwiGLU + requant -> grouped down GEMM
  -> combine
  -> combine backward: dY to the forward's permuted rows, quantized per token
  -> grouped dgrad GEMM (dH).

Prints one JSON line. ``value`` is tokens/s over all ranks with inputs
resident in HBM; ``e2e`` repeats the step through the same C-ABI calls with
inputs in pinned host memory, copied in (and y copied out) inside the timed
region; ``backward`` times the rest of the NVFP4 backward beside the step
(W_gate_up's dgrad copy, SwiGLU backward, gate_up dgrad GEMM, dX combine,
token-axis operands, weight-gradient GEMMs). ``--impl reference`` times the
CPU oracle on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "NVFP4 grouped-GEMM TFLOP/s (% FP4 peak); MoE expert-MLP tokens/s, 1 GB300"
WORKLOAD = "skewed"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="minite", choices=["minite", "reference"])
    ap.add_argument("--workload", default=WORKLOAD, choices=["skewed", "mlp", "gate_up", "tiny"])
    ap.add_argument("--gemm-variant", type=int, default=0,
                    help="grouped-GEMM kernel: 0 automatic, 1 single-CTA one-chunk stages,"
                         " 5 single-CTA two-chunk stages, 6 CTA pair with five stages")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-backward", action="store_true",
                    help="skip timing the rest of the NVFP4 backward beside the step")
    ap.add_argument("--no-graph", action="store_true",
                    help="time eager launches only (default: the step replayed as one CUDA graph)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-sample-tokens", type=int, default=4096,
                    help="reference arm: tokens of the workload's batch each oracle step runs on")
    ap.add_argument("--cpu-baseline-reps", type=int, default=2)
    ap.add_argument("--cpu-baseline-only", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per-configuration measurements")
    ap.add_argument("--no-fused", action="store_true",
                    help="skip the fused gate_up + SwiGLU comparison")
    return ap.parse_args()


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- peaks

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sus=d["bf16_tflops_sustained"],
                    source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, source="fallback")


FP4_OVER_BF16 = 13.5 / 2.25  # nominal dense FP4 / BF16 tensor rates


def percentile(xs, q):
    """q-th percentile (linear interpolation) of a non-empty list."""
    s = sorted(xs)
    pos = (len(s) - 1) * q / 100.0
    lo = int(pos)
    hi = min(lo + 1, len(s) - 1)
    return s[lo] + (s[hi] - s[lo]) * (pos - lo)


# grouped-GEMM kernel of each `--gemm-variant` (0 = automatic = 6 on these shapes)
GEMM_KERNELS = {1: "grouped_gemm_kernel", 5: "grouped_gemm_dc_kernel",
                6: "grouped_gemm_pair_deep_kernel"}


def max_over_ranks(values, device):
    """Element-wise maximum of `values` (floats) over all ranks of the default
    process group (NCCL on GPUs, gloo in the CPU tests); identity when there
    is no process group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return list(values)
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def workload_name(name, cfg):
    """The `config.workload` string of both arms."""
    return f"{name}: T={cfg['T']} H={cfg['H']} E={cfg['E']} top{cfg['k']} I={cfg['I']}"


# ----------------------------------------------------------------------------- GPU step

class Step:
    """All device buffers of one step; ``run`` enqueues the whole path."""

    STAGES = ["wq_gate_up", "wq_down_both", "permute_x", "gemm_gate_up", "swiglu", "gemm_down",
              "combine", "combine_bwd_quant_dy", "gemm_dgrad"]

    def __init__(self, d, dev):
        import torch
        from nvfp4_w4a4_moe_permute_gb300 import minite as M
        self.M = M
        c = d["cfg"]
        self.T, self.H, self.E, self.k, self.I = c["T"], c["H"], c["E"], c["k"], c["I"]
        T, H, E, k, I = self.T, self.H, self.E, self.k, self.I
        bf = torch.bfloat16
        self.dev = dev

        def to_dev(a, dtype=None):
            import numpy as np
            if a.dtype == np.uint16:
                return torch.from_numpy(a.view(np.int16)).view(bf).to(dev)
            return torch.from_numpy(a).to(dev)

        self.to_dev = to_dev
        self.x = to_dev(d["x"])
        self.ids = to_dev(d["topk_ids"])
        self.w = to_dev(d["topk_w"])
        self.wgu_bf = to_dev(d["w_gate_up"])
        self.wd_bf = to_dev(d["w_down"])
        self.dy = to_dev(d["dy"]) if "dy" in d else to_dev(d["x"])
        u8, f32 = torch.uint8, torch.float32
        kc = lambda c: ((c // 16) + 3) // 4 * 4  # noqa: E731
        rp = lambda r: (r + 127) // 128 * 128  # noqa: E731
        # quantized weights (forward K-major) and the dgrad copy of W_down
        self.wgu = dict(codes=torch.empty((E, 2 * I, H // 2), dtype=u8, device=dev),
                        sf=torch.empty((E, rp(2 * I) * kc(H)), dtype=u8, device=dev),
                        g=torch.empty(E, dtype=f32, device=dev))
        self.wd = dict(codes=torch.empty((E, H, I // 2), dtype=u8, device=dev),
                       sf=torch.empty((E, rp(H) * kc(I)), dtype=u8, device=dev),
                       g=torch.empty(E, dtype=f32, device=dev))
        self.wdT = dict(codes=torch.empty((E, I, H // 2), dtype=u8, device=dev),
                        sf=torch.empty((E, rp(I) * kc(H)), dtype=u8, device=dev),
                        g=torch.empty(E, dtype=f32, device=dev))
        self.ws_q = torch.empty(M.minite_workspace_bytes(M.OP_QUANTIZE, E), dtype=u8, device=dev)
        self.mlp = M.MoEMLP(T, H, I, E, k, dev)
        self.bwd = M.MoEMLP(T, H, I, E, k, dev)  # permuted dY buffers (same routing)
        self.ws_cb = torch.empty(M.minite_workspace_bytes(M.OP_COMBINE_BACKWARD_QUANT, T, H),
                                 dtype=u8, device=dev)
        self.dh = torch.empty((T * k, I), dtype=bf, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.mlp.status = self.status
        self.bwd.status = self.status

    def bind(self, inputs, y):
        """Use the device tensors in `inputs` (any of x, ids, w, wgu_bf, wd_bf, dy)
        as this step's inputs and `y` as its output."""
        for n, t in inputs.items():
            setattr(self, n, t)
        self.mlp.y = y

    def run(self, stream, events=None, ready=None, y_done=None):
        """Enqueue the step on `stream`. `ready`: optional CUDA events of the
        step's input copies; the permutation waits for ready["x"] (x, ids and
        w) and the combine backward for ready["dy"]; the weight quantization
        needs neither (the weights are device-resident model state).
        `y_done`: optional event recorded once y is complete (after the
        combine), so that its read-back can overlap the rest of the step."""
        M, s = self.M, stream

        def mark(i):
            if events is not None:
                events[i].record(s)

        mark(0)
        M.minite_quantize_nvfp4(self.wgu_bf, M.SCALE_PER_GROUP, M.ALONG_COLS, self.wgu["codes"],
                                self.wgu["sf"], self.wgu["g"], None, self.ws_q, self.status, s)
        mark(1)
        # W_down in both orientations (forward K-major and the dgrad copy along N)
        M.minite_quantize_nvfp4_dual(self.wd_bf, self.wd["codes"], self.wd["sf"], self.wdT["codes"],
                                     self.wdT["sf"], self.wd["g"], self.ws_q, self.status, s)
        mark(2)
        if ready is not None:
            s.wait_event(ready["x"])
        mlp = self.mlp
        mlp.permute_quant(self.x, self.ids, self.w, s)
        mark(3)
        M.minite_grouped_gemm_nvfp4(mlp.a_codes, mlp.a_sf, mlp.a_g, self.wgu["codes"],
                                    self.wgu["sf"], self.wgu["g"], mlp.offsets, mlp.sf_offsets,
                                    mlp.gate_up, self.status, s)
        mark(4)
        M.minite_swiglu_weighted_quant(mlp.gate_up, mlp.perm_w, self.E, mlp.offsets,
                                       mlp.sf_offsets, mlp.h_codes, mlp.h_sf, mlp.h_g,
                                       self.status, s)
        mark(5)
        M.minite_grouped_gemm_nvfp4(mlp.h_codes, mlp.h_sf, mlp.h_g, self.wd["codes"],
                                    self.wd["sf"], self.wd["g"], mlp.offsets, mlp.sf_offsets,
                                    mlp.down, self.status, s)
        mark(6)
        M.minite_moe_combine(mlp.down, mlp.dest_row, mlp.y, self.status, s)
        if y_done is not None:
            y_done.record(s)
        mark(7)
        if ready is not None:
            s.wait_event(ready["dy"])
        # backward of the combine: dY to the forward's permuted rows, quantized
        b = self.bwd
        M.minite_moe_combine_backward_quant(self.dy, self.E, mlp.dest_row, mlp.offsets,
                                            mlp.sf_offsets, mlp.perm_src, b.a_codes, b.a_sf,
                                            b.a_g, self.ws_cb, self.status, s)
        mark(8)
        M.minite_grouped_gemm_nvfp4(b.a_codes, b.a_sf, b.a_g, self.wdT["codes"], self.wdT["sf"],
                                    self.wd["g"], mlp.offsets, mlp.sf_offsets, self.dh,
                                    self.status, s)
        mark(9)

    # The rest of the NVFP4 backward of the expert MLP, timed beside the step:
    # W_gate_up's dgrad copy (blocks along N, with the global scales the
    # forward step computed), SwiGLU backward with its per-row requantization,
    # the gate_up dgrad GEMM (K = 2I, N = H), the combine of dX back into token
    # order, the token-axis operands and the two weight-gradient GEMMs.
    BWD_STAGES = ["wq_gate_up_T", "swiglu_keep_h", "swiglu_bwd_keep", "gemm_dgrad_gate_up",
                  "combine_dx", "quant_tokens", "gemm_wgrad_down", "gemm_wgrad_gate_up"]
    # W_gate_up along N 1 (no maxima pass), SwiGLU 1, SwiGLU backward 1, GEMM 1, combine 1, token-axis operands (gathered dY
    # and x: source-row maxima, expert maxima, encoding; h and [dg | du] with their producers'
    # row maxima: expert maxima, encoding) 3 + 2 + 2 + 3, 2 GEMMs
    BWD_LAUNCHES = 1 + 1 + 1 + 1 + 1 + 10 + 2

    def init_backward(self):
        import torch
        T, H, E, k, I = self.T, self.H, self.E, self.k, self.I
        dev, u8, f32 = self.dev, torch.uint8, torch.float32
        M_ = T * k
        self.wguT = dict(codes=torch.empty((E, H, I), dtype=u8, device=dev),
                         sf=torch.empty((E, self.M.sf_bytes((H + 127) // 128 * 128, 2 * I)),
                                        dtype=u8, device=dev))
        self.dgu = dict(codes=torch.empty((M_, I), dtype=u8, device=dev),
                        sf=torch.empty(self.M.sf_bytes(M_ + 128 * E, 2 * I), dtype=u8, device=dev),
                        g=torch.empty(M_, dtype=f32, device=dev))
        self.dx_perm = torch.empty((M_, H), dtype=torch.bfloat16, device=dev)
        self.dx = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        # weight gradients: BF16 h and [dg | du] kept, their token-axis operands
        self.h_bf = torch.zeros((M_, I), dtype=torch.bfloat16, device=dev)
        self.dgu_bf = torch.zeros((M_, 2 * I), dtype=torch.bfloat16, device=dev)
        # their row maxima, written by the SwiGLU passes that produce them
        self.h_amax = torch.zeros(M_, dtype=f32, device=dev)
        self.dgu_amax = torch.zeros(M_, dtype=f32, device=dev)
        mlp = self.mlp
        self.tok = {}
        for name, src, rs, ra in (("dy", self.dy, mlp.perm_src, None),
                                  ("h", self.h_bf, None, self.h_amax),
                                  ("dgu", self.dgu_bf, None, self.dgu_amax),
                                  ("x", self.x, mlp.perm_src, None)):
            self.tok[name] = (src, rs, ra, self.M.quantize_tokens(src, mlp.offsets, E, row_src=rs,
                                                                  m_cap=M_))
        self.ws_tok = torch.empty(max(4, self.M.minite_workspace_bytes(self.M.OP_QUANTIZE_TOKENS, E,
                                                                       T)),
                                  dtype=u8, device=dev)
        self.dWd = torch.empty((E, H, I), dtype=f32, device=dev)
        self.dWgu = torch.empty((E, 2 * I, H), dtype=f32, device=dev)

    def run_backward(self, stream, events=None):
        M, s, mlp = self.M, stream, self.mlp

        def mark(i):
            if events is not None:
                events[i].record(s)

        mark(0)
        # the dgrad copy of W_gate_up, with the forward step's per-expert g
        M.minite_quantize_nvfp4(self.wgu_bf, M.SCALE_PER_GROUP, M.ALONG_ROWS, self.wguT["codes"],
                                self.wguT["sf"], self.wgu["g"], self.wgu["g"], None, self.status, s)
        mark(1)
        # the forward's SwiGLU keeping BF16 h for the down projection's weight gradient
        M.minite_swiglu_weighted_quant_keep_h(mlp.gate_up, mlp.perm_w, self.E, mlp.offsets,
                                              mlp.sf_offsets, mlp.h_codes, mlp.h_sf, mlp.h_g,
                                              self.h_bf, self.status, s, h_amax=self.h_amax)
        mark(2)
        M.minite_swiglu_backward_quant_keep(mlp.gate_up, self.dh, mlp.perm_w, self.E, mlp.offsets,
                                            mlp.sf_offsets, self.dgu["codes"], self.dgu["sf"],
                                            self.dgu["g"], self.dgu_bf, self.status, s,
                                            dgu_amax=self.dgu_amax)
        mark(3)
        M.minite_grouped_gemm_nvfp4(self.dgu["codes"], self.dgu["sf"], self.dgu["g"],
                                    self.wguT["codes"], self.wguT["sf"], self.wgu["g"],
                                    mlp.offsets, mlp.sf_offsets, self.dx_perm, self.status, s)
        mark(4)
        M.minite_moe_combine(self.dx_perm, mlp.dest_row, self.dx, self.status, s)
        mark(5)
        M_ = self.T * self.k
        for src, rs, ra, q in self.tok.values():
            M.minite_quantize_tokens_nvfp4(src, rs, M_, self.E, mlp.offsets, q["k_cap"], q["codes"],
                                           q["sf"], q["g"], q["kofs"], self.ws_tok, self.status, s,
                                           row_amax=ra)
        mark(6)
        M.minite_grouped_gemm_wgrad_nvfp4(self.tok["dy"][3], self.tok["h"][3], self.dWd,
                                          self.status, s)
        mark(7)
        M.minite_grouped_gemm_wgrad_nvfp4(self.tok["dgu"][3], self.tok["x"][3], self.dWgu,
                                          self.status, s)
        mark(8)

    # kernels launched per step by the library (memsets not counted): weight
    # quantization 2 + 2, permutation 4 (rank, scan, quant, scale gather),
    # GEMM 1, SwiGLU 1, GEMM 1, combine 1, combine backward with dY
    # quantization 2, GEMM 1
    LAUNCHES = 2 + 2 + 4 + 1 + 1 + 1 + 1 + 2 + 1

    def flops(self):
        Mu = int(self.mlp.offsets[-1].item())
        H, I = self.H, self.I
        return dict(gemm_gate_up=2.0 * Mu * 2 * I * H, gemm_down=2.0 * Mu * H * I,
                    gemm_dgrad=2.0 * Mu * I * H, used_rows=Mu)

    def gemm_gate_up_bytes(self):
        """Bytes the gate_up GEMM must move at minimum: A codes and scales (rows
        padded to 128 per expert), every expert's W codes and scales once, the
        BF16 output."""
        Mu = int(self.mlp.offsets[-1].item())
        Mp = int(self.mlp.sf_offsets[-1].item())
        H, I, E = self.H, self.I, self.E
        return (Mu * H / 2 + Mp * H / 16 + E * 2 * I * H / 2 + E * 2 * I * H / 16 +
                Mu * 2 * I * 2)

    def backward_algorithmic_bytes(self):
        """Bytes each backward stage must move at minimum (read once + write once)."""
        T, H, E, k, I = self.T, self.H, self.E, self.k, self.I
        Mu = int(self.mlp.offsets[-1].item())
        sfb = lambda r, c: r * c / 16  # noqa: E731
        return dict(
            wq_gate_up_T=E * 2 * I * H * 2 + E * 2 * I * H / 2 + sfb(E * 2 * I, H),
            # + the kept BF16 rows and their row maxima
            swiglu_keep_h=Mu * 2 * I * 2 + Mu * (I / 2 + I / 16 + 4) + Mu * (I * 2 + 4),
            swiglu_bwd_keep=Mu * (2 * I * 2 + I * 2 + 4) + Mu * (I + 2 * I / 16 + 4) +
            Mu * (2 * I * 2 + 4),
            combine_dx=Mu * H * 2 + T * H * 2 + T * k * 4,
            # four operands: each permuted row read once, codes + scales written
            quant_tokens=sum(Mu * C * 2 + Mu * C / 2 + Mu * C / 16 for C in (H, I, 2 * I, H)),
        )

    def algorithmic_bytes(self):
        """Bytes each stage must move at minimum (read once + write once)."""
        T, H, E, k, I = self.T, self.H, self.E, self.k, self.I
        Mu = int(self.mlp.offsets[-1].item())
        sfb = lambda r, c: r * c / 16  # noqa: E731  one scale byte per 16 values
        return dict(
            wq_gate_up=E * 2 * I * H * 2 + E * 2 * I * H / 2 + sfb(E * 2 * I, H),
            wq_down_both=E * H * I * 2 + E * H * I + sfb(E * H, I) + sfb(E * I, H),
            permute_x=T * H * 2 + T * k * 8 + Mu * (H / 2 + H / 16 + 4 + 12),
            swiglu=Mu * 2 * I * 2 + Mu * (I / 2 + I / 16 + 4),
            combine=Mu * H * 2 + T * H * 2 + T * k * 4,
            combine_bwd_quant_dy=T * H * 2 + T * k * 4 + Mu * (H / 2 + H / 16 + 4 + 4),
        )


def time_launches(fn, stream, reps=10, warmup=3, flush=None):
    """Per-launch times (ms) of `fn()` on `stream` from CUDA events recorded
    around each launch; `flush` (a device buffer larger than L2) is
    overwritten before every launch so that no launch finds its inputs in L2."""
    import torch
    for _ in range(warmup):
        fn()
    out = []
    for _ in range(reps):
        if flush is not None:
            flush.fill_(1)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        e1.synchronize()
        out.append(e0.elapsed_time(e1))
    return out


def fused_gate_up_swiglu(step, stream, dev, reps=10):
    """The fused gate_up GEMM + weighted SwiGLU + requantization
    (minite_gate_up_swiglu_quant_nvfp4, no BF16 gate_up kept) against the
    gate_up GEMM followed by the SwiGLU kernel, both on the step's buffers,
    L2 flushed before every launch (median, p10, p90 of `reps`)."""
    import torch

    from nvfp4_w4a4_moe_permute_gb300 import minite as M
    mlp = step.mlp
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)

    def stats(ts):
        return {"median": round(statistics.median(ts), 5), "p10": round(percentile(ts, 10), 5),
                "p90": round(percentile(ts, 90), 5)}

    def unfused():
        M.minite_grouped_gemm_nvfp4(mlp.a_codes, mlp.a_sf, mlp.a_g, step.wgu["codes"],
                                    step.wgu["sf"], step.wgu["g"], mlp.offsets, mlp.sf_offsets,
                                    mlp.gate_up, mlp.status, stream)
        M.minite_swiglu_weighted_quant(mlp.gate_up, mlp.perm_w, mlp.E, mlp.offsets,
                                       mlp.sf_offsets, mlp.h_codes, mlp.h_sf, mlp.h_g,
                                       mlp.status, stream)

    tu = time_launches(unfused, stream, reps=reps, flush=flush)
    tf = time_launches(lambda: mlp.gate_up_swiglu(step.wgu, stream, fused=True), stream,
                       reps=reps, flush=flush)
    torch.cuda.synchronize(dev)
    assert int(mlp.status.item()) == 0
    return {"workload": "the benchmarked step's gate_up layer",
            "fused_ms": stats(tf), "gemm_then_swiglu_ms": stats(tu),
            "used_in_step": False}


def per_config(dev, fp4_peak, peaks):
    """The other configurations the metric names, each timed per launch with
    L2 flushed before every launch (median, p10, p90 of 10):
      dense: the single NVFP4 GEMM M=4096 N=1536 K=2048 (A quantized per row,
        1% outlier channels x20), BF16 and FP32 output, and the quantization
        of A;
      gate_up layer (4096 tokens, 128 experts top-8): the permutation with
        fused quantization and the gate_up grouped GEMM;
      MLP forward (4096 tokens): permutation -> gate_up GEMM -> SwiGLU ->
        down GEMM -> combine, as one timed unit (weights quantized before).
    The gate_up layer and the MLP forward use the same seeded batch."""
    import numpy as np
    import torch

    from nvfp4_w4a4_moe_permute_gb300 import inputs as IN
    from nvfp4_w4a4_moe_permute_gb300 import minite as M
    s = torch.cuda.current_stream(dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    hbm = peaks["hbm"]

    def bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    def stats(ts):
        return {"median": round(statistics.median(ts), 5), "p10": round(percentile(ts, 10), 5),
                "p90": round(percentile(ts, 90), 5)}

    out = {"peak_basis": f"FP4 {fp4_peak:.0f} TFLOP/s (measured bf16 burst x {FP4_OVER_BF16:g}),"
                         f" HBM {hbm:.0f} GB/s (measured copy)", "l2": "flushed before every launch"}
    # ---- dense GEMM
    dd = IN.make_dense_inputs()
    c = dd["cfg"]
    Mr, N, K = c["M"], c["N"], c["K"]
    a = bf16(dd["a"])
    w = bf16(dd["w"][None])
    qw = M.quantize(w, per_group=True)
    qa = M.quantize(a)
    torch.cuda.synchronize(dev)
    off = torch.tensor([0, Mr], dtype=torch.int32, device=dev)
    sfo = torch.tensor([0, (Mr + 127) // 128 * 128], dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    flops = 2.0 * Mr * N * K
    dense = {"shape": f"M={Mr} N={N} K={K}, E=1"}
    ta = time_launches(lambda: M.quantize(a, stream=s), s, flush=flush)
    qbytes = Mr * K * 2 + Mr * K / 2 + Mr * K / 16 + Mr * 4
    dense["quantize_a"] = dict(stats(ta), gbs=round(qbytes / (statistics.median(ta) / 1e3) / 1e9, 1))
    for name, dt in (("bf16_out", torch.bfloat16), ("fp32_out", torch.float32)):
        o = torch.empty((Mr, N), dtype=dt, device=dev)
        tg = time_launches(lambda: M.minite_grouped_gemm_nvfp4(
            qa["codes"], qa["sf"], qa["g"], qw["codes"], qw["sf"], qw["g"], off, sfo, o, st, s),
            s, flush=flush)
        med = statistics.median(tg)
        obytes = Mr * N * (2 if dt == torch.bfloat16 else 4)
        byts = Mr * K / 2 + Mr * K / 16 + N * K / 2 + N * K / 16 + obytes
        dense[name] = dict(stats(tg), tflops=round(flops / (med / 1e3) / 1e12, 1),
                           frac_fp4_peak=round(flops / (med / 1e3) / 1e12 / fp4_peak, 4),
                           attainable_tflops=round(min(fp4_peak, flops / byts * hbm / 1e3), 1))
    assert int(st.item()) == 0
    out["dense_gemm"] = dense
    del a, w, qw, qa, dd
    # ---- gate_up layer and MLP forward (one seeded batch)
    d = IN.make_moe_inputs("mlp")
    c = d["cfg"]
    T, H, E, k, I = c["T"], c["H"], c["E"], c["k"], c["I"]
    wgu = M.quantize(bf16(d["w_gate_up"]), per_group=True)
    wd = M.quantize(bf16(d["w_down"]), per_group=True)
    x, ids, tw = bf16(d["x"]), torch.from_numpy(d["topk_ids"]).to(dev), torch.from_numpy(d["topk_w"]).to(dev)
    mlp = M.MoEMLP(T, H, I, E, k, dev)
    mlp.forward(x, ids, tw, wgu, wd, s)
    torch.cuda.synchronize(dev)
    assert int(mlp.status.item()) == 0
    Mu = int(mlp.offsets[-1].item())
    tp = time_launches(lambda: mlp.permute_quant(x, ids, tw, s), s, flush=flush)
    pbytes = T * H * 2 + T * k * 8 + Mu * (H / 2 + H / 16 + 4 + 12)
    tgu = time_launches(lambda: M.minite_grouped_gemm_nvfp4(
        mlp.a_codes, mlp.a_sf, mlp.a_g, wgu["codes"], wgu["sf"], wgu["g"], mlp.offsets,
        mlp.sf_offsets, mlp.gate_up, mlp.status, s), s, flush=flush)
    gfl = 2.0 * Mu * 2 * I * H
    gbytes = Mu * H / 2 + int(mlp.sf_offsets[-1].item()) * H / 16 + E * 2 * I * H * (1 / 2 + 1 / 16) \
        + Mu * 2 * I * 2
    gmed = statistics.median(tgu)
    out["gate_up_layer"] = {
        "workload": workload_name("gate_up", c),
        "permute_quant": dict(stats(tp), gbs=round(pbytes / (statistics.median(tp) / 1e3) / 1e9, 1),
                              frac_hbm=round(pbytes / (statistics.median(tp) / 1e3) / 1e9 / hbm, 3)),
        "gemm_gate_up": dict(stats(tgu), tflops=round(gfl / (gmed / 1e3) / 1e12, 1),
                             frac_fp4_peak=round(gfl / (gmed / 1e3) / 1e12 / fp4_peak, 4),
                             attainable_tflops=round(min(fp4_peak, gfl / gbytes * hbm / 1e3), 1),
                             hbm_gbs=round(gbytes / (gmed / 1e3) / 1e9, 1))}
    tf = time_launches(lambda: mlp.forward(x, ids, tw, wgu, wd, s), s, flush=flush)
    fmed = statistics.median(tf)
    out["mlp_forward"] = {"workload": workload_name("mlp", c), **stats(tf),
                          "tokens_per_s": round(T / (fmed / 1e3)),
                          "launches": 5 + 1 + 1 + 1 + 1}
    if mlp.fused_ok:
        # the gate_up GEMM + SwiGLU as one fused launch against the two launches
        tu = time_launches(lambda: mlp.gate_up_swiglu(wgu, s, fused=False), s, flush=flush)
        tfu = time_launches(lambda: mlp.gate_up_swiglu(wgu, s, fused=True), s, flush=flush)
        out["mlp_forward"]["gate_up_swiglu"] = {"fused_ms": stats(tfu),
                                                "gemm_then_swiglu_ms": stats(tu)}
    assert int(mlp.status.item()) == 0
    return out


def run_gpu(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    from nvfp4_w4a4_moe_permute_gb300 import build as B
    from nvfp4_w4a4_moe_permute_gb300 import inputs as IN

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    B.build()
    from nvfp4_w4a4_moe_permute_gb300 import minite as M
    M.minite_set_gemm_variant(args.gemm_variant)
    d = IN.make_moe_inputs(args.workload, seed=rank)
    step = Step(d, dev)
    stream = torch.cuda.current_stream(dev)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(args.warmup):
        step.run(stream)
    barrier()
    assert int(step.status.item()) == 0, f"device status {int(step.status.item())}"

    nst = len(Step.STAGES)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nst + 1)] for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(args.steps):
        step.run(stream, ev[i])
    t1.record(stream)
    barrier()
    ms_eager = t0.elapsed_time(t1)
    # the same step captured once as a CUDA graph and replayed: no launch gaps
    ms_graph = None
    step_ms_list = [ev[i][0].elapsed_time(ev[i][-1]) for i in range(args.steps)]
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        with torch.cuda.graph(graph, stream=cap):
            step.run(torch.cuda.current_stream(dev))
        stream.wait_stream(cap)
        for _ in range(args.warmup):
            graph.replay()
        barrier()
        gev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
        gev[0].record(stream)
        for i in range(args.steps):
            graph.replay()
            gev[i + 1].record(stream)
        barrier()
        ms_graph = gev[0].elapsed_time(gev[-1])
        step_ms_list = [gev[i].elapsed_time(gev[i + 1]) for i in range(args.steps)]
        assert int(step.status.item()) == 0, f"device status {int(step.status.item())}"
    clk = clocks.stop()
    ms = ms_graph if ms_graph is not None else ms_eager
    ms, ms_eager = max_over_ranks([ms, ms_eager], dev)
    ms_per_step = ms / args.steps
    stage_ms = {s: statistics.mean(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(args.steps))
                for j, s in enumerate(Step.STAGES)}

    # the rest of the NVFP4 backward, eager, after the forward step's buffers
    # hold one step's results
    backward = None
    if not args.no_backward:
        step.init_backward()
        for _ in range(args.warmup):
            step.run_backward(stream)
        barrier()
        nb = len(Step.BWD_STAGES)
        bev = [[torch.cuda.Event(enable_timing=True) for _ in range(nb + 1)]
               for _ in range(args.steps)]
        for i in range(args.steps):
            step.run_backward(stream, bev[i])
        barrier()
        assert int(step.status.item()) == 0, f"device status {int(step.status.item())}"
        bst = {s: statistics.mean(bev[i][j].elapsed_time(bev[i][j + 1])
                                  for i in range(args.steps))
               for j, s in enumerate(Step.BWD_STAGES)}
        bab = step.backward_algorithmic_bytes()
        Mu = int(step.mlp.offsets[-1].item())
        dg_fl = 2.0 * Mu * 2 * step.I * step.H
        backward = {
            "stages": "W_gate_up dgrad copy (along N, the forward's global scales) + forward SwiGLU"
                      " keeping BF16 h + SwiGLU backward with per-row requant keeping BF16 dGU"
                      " + gate_up dgrad GEMM (K=2I, N=H) + combine of dX + token-axis NVFP4"
                      " operands (dY, h, dGU, x) + weight-gradient GEMMs of both projections",
            "ms": round(sum(bst.values()), 4),
            "stages_ms": {k_: round(v, 4) for k_, v in bst.items()},
            "stages_hbm_gbs": {k_: round(bab[k_] / (bst[k_] / 1e3) / 1e9, 1) for k_ in bab},
            "gemm_dgrad_gate_up_tflops": dg_fl / (bst["gemm_dgrad_gate_up"] / 1e3) / 1e12,
            "gemm_wgrad_down_tflops": 2.0 * Mu * step.H * step.I / (bst["gemm_wgrad_down"] / 1e3) / 1e12,
            "gemm_wgrad_gate_up_tflops": 2.0 * Mu * 2 * step.I * step.H
                                         / (bst["gemm_wgrad_gate_up"] / 1e3) / 1e12,
            "gpu_launches": Step.BWD_LAUNCHES * args.steps,
        }

    # end to end: every step copies its inputs (the token batch x, the routing
    # ids and weights, the incoming gradient dY) in from pinned host memory
    # and its result y out to pinned host memory; the BF16 weights are model
    # state that stays on the device between steps (an optimizer updates them
    # there), so they are not copied. Inputs and y are double-buffered on the
    # device, so the copies of step i+1 (copy stream) and the read-back of
    # step i (a second copy stream) overlap the compute of step i; each step
    # waits for its inputs where it first reads them (x, ids and w at the
    # permutation, dY at the combine backward), after the weight quantization.
    e2e = None
    if not args.no_e2e:
        names = ("x", "ids", "w", "dy")
        host = {n: getattr(step, n).cpu().pin_memory() for n in names}
        bufs = [{n: getattr(step, n) for n in names},
                {n: torch.empty_like(getattr(step, n)) for n in names}]
        ys = [step.mlp.y, torch.empty_like(step.mlp.y)]
        y_host = torch.empty(step.mlp.y.shape, dtype=step.mlp.y.dtype).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = y_host.numel() * y_host.element_size()
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in_x = [torch.cuda.Event() for _ in range(2)]  # x, ids, w of buffer b copied in
        ev_in_dy = [torch.cuda.Event() for _ in range(2)]  # dy of buffer b copied in
        ev_done = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]
        ev_y = [torch.cuda.Event() for _ in range(2)]  # y of buffer b complete

        def copy_in(b):
            with torch.cuda.stream(s_in):
                for n in ("x", "ids", "w"):
                    bufs[b][n].copy_(host[n], non_blocking=True)
                ev_in_x[b].record(s_in)
                bufs[b]["dy"].copy_(host["dy"], non_blocking=True)
                ev_in_dy[b].record(s_in)

        def e2e_run(n_steps):
            copy_in(0)
            for i in range(n_steps):
                cur, nxt = i % 2, (i + 1) % 2
                if i + 1 < n_steps:
                    if i > 0:
                        s_in.wait_event(ev_done[nxt])  # step i-1 is done with buffer nxt
                    copy_in(nxt)
                if i >= 2:
                    stream.wait_event(ev_out[cur])  # y of step i-2 has been read back
                step.bind(bufs[cur], ys[cur])
                # the step waits for its inputs where it first reads them
                step.run(stream, ready={"x": ev_in_x[cur], "dy": ev_in_dy[cur]},
                         y_done=ev_y[cur])
                ev_done[cur].record(stream)
                s_out.wait_event(ev_y[cur])
                with torch.cuda.stream(s_out):
                    y_host.copy_(ys[cur], non_blocking=True)
                    ev_out[cur].record(s_out)
            stream.wait_stream(s_out)

        e2e_run(max(1, args.warmup))
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        s_in.wait_stream(stream)
        e2e_run(args.steps)
        e1.record(stream)
        barrier()
        step.bind(bufs[0], ys[0])
        ems = max_over_ranks([e0.elapsed_time(e1)], dev)[0]
        e2e = {"value": step.T * world / (ems / args.steps / 1e3), "unit": "tokens/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": ems / args.steps}

    # the gate_up GEMM with the SwiGLU and requantization fused into its
    # epilogue, against the step's two launches, on the step's own buffers
    fused = None
    if rank == 0 and step.mlp.fused_ok and not args.no_fused:
        fused = fused_gate_up_swiglu(step, stream, dev)

    fl = step.flops()
    peaks = measured_peaks()
    # each GEMM launch is timed alone (CUDA events around it), so the burst
    # BF16 figure is the basis; the sustained one is reported beside it
    fp4_peak = peaks["bf16"] * FP4_OVER_BF16
    fp4_peak_sus = peaks["bf16_sus"] * FP4_OVER_BF16
    per_cfg = None
    if not args.no_per_config and rank == 0:
        per_cfg = per_config(dev, fp4_peak, peaks)
    gemm_s = stage_ms["gemm_gate_up"] / 1e3
    achieved = fl["gemm_gate_up"] / gemm_s / 1e12
    # the same launch against min(FP4 peak, arithmetic intensity x HBM bandwidth)
    gemm_bytes = step.gemm_gate_up_bytes()
    ai = fl["gemm_gate_up"] / gemm_bytes
    attainable = min(fp4_peak, ai * peaks["hbm"] / 1e3)
    traffic = None
    tp = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tp):
        traffic = json.load(open(tp)).get("gemm_gate_up_bytes_per_launch")
    ab = step.algorithmic_bytes()
    hbm = {s: ab[s] / (stage_ms[s] / 1e3) / 1e9 for s in ab}
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    out = {
        "metric": METRIC,
        "value": step.T * world / (ms_per_step / 1e3),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "ms_per_step_eager": ms_eager / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "nvfp4(e2m1+e4m3)xnvfp4->fp32 acc; bf16 io",
        "data": "synthetic (seeded numpy; Qwen3-30B-A3B shapes, random weights)",
        "config": {"workload": workload_name(args.workload, d["cfg"]),
                   "step": "wq(gate_up along K; down along K and along N in one pass) + permute+quant"
                           " + gate_up GEMM + SwiGLU+quant + down GEMM + combine + combine backward"
                           " with dY quant (forward routing) + dgrad GEMM",
                   "l2": "inputs larger than L2 (each step streams ~5 GB)",
                   "launch": "eager" if args.no_graph else "CUDA graph of the step, replayed",
                   "parallelism": f"replicas{world}"},
        "step_ms": {"median": round(statistics.median(step_ms_list), 4),
                    "p10": round(percentile(step_ms_list, 10), 4),
                    "p90": round(percentile(step_ms_list, 90), 4),
                    "of": "graph replays" if ms_graph is not None else "eager steps"},
        "gemm_gate_up_tflops": achieved,
        "gemm_gate_up_frac_fp4_peak": achieved / fp4_peak,
        "stages_ms": {s: round(v, 4) for s, v in stage_ms.items()},
        "stages_hbm_gbs": {s: round(v, 1) for s, v in hbm.items()},
        # each stage against its own bound: the measured HBM copy rate for the
        # bandwidth stages, the FP4 burst basis for the GEMMs
        "stages_frac_of_peak": dict(
            {s: round(v / peaks["hbm"], 3) for s, v in hbm.items()},
            **{g: round(fl[g] / (stage_ms[g] / 1e3) / 1e12 / fp4_peak, 3)
               for g in ("gemm_gate_up", "gemm_down", "gemm_dgrad")}),
        "gemms_tflops": {g: round(fl[g] / (stage_ms[g] / 1e3) / 1e12, 1)
                         for g in ("gemm_gate_up", "gemm_down", "gemm_dgrad")},
        "roofline": {"kernel": f"{GEMM_KERNELS.get(args.gemm_variant or 6)} (gate_up)",
                     "bound": "tensor",
                     "achieved": achieved, "peak": fp4_peak, "unit": "TFLOP/s",
                     "frac": achieved / fp4_peak, "traffic": traffic,
                     "peak_source": f"{peaks['source']} bf16 burst x {FP4_OVER_BF16:g} (nominal"
                                    f" dense FP4/BF16); the launch is timed alone",
                     "frac_of_sustained_basis": achieved / fp4_peak_sus,
                     "algorithmic_bytes": gemm_bytes, "flop_per_byte": ai,
                     "attainable": attainable, "frac_of_attainable": achieved / attainable,
                     "achieved_hbm_gbs": gemm_bytes / gemm_s / 1e9},
        "clocks": clk,
        "gpu_launches": Step.LAUNCHES * args.steps,
        "backward": backward,
        "per_config": per_cfg,
        "fused_gate_up_swiglu": fused,
        "e2e": e2e,
        "cpu_baseline": None,
    }
    if not args.no_cpu_baseline and world == 1 or (not args.no_cpu_baseline and rank == 0):
        out["cpu_baseline"] = cpu_baseline_subprocess(args)
    print(json.dumps(out), flush=True)
    if world > 1:
        dist.destroy_process_group()


# ----------------------------------------------------------------------------- CPU oracle
#
# The oracle (plain NumPy) timed on the host's cores. Work is sharded by
# expert over spawned processes (never forked from a CUDA process), each
# driving the unchanged oracle functions for its experts: the quantization of
# their weights and their permuted rows through the gate_up GEMM
# (float32-accumulate variant), the weighted SwiGLU with requantization, the
# down GEMM and, for the benchmarked step, the dgrad GEMM. The parent runs
# the permutations and the combine. Arrays travel through .npy files in
# shared memory. The oracle runs on a whole batch of the stated size; nothing
# is scaled.

def cpu_info():
    """(logical cores, CPU model string) of this host."""
    import platform
    model = platform.machine()
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                key = ln.split(":", 1)[0].strip().lower()
                if key in ("model name", "cpu part", "hardware"):
                    model = ln.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    return os.cpu_count() or 1, model


_ORC = {}


def _orc_init(dirpath):
    from oracle import nvfp4_moe_oracle as O
    _ORC["O"] = O
    _ORC["dir"] = dirpath


def _mm(name, mode="r"):
    import numpy as np
    return np.load(os.path.join(_ORC["dir"], name + ".npy"), mmap_mode=mode)


def _orc_quantize_weights(experts, dgrad):
    """Weights of `experts`: W_gate_up and W_down along K (forward), and W_down
    along N with the same global scales (dgrad copy) when `dgrad`."""
    O = _ORC["O"]
    wgu, wd = _mm("w_gate_up"), _mm("w_down")
    out = {n: _mm(n, "r+") for n in ("gu_c", "gu_sf", "gu_g", "d_c", "d_sf", "d_g")}
    if dgrad:
        out.update({n: _mm(n, "r+") for n in ("dT_c", "dT_sf")})
    for e in experts:
        c, sf, _, g = O.quantize_weights(wgu[e:e + 1])
        out["gu_c"][e], out["gu_sf"][e], out["gu_g"][e] = c[0], sf[0], g[0]
        c, sf, _, g = O.quantize_weights(wd[e:e + 1])
        out["d_c"][e], out["d_sf"][e], out["d_g"][e] = c[0], sf[0], g[0]
        if dgrad:
            c, sf, _, _ = O.quantize_weights(wd[e:e + 1], along_rows=True, g_in=g)
            out["dT_c"][e], out["dT_sf"][e] = c[0], sf[0]
    for m in out.values():
        m.flush()
    return len(experts)


def _orc_expert_rows(experts, dgrad):
    """The permuted rows of `experts` through gate_up GEMM -> BF16 -> weighted
    SwiGLU + requant -> down GEMM -> BF16 (and dY's rows through the dgrad
    GEMM when `dgrad`), each expert as a one-expert problem of the oracle."""
    import numpy as np
    O = _ORC["O"]
    off = _mm("offsets")
    a_c, a_sf, a_g, pw = _mm("a_c"), _mm("a_sf"), _mm("a_g"), _mm("perm_w")
    gu_c, gu_sf, gu_g = _mm("gu_c"), _mm("gu_sf"), _mm("gu_g")
    d_c, d_sf, d_g = _mm("d_c"), _mm("d_sf"), _mm("d_g")
    down = _mm("down", "r+")
    if dgrad:
        y_c, y_sf, y_g = _mm("dy_c"), _mm("dy_sf"), _mm("dy_g")
        dT_c, dT_sf = _mm("dT_c"), _mm("dT_sf")
        dh = _mm("dh", "r+")
    for e in experts:
        a, b = int(off[e]), int(off[e + 1])
        if a == b:
            continue
        o1 = np.array([0, b - a], dtype=np.int64)
        s1 = np.array([0, (b - a + 127) // 128 * 128], dtype=np.int64)
        gu = O.grouped_gemm_fp32_accumulate(a_c[a:b], a_sf[a:b], a_g[a:b], gu_c[e:e + 1],
                                            gu_sf[e:e + 1], gu_g[e:e + 1], o1)
        sw = O.swiglu_weighted_quant(O.f32_to_bf16(gu), pw[a:b], o1, s1)
        d = O.grouped_gemm_fp32_accumulate(sw["codes"], sw["sf"], sw["row_g"], d_c[e:e + 1],
                                           d_sf[e:e + 1], d_g[e:e + 1], o1)
        down[a:b] = O.f32_to_bf16(d)
        if dgrad:
            h = O.grouped_gemm_fp32_accumulate(y_c[a:b], y_sf[a:b], y_g[a:b], dT_c[e:e + 1],
                                               dT_sf[e:e + 1], d_g[e:e + 1], o1)
            dh[a:b] = O.f32_to_bf16(h)
    down.flush()
    if dgrad:
        dh.flush()
    return len(experts)


class OracleRunner:
    """The oracle on the host's cores for one MoE workload. `tokens` selects
    the batch (the first `tokens` tokens of the workload's seeded batch, with
    their routing); `dgrad` adds the combine backward's dY quantization and
    the dgrad GEMM; `weights_in_step` makes the weight quantization part of
    each timed step (else it runs once at set-up)."""

    def __init__(self, workload, tokens=None, dgrad=False, weights_in_step=False, procs=None):
        import multiprocessing as mp
        import tempfile

        import numpy as np

        from nvfp4_w4a4_moe_permute_gb300 import inputs as IN
        from oracle import nvfp4_moe_oracle as O
        self.O, self.np = O, np
        d = IN.make_moe_inputs(workload, seed=0)
        c = d["cfg"]
        self.cfg = c
        T, H, E, k, I = c["T"], c["H"], c["E"], c["k"], c["I"]
        self.tokens = T if tokens is None else min(int(tokens), T)
        self.E, self.dgrad, self.weights_in_step = E, dgrad, weights_in_step
        tok = np.arange(self.tokens)
        self.x, self.ids, self.w = d["x"][tok], d["topk_ids"][tok], d["topk_w"][tok]
        # the incoming gradient (workloads without one use x in its place)
        self.dy = d.get("dy", d["x"])[tok] if dgrad else None
        base = "/dev/shm" if os.path.isdir("/dev/shm") else None
        self.dir = tempfile.mkdtemp(prefix="minite_oracle_", dir=base)
        M = self.tokens * k

        def put(name, arr):
            np.save(os.path.join(self.dir, name + ".npy"), arr)

        def blank(name, shape, dtype):
            np.save(os.path.join(self.dir, name + ".npy"), np.zeros(shape, dtype=dtype))

        put("w_gate_up", d["w_gate_up"])
        put("w_down", d["w_down"])
        del d
        blank("gu_c", (E, 2 * I, H // 2), np.uint8)
        blank("gu_sf", (E, 2 * I, H // 16), np.uint8)
        blank("gu_g", (E,), np.float32)
        blank("d_c", (E, H, I // 2), np.uint8)
        blank("d_sf", (E, H, I // 16), np.uint8)
        blank("d_g", (E,), np.float32)
        if dgrad:
            blank("dT_c", (E, I, H // 2), np.uint8)
            blank("dT_sf", (E, I, H // 16), np.uint8)
        blank("down", (M, H), np.uint16)
        if dgrad:
            blank("dh", (M, I), np.uint16)
        self.procs = max(1, min(procs or os.cpu_count() or 1, 64))
        # experts spread over processes by their row counts plus a fixed cost
        # per expert (its weights are dequantized once per GEMM)
        rows = np.bincount(self.ids.ravel(), minlength=E)
        cost = rows / max(1.0, rows.mean()) + 1.0
        loads = [0.0] * self.procs
        self.shards = [[] for _ in range(self.procs)]
        for e in np.argsort(-cost, kind="stable"):
            i = int(np.argmin(loads))
            self.shards[i].append(int(e))
            loads[i] += float(cost[e])
        self.shards = [s for s in self.shards if s]
        ctx = mp.get_context("spawn")
        self.pool = ctx.Pool(len(self.shards), initializer=_orc_init, initargs=(self.dir,))
        if not weights_in_step:
            self.pool.starmap(_orc_quantize_weights, [(s, dgrad) for s in self.shards])

    def step(self):
        """One timed pass; returns seconds."""
        O, np = self.O, self.np
        t0 = time.perf_counter()
        if self.weights_in_step:
            self.pool.starmap(_orc_quantize_weights, [(s, self.dgrad) for s in self.shards])
        pq = O.moe_permute_quant(self.x, self.ids, self.w, self.E)
        for name, arr in (("a_c", pq["codes"]), ("a_sf", pq["sf"]), ("a_g", pq["row_g"]),
                          ("perm_w", pq["perm_w"]),
                          ("offsets", np.asarray(pq["expert_offsets"], dtype=np.int64))):
            np.save(os.path.join(self.dir, name + ".npy"), arr)
        if self.dgrad:
            pd = O.moe_permute_quant(self.dy, self.ids, None, self.E)
            for name, arr in (("dy_c", pd["codes"]), ("dy_sf", pd["sf"]), ("dy_g", pd["row_g"])):
                np.save(os.path.join(self.dir, name + ".npy"), arr)
        self.pool.starmap(_orc_expert_rows, [(s, self.dgrad) for s in self.shards])
        down = np.load(os.path.join(self.dir, "down.npy"), mmap_mode="r")
        O.moe_combine(np.asarray(down[:int(pq["expert_offsets"][-1])]), pq["dest_row"])
        return time.perf_counter() - t0

    def close(self):
        import shutil
        self.pool.terminate()
        self.pool.join()
        shutil.rmtree(self.dir, ignore_errors=True)


def cpu_baseline_run(args):
    """The oracle's whole 4096-token expert-MLP forward (Qwen3-30B-A3B layer:
    permutation + quantization, gate_up GEMM, weighted SwiGLU + requant,
    down GEMM, combine) on all host cores; one warm-up pass and
    `--cpu-baseline-reps` timed passes. Prints one JSON object."""
    cores, model = cpu_info()
    r = OracleRunner("mlp", procs=cores)
    try:
        r.step()
        times = [r.step() for _ in range(max(1, args.cpu_baseline_reps))]
    finally:
        r.close()
    s = statistics.median(times)
    print(json.dumps({"cpu_baseline": {
        "value": r.tokens / s, "unit": "tokens/s", "cores": len(r.shards), "cpu_model": model,
        "kind": "oracle", "extrapolated": False, "seconds": round(s, 3),
        "workload": workload_name("mlp", r.cfg),
        "sample": f"the whole {r.tokens}-token expert-MLP forward (not scaled), weights quantized"
                  f" beforehand; GEMMs in the oracle's float32-accumulate variant; expert shards"
                  f" over {len(r.shards)} spawned processes; median of {len(times)} passes"}}),
          flush=True)


def cpu_baseline_subprocess(args):
    """Run cpu_baseline_run in a fresh process with no GPU visible (its process
    pool is spawned there, never forked from this CUDA process)."""
    env = dict(os.environ)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[v] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    cmd = [sys.executable, os.path.abspath(__file__), "--cpu-baseline-only",
           "--cpu-baseline-reps", str(args.cpu_baseline_reps)]
    try:
        r = subprocess.run(cmd, env=env, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True,
                           timeout=1200)
        line = [ln for ln in r.stdout.splitlines() if ln.startswith("{")][-1]
        return json.loads(line)["cpu_baseline"]
    except Exception as exc:  # noqa: BLE001
        return {"value": None, "unit": "tokens/s", "error": repr(exc)[:200]}


def run_reference(args):
    """The reference arm: the oracle timed on the host's cores on the
    benchmark's workload and step (weight quantization of every expert, the
    permutation, both GEMMs, SwiGLU, combine, dY quantization and the dgrad
    GEMM), on a batch of the first `--cpu-sample-tokens` tokens of the seeded
    batch (with their routing) so that a step takes seconds, not minutes.
    Every step is measured; nothing is scaled."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[v] = "1"
    cores, model = cpu_info()
    r = OracleRunner(args.workload, tokens=args.cpu_sample_tokens, dgrad=True,
                     weights_in_step=True, procs=cores)
    try:
        for _ in range(args.warmup):
            r.step()
        times = [r.step() for _ in range(args.steps)]
    finally:
        r.close()
    ms = statistics.mean(times) * 1e3
    value = r.tokens / (ms / 1e3)
    T = r.cfg["T"]
    sample = (f"the benchmark's step on the first {r.tokens} of the workload's {T} tokens (their"
              f" routing; every expert's weights quantized each step, as in the GPU step), not"
              f" scaled; expert shards over {len(r.shards)} spawned processes")
    out = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 0, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None,
           "dtype": "fp32 quantization, float32-accumulate GEMMs (numpy)",
           "data": "synthetic (seeded numpy)", "impl": "reference",
           "config": {"workload": workload_name(args.workload, r.cfg),
                      "batch_tokens": r.tokens, "parallelism": f"host cpu, {len(r.shards)} processes"},
           "step_seconds": {"median": round(statistics.median(times), 3),
                            "min": round(min(times), 3), "max": round(max(times), 3)},
           "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": len(r.shards),
                            "cpu_model": model, "kind": "oracle", "extrapolated": False,
                            "seconds": round(ms / 1e3, 3), "sample": sample},
           "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main():
    args = parse()
    if args.cpu_baseline_only:
        cpu_baseline_run(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
