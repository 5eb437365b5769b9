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
    ap.add_argument("--cpu-sample-tokens", type=int, default=16)
    ap.add_argument("--cpu-sample-experts", type=int, default=2)
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
    # quantization 2 + 2, permutation 5, GEMM 1, SwiGLU 1, GEMM 1, combine 1,
    # combine backward with dY quantization 2, GEMM 1
    LAUNCHES = 2 + 2 + 5 + 1 + 1 + 1 + 1 + 2 + 1

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
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        g1.record(stream)
        barrier()
        ms_graph = g0.elapsed_time(g1)
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

    fl = step.flops()
    peaks = measured_peaks()
    fp4_peak = peaks["bf16_sus"] * FP4_OVER_BF16
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
        "gemm_gate_up_tflops": achieved,
        "gemm_gate_up_frac_fp4_peak": achieved / fp4_peak,
        "stages_ms": {s: round(v, 4) for s, v in stage_ms.items()},
        "stages_hbm_gbs": {s: round(v, 1) for s, v in hbm.items()},
        "roofline": {"kernel": "grouped_gemm_dc_kernel (gate_up)", "bound": "tensor",
                     "achieved": achieved, "peak": fp4_peak, "unit": "TFLOP/s",
                     "frac": achieved / fp4_peak, "traffic": traffic,
                     "peak_source": f"{peaks['source']} bf16 sustained x {FP4_OVER_BF16:g} (nominal FP4/BF16)",
                     "algorithmic_bytes": gemm_bytes, "flop_per_byte": ai,
                     "attainable": attainable, "frac_of_attainable": achieved / attainable,
                     "achieved_hbm_gbs": gemm_bytes / gemm_s / 1e9},
        "clocks": clk,
        "gpu_launches": Step.LAUNCHES * args.steps,
        "backward": backward,
        "e2e": e2e,
        "cpu_baseline": None,
    }
    if not args.no_cpu_baseline and world == 1 or (not args.no_cpu_baseline and rank == 0):
        out["cpu_baseline"] = cpu_baseline_subprocess(args)
    print(json.dumps(out), flush=True)
    if world > 1:
        dist.destroy_process_group()


# ----------------------------------------------------------------------------- CPU oracle

class CpuSample:
    """The oracle on a bounded sample of the step, scaled to one full step:
    the per-token chain (forward + dY permute/quant + dgrad GEMM) on n_tok
    tokens scaled by T/n_tok, plus the weight quantizations (both
    orientations) of n_exp experts scaled by E/n_exp."""

    def __init__(self, workload: str, n_tok: int, n_exp: int):
        import numpy as np

        from nvfp4_w4a4_moe_permute_gb300 import inputs as IN
        from oracle import nvfp4_moe_oracle as O
        self.O = O
        d = IN.make_moe_inputs(workload, seed=0)
        c = d["cfg"]
        self.T, self.E = c["T"], c["E"]
        self.n_tok, self.n_exp = n_tok, n_exp
        self.d = d
        self.tok = np.arange(n_tok)
        used = np.unique(d["topk_ids"][self.tok])
        # untimed: quantized weights of the experts the sampled tokens reach
        self.wgu = self._partial(d["w_gate_up"], used)
        self.wd = self._partial(d["w_down"], used)
        self.wdT = self._partial(d["w_down"], used, along_rows=True, g_in=self.wd[3])

    def _partial(self, w, used, along_rows=False, g_in=None):
        import numpy as np
        O = self.O
        q = O.quantize_weights(w[used], along_rows=along_rows,
                               g_in=None if g_in is None else g_in[used])
        full = []
        for a in q:
            z = np.zeros((self.E,) + a.shape[1:], dtype=a.dtype)
            z[used] = a
            full.append(z)
        return tuple(full)

    def run(self):
        O, d, tok, E = self.O, self.d, self.tok, self.E
        t0 = time.perf_counter()
        O.quantize_weights(d["w_gate_up"][:self.n_exp])
        wd = O.quantize_weights(d["w_down"][:self.n_exp])
        O.quantize_weights(d["w_down"][:self.n_exp], along_rows=True, g_in=wd[3])
        t_w = time.perf_counter() - t0
        t1 = time.perf_counter()
        O.moe_mlp_forward(d["x"][tok], d["topk_ids"][tok], d["topk_w"][tok], E, self.wgu, self.wd)
        dy = d.get("dy", d["x"])
        pq = O.moe_permute_quant(dy[tok], d["topk_ids"][tok], None, E)
        dh, _ = O.grouped_gemm_exact(pq["codes"], pq["sf"], pq["row_g"], self.wdT[0], self.wdT[1],
                                     self.wdT[3], pq["expert_offsets"])
        O.f64_to_bf16(dh)
        t_chain = time.perf_counter() - t1
        step_s = t_w * E / self.n_exp + t_chain * self.T / self.n_tok
        return step_s, dict(weights_s=round(t_w, 3), chain_s=round(t_chain, 3))


def cpu_baseline_subprocess(args):
    """Run the oracle in a fresh single-threaded process (spawned, never forked
    from this CUDA process) and return its cpu_baseline object."""
    env = dict(os.environ)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[v] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    cmd = [sys.executable, os.path.abspath(__file__), "--impl", "reference", "--steps", "1",
           "--warmup", "0", "--workload", args.workload, "--cpu-sample-tokens",
           str(args.cpu_sample_tokens), "--cpu-sample-experts", str(args.cpu_sample_experts)]
    try:
        r = subprocess.run(cmd, env=env, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True,
                           timeout=900)
        line = [ln for ln in r.stdout.splitlines() if ln.startswith("{")][-1]
        return json.loads(line)["cpu_baseline"]
    except Exception as exc:  # noqa: BLE001
        return {"value": None, "unit": "tokens/s", "error": repr(exc)[:200]}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ.setdefault(v, "1")
    smp = CpuSample(args.workload, args.cpu_sample_tokens, args.cpu_sample_experts)
    T = smp.T
    times = []
    parts = None
    for i in range(args.warmup + args.steps):
        step_s, parts = smp.run()
        if i >= args.warmup:
            times.append(step_s)
    ms = statistics.mean(times) * 1e3
    value = T / (ms / 1e3)
    threads = int(os.environ.get("OPENBLAS_NUM_THREADS", "1"))
    sample = (f"oracle chain (fwd + dY permute/quant + dgrad GEMM) on {args.cpu_sample_tokens} "
              f"tokens scaled x{T // args.cpu_sample_tokens}, plus weight quantization of "
              f"{args.cpu_sample_experts} experts scaled to all; last sample {parts}")
    out = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 0, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "fp32 quantization / fp64 GEMM (numpy)",
           "data": "synthetic (seeded numpy)", "impl": "reference",
           "config": {"workload": workload_name(args.workload, smp.d["cfg"]),
                      "parallelism": "host cpu"},
           "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads,
                            "kind": "oracle", "sample": sample},
           "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
