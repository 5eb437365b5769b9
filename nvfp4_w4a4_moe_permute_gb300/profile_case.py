"""Run one library entry point on a seeded synthetic case, a few times, for
profiling a single kernel (``ncu -k <kernel> ...``) at a size chosen on the
command line, without the memory of a whole layer step.

    python -m nvfp4_w4a4_moe_permute_gb300.profile_case quantize_tokens \\
        --rows 131072 --cols 1536 --experts 128
    python -m nvfp4_w4a4_moe_permute_gb300.profile_case quantize_tokens \\
        --rows 131072 --cols 2048 --experts 128 --gather 16384
    python -m nvfp4_w4a4_moe_permute_gb300.profile_case quantize_weights \\
        --experts 16 --rows 1536 --cols 2048 [--dual]
    python -m nvfp4_w4a4_moe_permute_gb300.profile_case permute_swiglu --tokens 16384
    python -m nvfp4_w4a4_moe_permute_gb300.profile_case gemm --tokens 8192 --gemm gate_up

Expert sizes follow a Zipf(1.5) draw over the experts (a skewed routing);
every call's device status is checked at the end.
"""
from __future__ import annotations

import argparse
import sys

import numpy as np
import torch

from . import build as _build


def _expert_offsets(rng, rows: int, experts: int, dev):
    w = rng.zipf(1.5, experts).astype(np.float64)
    cnt = np.floor(w / w.sum() * rows).astype(np.int64)
    cnt[0] += rows - cnt.sum()
    off = np.concatenate([[0], np.cumsum(cnt)]).astype(np.int32)
    return torch.tensor(off, device=dev)


def quantize_tokens(args, M, dev, status):
    """A weight-gradient operand: rows in place, or gathered from `--gather`
    source rows through a random row map."""
    rng = np.random.default_rng(args.seed)
    off = _expert_offsets(rng, args.rows, args.experts, dev)
    gen = torch.Generator(device=dev).manual_seed(args.seed)
    n_src = args.gather if args.gather > 0 else args.rows
    x = (torch.randn((n_src, args.cols), device=dev, generator=gen) * 0.1).to(torch.bfloat16)
    row_src = None
    if args.gather > 0:
        row_src = torch.randint(0, n_src, (args.rows,), device=dev, generator=gen,
                                dtype=torch.int32)
    q = M.quantize_tokens(x, off, args.experts, row_src=row_src, m_cap=args.rows)
    gathered = row_src is not None
    ws = torch.empty(max(4, M.minite_workspace_bytes(M.OP_QUANTIZE_TOKENS, args.experts,
                                                     n_src if gathered else 0)),
                     dtype=torch.uint8, device=dev)
    for _ in range(args.reps):
        M.minite_quantize_tokens_nvfp4(x, row_src, args.rows, args.experts, off, q["k_cap"],
                                       q["codes"], q["sf"], q["g"], q["kofs"], ws, status)


def quantize_weights(args, M, dev, status):
    """Per-expert weight quantization along cols, or both orientations."""
    gen = torch.Generator(device=dev).manual_seed(args.seed)
    w = (torch.randn((args.experts, args.rows, args.cols), device=dev, generator=gen) *
         0.02).to(torch.bfloat16)
    E, R, C = w.shape
    ws = torch.empty(M.minite_workspace_bytes(M.OP_QUANTIZE, E), dtype=torch.uint8, device=dev)
    ck = torch.empty((E, R, C // 2), dtype=torch.uint8, device=dev)
    sk = torch.empty((E, M.sf_bytes((R + 127) // 128 * 128, C)), dtype=torch.uint8, device=dev)
    g = torch.empty(E, dtype=torch.float32, device=dev)
    if args.dual:
        cn = torch.empty((E, C, R // 2), dtype=torch.uint8, device=dev)
        sn = torch.empty((E, M.sf_bytes((C + 127) // 128 * 128, R)), dtype=torch.uint8, device=dev)
    for _ in range(args.reps):
        if args.dual:
            M.minite_quantize_nvfp4_dual(w, ck, sk, cn, sn, g, ws, status)
        else:
            M.minite_quantize_nvfp4(w, M.SCALE_PER_GROUP, M.ALONG_COLS, ck, sk, g, None, ws,
                                    status)


def permute_swiglu(args, M, dev, status):
    """The permutation with fused quantization of x and the weighted SwiGLU
    with requantization, on the skewed layer's recipe at `--tokens` tokens
    (the SwiGLU's input is seeded N(0, 2) BF16 in place of the gate_up GEMM's
    output)."""
    from . import inputs as IN
    d = IN.make_moe_inputs("skewed", seed=args.seed, T=args.tokens, with_weights=False)
    c = d["cfg"]
    T, H, E, k, I = c["T"], c["H"], c["E"], c["k"], c["I"]

    def bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    x = bf16(d["x"])
    ids = torch.from_numpy(d["topk_ids"]).to(dev)
    w = torch.from_numpy(d["topk_w"]).to(dev)
    mlp = M.MoEMLP(T, H, I, E, k)
    gen = torch.Generator(device=dev).manual_seed(args.seed)
    mlp.gate_up.copy_((torch.randn(mlp.gate_up.shape, device=dev, generator=gen) * 2.0)
                      .to(torch.bfloat16))
    for _ in range(args.reps):
        mlp.permute_quant(x, ids, w)
        M.minite_swiglu_weighted_quant(mlp.gate_up, mlp.perm_w, E, mlp.offsets, mlp.sf_offsets,
                                       mlp.h_codes, mlp.h_sf, mlp.h_g, status)
    torch.cuda.synchronize(dev)
    if int(mlp.status.item()) != 0:
        status.fill_(int(mlp.status.item()))


def gemm(args, M, dev, status):
    """One grouped GEMM of the skewed layer's recipe at `--tokens` tokens
    (`--gemm` gate_up, gate_up_swiglu (the fused gate_up GEMM + SwiGLU +
    requantization), down or dgrad), its operands produced by the library
    (weight quantization, permutation, SwiGLU), with the automatic kernel or
    `--variant`. The GEMM is the last `--reps` launches."""
    from . import inputs as IN
    d = IN.make_moe_inputs("skewed", seed=args.seed, T=args.tokens)
    c = d["cfg"]
    T, H, E, k, I = c["T"], c["H"], c["E"], c["k"], c["I"]

    def bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    wgu = M.quantize(bf16(d["w_gate_up"]), per_group=True)
    wd_bf = bf16(d["w_down"])
    wd = M.quantize(wd_bf, per_group=True)
    wdT = M.quantize(wd_bf, per_group=True, along_rows=True, g_in=wd["g"])
    mlp = M.MoEMLP(T, H, I, E, k)
    mlp.status = status
    mlp.forward(bf16(d["x"]), torch.from_numpy(d["topk_ids"]).to(dev),
                torch.from_numpy(d["topk_w"]).to(dev), wgu, wd)
    dh = torch.empty((T * k, I), dtype=torch.bfloat16, device=dev)
    M.minite_set_gemm_variant(args.variant)
    for _ in range(args.reps):
        if args.gemm == "gate_up_swiglu":
            mlp.gate_up_swiglu(wgu, fused=True)
        elif args.gemm == "gate_up":
            M.minite_grouped_gemm_nvfp4(mlp.a_codes, mlp.a_sf, mlp.a_g, wgu["codes"], wgu["sf"],
                                        wgu["g"], mlp.offsets, mlp.sf_offsets, mlp.gate_up, status)
        elif args.gemm == "down":
            M.minite_grouped_gemm_nvfp4(mlp.h_codes, mlp.h_sf, mlp.h_g, wd["codes"], wd["sf"],
                                        wd["g"], mlp.offsets, mlp.sf_offsets, mlp.down, status)
        else:
            # the permuted x stands in for the permuted dY (same layout and routing)
            M.minite_grouped_gemm_nvfp4(mlp.a_codes, mlp.a_sf, mlp.a_g, wdT["codes"], wdT["sf"],
                                        wd["g"], mlp.offsets, mlp.sf_offsets, dh, status)
    M.minite_set_gemm_variant(0)


CASES = {"quantize_tokens": quantize_tokens, "quantize_weights": quantize_weights,
         "permute_swiglu": permute_swiglu, "gemm": gemm}


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("case", choices=sorted(CASES))
    ap.add_argument("--rows", type=int, default=131072)
    ap.add_argument("--cols", type=int, default=1536)
    ap.add_argument("--experts", type=int, default=128)
    ap.add_argument("--tokens", type=int, default=16384, help="permute_swiglu: tokens")
    ap.add_argument("--gather", type=int, default=0, help="source rows (0: rows in place)")
    ap.add_argument("--dual", action="store_true", help="weights: both orientations")
    ap.add_argument("--gemm", default="gate_up",
                    choices=["gate_up", "gate_up_swiglu", "down", "dgrad"])
    ap.add_argument("--variant", type=int, default=0, help="gemm: grouped-GEMM kernel (0 automatic)")
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--seed", type=int, default=0)
    args = ap.parse_args(argv)
    _build.build()
    from . import minite as M
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    CASES[args.case](args, M, dev, status)
    torch.cuda.synchronize(dev)
    st = int(status.item())
    print(f"{args.case}: {args.reps} calls, device status {st}")
    return 0 if st == 0 else 1


if __name__ == "__main__":
    sys.exit(main())
