"""Seeded synthetic inputs for the W4A4 MoE expert MLP.

This module is shared by the CUDA path's tests and benchmark and by the CPU
oracle's tests. It holds no arithmetic of the method itself: it only draws
random numbers, rounds them to BF16 storage, and turns router logits into
top-k routing (the router is not part of the expert MLP; its outputs are
inputs here).

Shapes follow the Qwen3-30B-A3B MoE layer named on the news.hamidun.com page
("miniTE accélère le RL en NVFP4 sur B300", section "Paramètres clés"):
hidden 2048, 128 experts, top-8, expert intermediate 768. Sequence length
4096 with micro-batch 1 follows the miniTE report summary, section
"Respect the timing boundaries".

Every array comes from ``np.random.default_rng(seed)``, drawn in the fixed
order logits, x, W_gate_up, W_down, dY; values are float32 rounded to BF16
by round-to-nearest-even. BF16 tensors are returned as ``uint16`` bit
patterns so that no library's BF16 conversion is involved.
"""
from __future__ import annotations

import numpy as np

# name -> shape parameters. T tokens, H hidden, E experts, k top-k,
# I expert intermediate size (gate_up projects H -> 2I, down projects I -> H).
CONFIGS = {
    # Tiny correctness case: 64 tokens, K=64, 4 experts, expert out N=2I=128, top-2.
    "tiny": dict(T=64, H=64, E=4, k=2, I=64),
    # Single dense NVFP4 GEMM M=4096 N=1536 K=2048 with 1% outlier channels x20.
    "dense": dict(M=4096, N=1536, K=2048, n_outlier=20, outlier_gain=20.0),
    # Qwen3-30B-A3B gate_up layer: 4096 tokens, hidden 2048, 128 experts, top-8, N=1536.
    "gate_up": dict(T=4096, H=2048, E=128, k=8, I=768),
    # Full Qwen3-30B-A3B expert MLP forward, 4096 tokens.
    "mlp": dict(T=4096, H=2048, E=128, k=8, I=768),
    # Skewed-load MLP: 32768 tokens, Zipf(1.2)-shaped expert load, 8 empty experts,
    # plus the dgrad-layout weight requant and one dgrad grouped GEMM.
    "skewed": dict(T=32768, H=2048, E=128, k=8, I=768, zipf_s=1.2, n_empty=8),
}

WEIGHT_STD = 0.02
# Scale on -s*ln(rank) in the skewed router bias, chosen so that the
# resulting per-expert load, fitted on log-log axes over the non-saturated
# experts, has slope close to -1.2 (the fit is reported by ``zipf_fit``).
ZIPF_BIAS_GAIN = 0.55


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to BF16 (nearest, ties to even) and return the bits."""
    b = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    out = rounded.astype(np.uint16)
    out[np.isnan(a)] = 0x7FC0
    return out


def bf16_bits_to_f32(u: np.ndarray) -> np.ndarray:
    return (np.asarray(u, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def topk_softmax_routing(logits: np.ndarray, k: int):
    """Top-k of softmax(logits); lower expert id wins ties; weights renormalised to sum 1."""
    z = logits.astype(np.float64)
    z = z - z.max(axis=1, keepdims=True)
    p = np.exp(z)
    p /= p.sum(axis=1, keepdims=True)
    order = np.argsort(-p, axis=1, kind="stable")[:, :k]
    w = np.take_along_axis(p, order, axis=1)
    w = w / w.sum(axis=1, keepdims=True)
    return order.astype(np.int32), w.astype(np.float32)


def skewed_bias(rng: np.random.Generator, E: int, s: float, n_empty: int) -> np.ndarray:
    """Router bias b_e = -gain*s*ln(rank_e) over a random rank permutation;
    the n_empty lowest-ranked experts get -1e4 so that no token reaches them."""
    rank = rng.permutation(E) + 1  # rank[e] in 1..E
    b = -ZIPF_BIAS_GAIN * s * np.log(rank.astype(np.float64))
    b[rank > E - n_empty] = -1.0e4
    return b.astype(np.float32)


def zipf_fit(topk_ids: np.ndarray, E: int):
    """Least-squares slope of log(load) vs log(rank) over experts that are
    neither empty nor saturated (load < number of tokens)."""
    counts = np.bincount(topk_ids.ravel(), minlength=E).astype(np.float64)
    T = topk_ids.shape[0]
    srt = np.sort(counts)[::-1]
    r = np.arange(1, E + 1, dtype=np.float64)
    keep = (srt > 0) & (srt < T)
    if keep.sum() < 2:
        return float("nan"), counts
    slope = np.polyfit(np.log(r[keep]), np.log(srt[keep]), 1)[0]
    return float(slope), counts


def _normal_bf16(rng, shape, std=1.0):
    a = rng.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return f32_to_bf16_bits(a)


def make_moe_inputs(name: str, seed: int = 0, T: int | None = None, with_weights: bool = True):
    """Inputs of a MoE config: x, routing, expert weights (and dY for 'skewed').

    ``T`` overrides the token count (same recipe, fewer or more tokens).
    Returns a dict of numpy arrays: x [T,H] bf16 bits, topk_ids [T,k] int32,
    topk_w [T,k] float32, w_gate_up [E,2I,H] bf16 bits (rows 0..I-1 are the
    gate projection, rows I..2I-1 the up projection), w_down [E,H,I] bf16 bits,
    dy [T,H] bf16 bits ('skewed' only).
    """
    c = dict(CONFIGS[name])
    if T is not None:
        c["T"] = T
    T, H, E, k, I = c["T"], c["H"], c["E"], c["k"], c["I"]
    rng = np.random.default_rng(seed)
    logits = rng.standard_normal((T, E), dtype=np.float32)
    if "zipf_s" in c:
        logits = logits + skewed_bias(rng, E, c["zipf_s"], c["n_empty"])[None, :]
    topk_ids, topk_w = topk_softmax_routing(logits, k)
    out = dict(cfg=c, topk_ids=topk_ids, topk_w=topk_w)
    out["x"] = _normal_bf16(rng, (T, H))
    if with_weights:
        out["w_gate_up"] = _normal_bf16(rng, (E, 2 * I, H), WEIGHT_STD)
        out["w_down"] = _normal_bf16(rng, (E, H, I), WEIGHT_STD)
        if name == "skewed":
            out["dy"] = _normal_bf16(rng, (T, H))
    return out


def make_dense_inputs(seed: int = 0, M: int | None = None):
    """Dense GEMM case: A [M,K] ~N(0,1) with 1% outlier channels x20, W [N,K] ~N(0,0.02)."""
    c = dict(CONFIGS["dense"])
    if M is not None:
        c["M"] = M
    M, N, K = c["M"], c["N"], c["K"]
    rng = np.random.default_rng(seed)
    a = rng.standard_normal((M, K), dtype=np.float32)
    cols = rng.choice(K, size=c["n_outlier"], replace=False)
    a[:, cols] *= np.float32(c["outlier_gain"])
    w = rng.standard_normal((N, K), dtype=np.float32) * np.float32(WEIGHT_STD)
    return dict(cfg=c, a=f32_to_bf16_bits(a), w=f32_to_bf16_bits(w), outlier_cols=np.sort(cols))
