"""Plain CPU oracle for the native-NVFP4 W4A4 MoE expert MLP.

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this module. The product path (the
CUDA library and its Python binding) never calls it, and it shares no code
with that path: it has its own BF16, E2M1 and E4M3 arithmetic, its own
scale-layout indexing and its own SwiGLU exponential, written from the
definitions below. Inputs come from the seeded generator module, which holds
none of this arithmetic.

What the pages fix, and where:
  * W4A4: weights and activations are both 4-bit NVFP4 ("miniTE accélère le RL
    en NVFP4 sur B300", lead paragraph; "Hugging Face Releases miniTE
    Framework", section "Technical Mechanism Analysis").
  * Per-token activation scaling: a token's scale must not depend on the other
    tokens of its batch (miniTE report summary, section "Follow the numerical
    execution path").
  * The activation amax is taken inside the MoE permutation and inside the
    routing-weighted SwiGLU, the scale-layout conversion is fused with
    quantization, and experts live in contiguous buffers described by
    device-side offsets (miniTE report summary, section "Two complementary
    interventions").
  * Grouped GEMMs over the experts of a MoE layer ("miniTE accélère le RL en
    NVFP4 sur B300", section "Diagnostic, alignement et noyaux rapides").

What the pages leave open, and the reading taken here (each one is also
listed in the design notes):
  * NVFP4 at the bit level: E2M1 codes (sign bit 3, magnitudes
    {0, .5, 1, 1.5, 2, 3, 4, 6}), one unsigned E4M3 scale per 16 consecutive
    elements of a row, one FP32 global scale per row (activations) or per
    expert matrix (weights).
  * Global scale g = 2688 / amax (2688 = 448 * 6, the largest E4M3 value
    times the largest E2M1 value), or 1 when amax is 0, capped at FLT_MAX.
  * Block scale: s = (amax_block / 6) * g, rounded to E4M3 (nearest, ties to
    even, saturating at 448). Encode factor enc = min(g / sf, FLT_MAX); code
    = E2M1(x * enc) rounded to nearest, ties to the even code, saturating at
    6, keeping the sign (a negative value that rounds to zero gives code 0x8).
    A block whose scale rounds to 0 stores all codes as 0x0.
  * Every fp32 step above is one IEEE operation rounded to nearest, in the
    order written; no fused multiply-add.
  * Dequantized value: val(code) * sf / g.
  * Permuted order: rows sorted by (expert, token, slot); routing ids outside
    [0, E) are dropped.
  * Scale-factor layout: 128-row x 4-column atoms of 512 bytes,
    byte(r, c) = atom*512 + (r%32)*16 + ((r%128)/32)*4 + c%4 with
    atom = (r/128)*(Kc/4) + c/4 and Kc = roundup(K/16, 4); each expert's rows
    are padded to a multiple of 128 and padding bytes are 0.
  * SwiGLU input: the first I columns of gate_up are the gate, the next I the
    up projection; the routing weight is applied in the SwiGLU, not in the
    combine: h = (silu(gate) * up) * w with silu(g) = g / (1 + exp(-g)), where
    exp is the specified function ``exp_spec`` below.
  * Combine: y[t] = BF16(sum over slots j, in slot order, of D[dest_row[t, j]])
    accumulated in fp32.

Every function pinned by the non-GPU tests names its pins in its docstring.
"""
from __future__ import annotations

import numpy as np

F32 = np.float32
FLT_MAX = F32(np.finfo(np.float32).max)
E2M1_MAX = 6.0
E4M3_MAX = 448.0
GLOBAL_NUMERATOR = F32(E4M3_MAX * E2M1_MAX)  # 2688
BLOCK = 16

# --------------------------------------------------------------------------
# BF16 storage
# --------------------------------------------------------------------------


def bf16_to_f32(u: np.ndarray) -> np.ndarray:
    """BF16 bits (uint16) -> float32: the BF16 bits are the top half of the float32."""
    return (np.asarray(u, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(a: np.ndarray) -> np.ndarray:
    """float32 -> BF16 bits, round to nearest, ties to even (drop 16 low bits).

    Pinned against torch's CPU BF16 cast in the tests."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    bits = a.view(np.uint32).astype(np.uint64)
    low = bits & 0xFFFF
    hi = bits >> 16
    round_up = (low > 0x8000) | ((low == 0x8000) & ((hi & 1) == 1))
    out = (hi + round_up.astype(np.uint64)).astype(np.uint16)
    out = np.where(np.isnan(a), np.uint16(0x7FC0), out)
    return out


def f64_to_bf16(a: np.ndarray) -> np.ndarray:
    """float64 -> BF16 bits rounded to nearest-even directly from the float64 value
    (one rounding; used to round exact GEMM results)."""
    a = np.asarray(a, dtype=np.float64)
    out = np.zeros(a.shape, dtype=np.uint16)
    fin = np.isfinite(a) & (a != 0)
    m, e = np.frexp(np.abs(a[fin]))  # |a| = m * 2^e, m in [0.5, 1)
    # BF16 has 8 significant bits; below 2^-126 the quantum is 2^-133.
    q_exp = np.maximum(e - 8, -133)
    q = np.rint(np.ldexp(np.abs(a[fin]), -q_exp))
    val = np.ldexp(q, q_exp)
    f = val.astype(np.float32)  # exact: val has <= 8 significant bits and is in range
    f = np.where(np.signbit(a[fin]), -f, f).astype(np.float32)
    out[fin] = (f.view(np.uint32) >> 16).astype(np.uint16)
    out[a == 0] = np.where(np.signbit(a[a == 0]), 0x8000, 0).astype(np.uint16)
    out[np.isinf(a)] = np.where(a[np.isinf(a)] > 0, 0x7F80, 0xFF80).astype(np.uint16)
    return out


# --------------------------------------------------------------------------
# Scalar formats
# --------------------------------------------------------------------------

E2M1_MAGNITUDES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
# Midpoints between neighbouring magnitudes: a magnitude above midpoint i
# rounds to code i+1 or higher.
_E2M1_MIDPOINTS = (E2M1_MAGNITUDES[:-1] + E2M1_MAGNITUDES[1:]) / 2


def e2m1_decode(codes: np.ndarray) -> np.ndarray:
    """4-bit E2M1 code -> value (float64). Bit 3 is the sign, bits 0..2 index
    the magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6}.

    Pins: all 16 codes against ml_dtypes float4_e2m1fn."""
    c = np.asarray(codes).astype(np.int64)
    mag = E2M1_MAGNITUDES[c & 7]
    return np.where((c & 8) != 0, -mag, mag)


def e2m1_rn(v: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest E2M1 value (ties to the even code,
    saturating at 6) and return the 4-bit codes (uint8, sign in bit 3).

    Pins: ties 0.25->0, 0.75->1, 1.25->1, 1.75->2, 2.5->2, 3.5->4, 5->4;
    brute-force nearest-value search on a dense sweep; ml_dtypes
    float4_e2m1fn on the same sweep."""
    v = np.asarray(v, dtype=np.float32)
    mag = np.abs(v).astype(np.float64)
    # number of midpoints strictly below |v| = code, except that a value exactly
    # on a midpoint sits between codes i and i+1 and takes the even one.
    code = np.searchsorted(_E2M1_MIDPOINTS, mag, side="left")
    on_mid = (code < 7) & (mag == _E2M1_MIDPOINTS[np.minimum(code, 6)])
    code = np.where(on_mid & (code % 2 == 1), code + 1, code)
    sign = np.signbit(v).astype(np.int64)
    return (code | (sign << 3)).astype(np.uint8)


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """Unsigned E4M3 (bias 7, 3 mantissa bits, subnormals m * 2^-9) -> float32.
    Code 0x7F is NaN and is never produced by the encoder.

    Pins: all 256 codes against ml_dtypes float8_e4m3fn."""
    c = np.asarray(codes).astype(np.int64)
    e = (c >> 3) & 0xF
    m = c & 7
    val = np.where(e == 0, np.ldexp(m.astype(np.float64), -9),
                   np.ldexp(1.0 + m / 8.0, e - 7))
    val = np.where((c & 0x7F) == 0x7F, np.nan, val)
    val = np.where((c & 0x80) != 0, -val, val)
    return val.astype(np.float32)


def e4m3_rn_satfinite(s: np.ndarray) -> np.ndarray:
    """Round non-negative finite float32 values to unsigned E4M3, nearest with
    ties to even, saturating at 448; return the 8-bit codes.

    Pins: ml_dtypes float8_e4m3fn (after clamping to 448, since its cast does
    not saturate) over a dense sweep and all E4M3 midpoints; torch's
    float8_e4m3fn cast likewise."""
    s = np.minimum(np.asarray(s, dtype=np.float64), E4M3_MAX)
    _, e = np.frexp(s)
    lead = e - 1  # s in [2^lead, 2^(lead+1))
    # spacing of E4M3 values: 2^(lead-3) for normals (lead >= -6), 2^-9 below
    q_exp = np.where(lead < -6, -9, lead - 3)
    q = np.rint(np.ldexp(s, -q_exp))  # ties to even on the integer count
    val = np.ldexp(q, q_exp)
    # encode the (exactly representable) value
    _, e2 = np.frexp(val)
    lead2 = e2 - 1
    normal = val >= 2.0 ** -6
    man = np.where(normal, np.ldexp(val, -lead2) * 8 - 8, 0).astype(np.int64)
    sub = np.where(normal, 0, np.ldexp(val, 9)).astype(np.int64)
    code = np.where(normal, ((lead2 + 7) << 3) | man, sub)
    return code.astype(np.uint8)


# --------------------------------------------------------------------------
# Quantization (per-token / per-group NVFP4)
# --------------------------------------------------------------------------


def global_scale(amax: np.ndarray) -> np.ndarray:
    """g = min(2688 / amax, FLT_MAX) for amax > 0, else 1 (fp32 division)."""
    amax = np.asarray(amax, dtype=F32)
    with np.errstate(divide="ignore", over="ignore"):
        g = np.where(amax > 0, np.minimum(GLOBAL_NUMERATOR / amax, FLT_MAX), F32(1.0))
    return g.astype(F32)


def quantize_rows(x: np.ndarray, g: np.ndarray):
    """Quantize rows of x (float32 [R, C], C % 16 == 0) with per-row global
    scales g (float32 [R]). Returns (codes uint8 [R, C/2] with element 2i in
    the low nibble, sf uint8 [R, C/16], row-major, not swizzled).

    Steps per 16-element block b of a row: amax_b = max|x|; s = (amax_b / 6) * g;
    sf = E4M3(s); if sf == 0 every code is 0x0, otherwise enc = min(g / sf,
    FLT_MAX) and code_i = E2M1(x_i * enc).

    Pins: exact round trip of grid * 2^j rows; the dequantization error bound;
    the row maximum maps to code +-6 with scale 448; zero and denormal rows;
    batch-reshuffle invariance; tensor-wide negative control."""
    x = np.asarray(x, dtype=F32)
    R, C = x.shape
    assert C % BLOCK == 0
    g = np.asarray(g, dtype=F32).reshape(R, 1, 1)
    blocks = x.reshape(R, C // BLOCK, BLOCK)
    amax_b = np.max(np.abs(blocks), axis=2, keepdims=True)
    s = (amax_b / F32(E2M1_MAX)) * g
    sf = e4m3_rn_satfinite(s[..., 0])
    sf_val = e4m3_decode(sf)[..., None]
    with np.errstate(divide="ignore", over="ignore", invalid="ignore"):
        enc = np.where(sf_val > 0, np.minimum(g / sf_val, FLT_MAX), F32(0)).astype(F32)
        scaled = (blocks * enc).astype(F32)
    q = e2m1_rn(scaled)
    q = np.where(sf[..., None] == 0, np.uint8(0), q).reshape(R, C)
    codes = (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)
    return codes, sf


def quantize_per_row(x: np.ndarray):
    """Activation mode: each row gets its own global scale from its own amax
    (per-token scaling, miniTE report summary, "Follow the numerical execution
    path"). Returns (codes, sf, g)."""
    x = np.asarray(x, dtype=F32)
    g = global_scale(np.max(np.abs(x), axis=1))
    codes, sf = quantize_rows(x, g)
    return codes, sf, g


def quantize_per_tensor(x: np.ndarray, g: np.ndarray | None = None):
    """Weight mode: one global scale for the whole matrix (one expert's weight),
    from its amax unless g is given. Returns (codes, sf, g scalar)."""
    x = np.asarray(x, dtype=F32)
    if g is None:
        g = global_scale(np.max(np.abs(x)))
    g = F32(g)
    codes, sf = quantize_rows(x, np.full(x.shape[0], g, dtype=F32))
    return codes, sf, g


def quantize_tensor_wide_activations(x: np.ndarray):
    """NEGATIVE CONTROL, not part of the path: activations scaled by one amax
    over the whole batch, the policy whose batch dependence per-token scaling
    removes (miniTE report summary, "Follow the numerical execution path")."""
    x = np.asarray(x, dtype=F32)
    g = global_scale(np.max(np.abs(x)))
    codes, sf = quantize_rows(x, np.full(x.shape[0], g, dtype=F32))
    return codes, sf, np.full(x.shape[0], g, dtype=F32)


def unpack_codes(codes: np.ndarray) -> np.ndarray:
    """uint8 [R, C/2] packed codes -> uint8 [R, C] codes (low nibble first)."""
    c = np.asarray(codes, dtype=np.uint8)
    out = np.empty(c.shape[:-1] + (c.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = c & 0xF
    out[..., 1::2] = c >> 4
    return out


def dequantize(codes: np.ndarray, sf: np.ndarray, g) -> np.ndarray:
    """float64 [R, C] values val(code) * sf / g (g per row or scalar)."""
    v = e2m1_decode(unpack_codes(codes))
    R, C = v.shape
    s = np.repeat(e4m3_decode(sf).astype(np.float64), BLOCK, axis=1)
    g = np.broadcast_to(np.asarray(g, dtype=np.float64).reshape(-1, 1), (R, 1))
    return v * s / g


# --------------------------------------------------------------------------
# Scale-factor layout (MMA-ready 128x4 atoms)
# --------------------------------------------------------------------------


def roundup(a: int, b: int) -> int:
    return (a + b - 1) // b * b


def sf_swizzle_offset(r: np.ndarray, c: np.ndarray, kc: int) -> np.ndarray:
    """Byte offset of the scale of row r, block column c inside a region whose
    rows are padded to 128 and columns to kc = roundup(K/16, 4)."""
    r = np.asarray(r, dtype=np.int64)
    c = np.asarray(c, dtype=np.int64)
    atom = (r // 128) * (kc // 4) + c // 4
    return atom * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + c % 4


def swizzle_sf(sf: np.ndarray) -> np.ndarray:
    """Row-major sf [R, C16] -> flat uint8 [roundup(R,128) * roundup(C16,4)] in
    the 128x4-atom layout, padding bytes 0.

    Pins: equals the documented reshape [R/128, 4, 32, Kc/4, 4] ->
    [R/128, Kc/4, 32, 4, 4] of the padded matrix; it is a bijection."""
    R, C16 = sf.shape
    kc = roundup(C16, 4)
    out = np.zeros(roundup(R, 128) * kc, dtype=np.uint8)
    r, c = np.meshgrid(np.arange(R), np.arange(C16), indexing="ij")
    out[sf_swizzle_offset(r, c, kc)] = sf
    return out


def unswizzle_sf(buf: np.ndarray, R: int, C16: int) -> np.ndarray:
    kc = roundup(C16, 4)
    r, c = np.meshgrid(np.arange(R), np.arange(C16), indexing="ij")
    return np.asarray(buf)[sf_swizzle_offset(r, c, kc)]


# --------------------------------------------------------------------------
# Weight quantization (per expert), along K or along N (dgrad layout)
# --------------------------------------------------------------------------


def quantize_weights(w_bf16: np.ndarray, along_rows: bool = False, g_in=None):
    """Quantize each expert matrix w[e] ([R, C] BF16) with one global scale per
    expert. along_rows=False: blocks of 16 along C (the forward K-major
    layout), output codes [E, R, C/2]. along_rows=True: the matrix is
    transposed first and blocks run along R (the dgrad layout of the same
    weight), output codes [E, C, R/2]. The global scale depends only on the
    expert's amax, so both orientations share it (g_in may pass it in).

    Returns (codes [E, rows', cols'/2], sf [E, rows', cols'/16] row-major,
    sf_swizzled [E, roundup(rows',128) * roundup(cols'/16,4)], g [E])."""
    E = w_bf16.shape[0]
    codes_l, sf_l, sw_l, g_l = [], [], [], []
    for e in range(E):
        we = bf16_to_f32(w_bf16[e])
        if along_rows:
            we = np.ascontiguousarray(we.T)
        ge = None if g_in is None else F32(np.asarray(g_in, dtype=F32)[e])
        c, s, g = quantize_per_tensor(we, ge)
        codes_l.append(c)
        sf_l.append(s)
        sw_l.append(swizzle_sf(s))
        g_l.append(g)
    return (np.stack(codes_l), np.stack(sf_l), np.stack(sw_l), np.array(g_l, dtype=F32))


# --------------------------------------------------------------------------
# MoE permutation fused with per-token quantization
# --------------------------------------------------------------------------


def moe_permute(topk_ids: np.ndarray, E: int):
    """Expert-contiguous order of the (token, slot) pairs.

    Rows are ordered by (expert, token, slot) ascending; pairs whose id is
    outside [0, E) are dropped. Returns dict with expert_offsets [E+1]
    (exclusive prefix of counts), sf_row_offsets [E+1] (prefix of counts
    rounded up to 128), perm_src [M] (token of each row), perm_slot [M],
    dest_row [T, k] (row of each pair, -1 if dropped), n_bad (dropped pairs).

    Pins: brute-force sort on tiny inputs; counts sum to the kept pairs;
    dest_row inverts perm_src; empty experts have equal offsets."""
    ids = np.asarray(topk_ids, dtype=np.int64)
    T, k = ids.shape
    tok, slot = np.meshgrid(np.arange(T), np.arange(k), indexing="ij")
    ok = (ids >= 0) & (ids < E)
    t_ok, j_ok, e_ok = tok[ok], slot[ok], ids[ok]
    order = np.lexsort((j_ok, t_ok, e_ok))  # last key is the primary key
    perm_src = t_ok[order]
    perm_slot = j_ok[order]
    counts = np.bincount(e_ok, minlength=E)
    expert_offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    padded = (counts + 127) // 128 * 128
    sf_row_offsets = np.concatenate([[0], np.cumsum(padded)]).astype(np.int32)
    dest_row = np.full((T, k), -1, dtype=np.int32)
    dest_row[perm_src, perm_slot] = np.arange(len(order), dtype=np.int32)
    return dict(expert_offsets=expert_offsets, sf_row_offsets=sf_row_offsets,
                perm_src=perm_src.astype(np.int32), perm_slot=perm_slot.astype(np.int32),
                dest_row=dest_row, n_bad=int((~ok).sum()))


def place_sf_per_expert(sf_rows: np.ndarray, expert_offsets, sf_row_offsets) -> np.ndarray:
    """Swizzle the row-major scales of permuted rows into per-expert regions:
    expert e's rows start at padded row sf_row_offsets[e]; padding is 0.
    Returns flat uint8 [sf_row_offsets[E] * Kc]."""
    C16 = sf_rows.shape[1]
    kc = roundup(C16, 4)
    E = len(expert_offsets) - 1
    out = np.zeros(int(sf_row_offsets[E]) * kc, dtype=np.uint8)
    for e in range(E):
        a, b = int(expert_offsets[e]), int(expert_offsets[e + 1])
        if b == a:
            continue
        reg = swizzle_sf(sf_rows[a:b])
        base = int(sf_row_offsets[e]) * kc
        out[base:base + reg.size] = reg
    return out


def moe_permute_quant(x_bf16: np.ndarray, topk_ids: np.ndarray, topk_w, E: int):
    """The permute step: expert-contiguous rows of per-token NVFP4 codes.

    Each permuted row p holds quantize_per_row(x[perm_src[p]]); since a row's
    quantization depends on that row alone (per-token scaling), the token is
    quantized once and its result copied to each of its k rows. Returns the
    permutation dict plus codes [M, H/2], sf (row-major [M, H/16]), sf_swizzled
    (per-expert regions), row_g [M], perm_w [M] (or None)."""
    perm = moe_permute(topk_ids, E)
    xf = bf16_to_f32(x_bf16)
    codes_t, sf_t, g_t = quantize_per_row(xf)
    src = perm["perm_src"]
    out = dict(perm)
    out["codes"] = codes_t[src]
    out["sf"] = sf_t[src]
    out["row_g"] = g_t[src]
    out["sf_swizzled"] = place_sf_per_expert(out["sf"], perm["expert_offsets"], perm["sf_row_offsets"])
    out["perm_w"] = None if topk_w is None else np.asarray(topk_w, dtype=F32)[src, perm["perm_slot"]]
    return out


# --------------------------------------------------------------------------
# Grouped GEMM (exact)
# --------------------------------------------------------------------------


def row_experts(expert_offsets, rows) -> np.ndarray:
    """Expert of each permuted row (the e with offsets[e] <= row < offsets[e+1])."""
    off = np.asarray(expert_offsets, dtype=np.int64)
    return np.searchsorted(off, np.asarray(rows), side="right") - 1


def grouped_gemm_exact(a_codes, a_sf, a_g, b_codes, b_sf, b_g, expert_offsets, rows=None):
    """y[m, n] = sum_k xhat[m, k] * what_e[n, k] for e = expert of row m, with
    xhat = val * sf / g (NVFP4 dequantization), computed in float64.

    The products val*sf are exact in float64, so the only roundings are the
    float64 sums and the final division by g_a * g_w. Returns (y [rows, N]
    float64, abs_sum [rows, N] = sum_k |xhat_k * what_k|, the scale of the
    tolerance). ``rows`` selects permuted rows (default all).

    Pins: brute-force exact tiny GEMMs with rational arithmetic; one-hot weight
    rows reproduce xhat; E=1 equals the dense matmul of the dequantized
    operands."""
    off = np.asarray(expert_offsets, dtype=np.int64)
    M = int(off[-1])
    rows = np.arange(M) if rows is None else np.asarray(rows, dtype=np.int64)
    ex = row_experts(off, rows)
    N = b_codes.shape[1]
    y = np.zeros((len(rows), N))
    bound = np.zeros((len(rows), N))
    va = e2m1_decode(unpack_codes(a_codes[rows]))
    sa = np.repeat(e4m3_decode(a_sf[rows]).astype(np.float64), BLOCK, axis=1)
    a_s = va * sa
    for e in np.unique(ex):
        sel = np.nonzero(ex == e)[0]
        vb = e2m1_decode(unpack_codes(b_codes[e]))
        sb = np.repeat(e4m3_decode(b_sf[e]).astype(np.float64), BLOCK, axis=1)
        b_s = vb * sb
        denom = np.asarray(a_g, dtype=np.float64)[rows[sel]][:, None] * np.float64(b_g[e])
        y[sel] = (a_s[sel] @ b_s.T) / denom
        bound[sel] = (np.abs(a_s[sel]) @ np.abs(b_s).T) / denom
    return y, bound


def grouped_gemm_fp32_accumulate(a_codes, a_sf, a_g, b_codes, b_sf, b_g, expert_offsets):
    """The same grouped GEMM with float32 dequantized operands and float32
    accumulation (numpy matmul in float32, summation order left to the
    library). This is the timed CPU baseline; parity uses
    ``grouped_gemm_exact``.

    Pins: within the float32 summation bound (K + 2) * 2^-24 * sum|ahat bhat|
    of the rational brute force on tiny multi-expert GEMMs; one-hot weights
    of value 1 give exactly the float32 nearest to the rational activation;
    within the same bound of the exact GEMM at K = 512 with an empty expert."""
    off = np.asarray(expert_offsets, dtype=np.int64)
    M = int(off[-1])
    N = b_codes.shape[1]
    y = np.zeros((M, N), dtype=F32)
    for e in range(len(off) - 1):
        a0, a1 = int(off[e]), int(off[e + 1])
        if a1 == a0:
            continue
        xa = dequantize(a_codes[a0:a1], a_sf[a0:a1], a_g[a0:a1]).astype(F32)
        xb = dequantize(b_codes[e], b_sf[e], b_g[e]).astype(F32)
        y[a0:a1] = xa @ xb.T
    return y


# --------------------------------------------------------------------------
# Routing-weighted SwiGLU fused with per-row requantization
# --------------------------------------------------------------------------

# Cody-Waite reduction constants: LN2_HI is ln 2 truncated to 15 significant
# bits (so n * LN2_HI is exact for |n| < 512), LN2_LO the float32 rounding of
# the remainder ln 2 - LN2_HI.
_LN2 = 0.6931471805599453094
LN2_HI = F32(np.ldexp(np.floor(np.ldexp(_LN2, 15)), -15))
LN2_LO = F32(_LN2 - float(LN2_HI))
LOG2E = F32(1.4426950408889634074)
# Taylor coefficients 1/n! for n = 0..7, rounded to float32.
EXP_COEFFS = [F32(1.0 / f) for f in (1, 1, 2, 6, 24, 120, 720, 5040)]
EXP_CLAMP_LO = F32(-87.0)
EXP_CLAMP_HI = F32(88.0)


def exp_spec(x: np.ndarray) -> np.ndarray:
    """Specified float32 exponential (Cody and Waite's additive range reduction
    with a two-part ln 2, then a degree-7 Taylor polynomial of e^r):

        x <- clamp(x, -87, 88)
        n <- rint(x * LOG2E)                (ties to even)
        r <- (x - n * LN2_HI) - n * LN2_LO
        p <- c7; p <- p * r + c_i for i = 6..0   (separate multiply and add)
        result <- p * 2^n

    Every operation is one float32 IEEE operation rounded to nearest; no fused
    multiply-add. Pins: within 2 ulp of the correctly rounded e^x on a dense
    sweep of [-87, 88]; exact at x = 0."""
    x = np.clip(np.asarray(x, dtype=F32), EXP_CLAMP_LO, EXP_CLAMP_HI).astype(F32)
    n = np.rint((x * LOG2E).astype(F32)).astype(F32)
    r = ((x - (n * LN2_HI).astype(F32)).astype(F32) - (n * LN2_LO).astype(F32)).astype(F32)
    p = EXP_COEFFS[7] * np.ones_like(r)
    for c in reversed(EXP_COEFFS[:7]):
        p = ((p * r).astype(F32) + c).astype(F32)
    return np.ldexp(p, n.astype(np.int32)).astype(F32)


def swiglu_weighted(gate_up: np.ndarray, perm_w) -> np.ndarray:
    """h = (silu(g) * u) * w in float32, silu(g) = g / (1 + exp_spec(-g)),
    g = gate_up[:, :I], u = gate_up[:, I:], w the routing weight of the row
    (1 when perm_w is None)."""
    gu = np.asarray(gate_up, dtype=F32)
    I = gu.shape[1] // 2
    g, u = gu[:, :I], gu[:, I:]
    silu = (g / (F32(1.0) + exp_spec(-g)).astype(F32)).astype(F32)
    h = (silu * u).astype(F32)
    if perm_w is not None:
        h = (h * np.asarray(perm_w, dtype=F32)[:, None]).astype(F32)
    return h


def swiglu_weighted_quant(gate_up_bf16: np.ndarray, perm_w, expert_offsets, sf_row_offsets):
    """The weighted SwiGLU step: h per permuted row, then per-row NVFP4 with the
    amax taken over h (miniTE report summary, "Two complementary
    interventions"). Rows at or beyond expert_offsets[E] are not produced.
    Returns dict codes [M, I/2], sf [M, I/16], sf_swizzled, row_g [M], h."""
    M = int(np.asarray(expert_offsets)[-1])
    gu = bf16_to_f32(gate_up_bf16[:M])
    w = None if perm_w is None else np.asarray(perm_w)[:M]
    h = swiglu_weighted(gu, w)
    codes, sf, g = quantize_per_row(h)
    return dict(codes=codes, sf=sf, row_g=g, h=h,
                sf_swizzled=place_sf_per_expert(sf, expert_offsets, sf_row_offsets))


def swiglu_backward(gate_up: np.ndarray, dh: np.ndarray, perm_w) -> np.ndarray:
    """Gradient of h = (silu(g) * u) * w with respect to gate_up = [g | u],
    given the gradient dh of h (float32 [M, I]); the routing weight w is a
    constant here. With d = 1 + exp_spec(-g), the sigmoid s = 1 / d and
    silu = g / d (as in the forward), the chain rule gives
        silu'(g) = s * (1 + g * (1 - s))
        dg = ((dh * u) * w) * silu'(g)
        du = (dh * silu) * w
    every step one float32 IEEE operation rounded to nearest, in this order.
    Returns float32 [M, 2I] = [dg | du].

    Pins: the float64 derivative of the forward formula (central differences
    of swiglu_weighted and the closed form), g = 0 (silu' = 1/2, du = 0),
    large |g| (silu' -> 1 or 0)."""
    gu = np.asarray(gate_up, dtype=F32)
    I = gu.shape[1] // 2
    g, u = gu[:, :I], gu[:, I:]
    dh = np.asarray(dh, dtype=F32)
    w = F32(1.0) if perm_w is None else np.asarray(perm_w, dtype=F32)[:, None]
    d = (F32(1.0) + exp_spec(-g)).astype(F32)
    sig = (F32(1.0) / d).astype(F32)
    silu = (g / d).astype(F32)
    dsilu = (sig * (F32(1.0) + (g * (F32(1.0) - sig).astype(F32)).astype(F32)).astype(F32)).astype(F32)
    dg = ((((dh * u).astype(F32)) * w).astype(F32) * dsilu).astype(F32)
    du = (((dh * silu).astype(F32)) * w).astype(F32)
    return np.concatenate([dg, du], axis=1)


def swiglu_backward_quant(gate_up_bf16: np.ndarray, dh_bf16: np.ndarray, perm_w,
                          expert_offsets, sf_row_offsets):
    """The SwiGLU backward step: [dg | du] per permuted row, then per-row NVFP4
    over its 2I values, scales placed per expert like every permuted
    activation (input of the gate_up dgrad GEMM). Rows at or beyond
    expert_offsets[E] are not produced. Returns dict codes [M, I] (2I/2
    bytes), sf [M, 2I/16], sf_swizzled, row_g [M], dgu."""
    M = int(np.asarray(expert_offsets)[-1])
    gu = bf16_to_f32(gate_up_bf16[:M])
    dh = bf16_to_f32(dh_bf16[:M])
    w = None if perm_w is None else np.asarray(perm_w)[:M]
    dgu = swiglu_backward(gu, dh, w)
    codes, sf, g = quantize_per_row(dgu)
    return dict(codes=codes, sf=sf, row_g=g, dgu=dgu,
                sf_swizzled=place_sf_per_expert(sf, expert_offsets, sf_row_offsets))


# --------------------------------------------------------------------------
# Weight gradient: operands quantized along tokens, K ragged per expert
# --------------------------------------------------------------------------

WGRAD_K_ALIGN = 256  # tokens: each expert's K range is padded to a multiple of this


def wgrad_token_offsets(expert_offsets) -> np.ndarray:
    """K layout of the token-axis operands of a weight-gradient GEMM: expert
    e's tokens occupy columns [kofs[e], kofs[e] + count_e) of a [C, kofs[E]]
    matrix, kofs being the prefix of the counts rounded up to 256 (reading:
    the pages do not describe the backward's layout; 256 tokens is one
    128-byte chunk of E2M1 codes). Columns past an expert's count are 0."""
    off = np.asarray(expert_offsets, dtype=np.int64)
    counts = off[1:] - off[:-1]
    padded = (counts + WGRAD_K_ALIGN - 1) // WGRAD_K_ALIGN * WGRAD_K_ALIGN
    return np.concatenate([[0], np.cumsum(padded)]).astype(np.int32)


def quantize_tokens_per_expert(rows: np.ndarray, expert_offsets):
    """One operand of a weight-gradient GEMM. rows: float32 [M, C], the
    permuted rows (expert-contiguous, expert_offsets). For each expert e the
    rows X_e [count_e, C] are transposed to [C, count_e], zero-padded to the
    expert's K range, and quantized with one global scale per expert (from
    the amax of X_e; 1 for an empty expert) and blocks of 16 consecutive
    tokens (reading: the gradient sums over the expert's tokens, so the
    scale cannot vary along them; one scale per expert, as for weights).
    Returns dict codes [C, K/2], sf [C, K/16] row-major, sf_swizzled
    (roundup(C, 128) x K/16 atoms), g [E], kofs [E+1] (K = kofs[E]).

    Pins: per expert, equal to the per-expert weight quantization of the
    padded block along its rows; exact round trip of grid values; the
    dequantization error bound."""
    x = np.asarray(rows, dtype=F32)
    off = np.asarray(expert_offsets, dtype=np.int64)
    kofs = wgrad_token_offsets(off)
    E = len(off) - 1
    C = x.shape[1]
    K = int(kofs[E])
    codes = np.zeros((C, K // 2), dtype=np.uint8)
    sf = np.zeros((C, K // BLOCK), dtype=np.uint8)
    g = np.ones(E, dtype=F32)
    for e in range(E):
        a, b = int(off[e]), int(off[e + 1])
        if b == a:
            continue
        k0, k1 = int(kofs[e]), int(kofs[e + 1])
        xt = np.zeros((C, k1 - k0), dtype=F32)
        xt[:, :b - a] = x[a:b].T
        ce, se, ge = quantize_per_tensor(xt)
        codes[:, k0 // 2:k1 // 2] = ce
        sf[:, k0 // BLOCK:k1 // BLOCK] = se
        g[e] = ge
    return dict(codes=codes, sf=sf, sf_swizzled=swizzle_sf(sf) if K else np.zeros(0, np.uint8),
                g=g, kofs=kofs)


def wgrad_exact(a, b):
    """Weight gradient per expert from two token-axis operands (dicts of
    ``quantize_tokens_per_expert`` over the same routing):
        out[e, n, i] = sum_{k in expert e's K range} ahat[n, k] * bhat[i, k]
    with xhat = val * sf / g_e, in float64 (val*sf exact; the only roundings
    are the float64 sums and the final division by g_a[e] * g_b[e]). Returns
    (out [E, Ca, Cb] float64, abs_sum [E, Ca, Cb], the tolerance scale).

    Pins: rational brute force on tiny operands; equality with the matmul of
    the dequantized per-expert operands."""
    kofs = np.asarray(a["kofs"], dtype=np.int64)
    E = len(kofs) - 1
    va = e2m1_decode(unpack_codes(a["codes"])) * np.repeat(
        e4m3_decode(a["sf"]).astype(np.float64), BLOCK, axis=1)
    vb = e2m1_decode(unpack_codes(b["codes"])) * np.repeat(
        e4m3_decode(b["sf"]).astype(np.float64), BLOCK, axis=1)
    Ca, Cb = va.shape[0], vb.shape[0]
    out = np.zeros((E, Ca, Cb))
    bound = np.zeros((E, Ca, Cb))
    for e in range(E):
        k0, k1 = int(kofs[e]), int(kofs[e + 1])
        if k1 == k0:
            continue
        denom = np.float64(a["g"][e]) * np.float64(b["g"][e])
        out[e] = (va[:, k0:k1] @ vb[:, k0:k1].T) / denom
        bound[e] = (np.abs(va[:, k0:k1]) @ np.abs(vb[:, k0:k1]).T) / denom
    return out, bound


# --------------------------------------------------------------------------
# Combine (unpermute)
# --------------------------------------------------------------------------


def moe_combine(expert_out_bf16: np.ndarray, dest_row: np.ndarray) -> np.ndarray:
    """y[t] = BF16(sum_j D[dest_row[t, j]]): float32 running sum in slot order
    starting from 0, skipping dropped pairs (dest_row -1), one final rounding
    to BF16. Returns BF16 bits [T, N]."""
    D = bf16_to_f32(expert_out_bf16)
    T, k = dest_row.shape
    acc = np.zeros((T, D.shape[1]), dtype=F32)
    for j in range(k):
        d = dest_row[:, j]
        ok = d >= 0
        acc[ok] = (acc[ok] + D[d[ok]]).astype(F32)
    return f32_to_bf16(acc)


# --------------------------------------------------------------------------
# The whole expert MLP forward
# --------------------------------------------------------------------------


def moe_mlp_forward(x_bf16, topk_ids, topk_w, E, wgu_q, wd_q, rows_only=None):
    """Chain: permute+quant -> grouped gate_up GEMM (BF16 out, exact then one
    rounding) -> weighted SwiGLU + requant -> grouped down GEMM (BF16 out) ->
    combine. wgu_q / wd_q are the (codes, sf, sf_swizzled, g) tuples of
    ``quantize_weights``. Returns dict with every intermediate."""
    pq = moe_permute_quant(x_bf16, topk_ids, topk_w, E)
    off = pq["expert_offsets"]
    gu, _ = grouped_gemm_exact(pq["codes"], pq["sf"], pq["row_g"], wgu_q[0], wgu_q[1], wgu_q[3], off)
    gu_bf16 = f64_to_bf16(gu)
    sw = swiglu_weighted_quant(gu_bf16, pq["perm_w"], off, pq["sf_row_offsets"])
    d, _ = grouped_gemm_exact(sw["codes"], sw["sf"], sw["row_g"], wd_q[0], wd_q[1], wd_q[3], off)
    d_bf16 = f64_to_bf16(d)
    y = moe_combine(d_bf16, pq["dest_row"])
    return dict(permute=pq, gate_up=gu_bf16, swiglu=sw, down=d_bf16, y=y)
