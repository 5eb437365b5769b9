"""Python binding of libminite.so (include/minite.h) through ctypes.

Argument marshalling only: every step of the path runs in the library's CUDA
kernels. PyTorch provides device memory and streams. The functions named
``minite_*`` mirror the C entry points one to one and take torch tensors;
the helpers below them only allocate outputs with torch and call those.
Nothing here falls back to a CPU implementation: without the built library
every call raises ``MiniteError``.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

SCALE_PER_ROW, SCALE_PER_GROUP = 0, 1
ALONG_COLS, ALONG_ROWS = 0, 1
OUT_BF16, OUT_FP32 = 0, 1
OP_QUANTIZE, OP_PERMUTE_QUANT, OP_COMBINE_BACKWARD_QUANT, OP_QUANTIZE_TOKENS = 0, 1, 2, 3
OP_GATE_UP_SWIGLU = 4
ERR_TIMEOUT, ERR_BAD_ROUTING = 4, 5

EXPORTS = [
    "minite_quantize_nvfp4", "minite_moe_permute_quant", "minite_grouped_gemm_nvfp4",
    "minite_swiglu_weighted_quant", "minite_swiglu_backward_quant", "minite_moe_combine",
    "minite_workspace_bytes",
    "minite_status_string", "minite_version", "minite_test_convert",
    "minite_set_wait_budget_ns", "minite_moe_permute_quant_noalloc", "minite_set_gemm_variant",
    "minite_test_div6_exhaustive", "minite_test_convert_digest", "minite_quantize_nvfp4_dual",
    "minite_moe_combine_backward_quant", "minite_quantize_tokens_nvfp4",
    "minite_swiglu_weighted_quant_keep_h", "minite_grouped_gemm_wgrad_nvfp4",
    "minite_swiglu_backward_quant_keep", "minite_gate_up_swiglu_quant_nvfp4",
]


class MiniteError(RuntimeError):
    pass


_LIB = None
_vp, _i64, _i32, _int, _sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int, ctypes.c_size_t


def load(path: str | None = None):
    """Load libminite.so (built in-tree by ``build.build()``)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = path or _build.LIB
    if not os.path.exists(path):
        raise MiniteError(f"{path} is not built; run nvfp4_w4a4_moe_permute_gb300.build.build()")
    lib = ctypes.CDLL(path)
    sig = {
        "minite_quantize_nvfp4": [_vp, _i64, _i64, _i64, _int, _int, _vp, _vp, _vp, _vp, _vp, _sz, _vp, _vp],
        "minite_quantize_nvfp4_dual": [_vp, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp,
                                       _vp],
        "minite_moe_permute_quant": [_vp, _vp, _vp, _i64, _i64, _i32, _i32, _vp, _vp, _vp, _vp, _vp,
                                     _vp, _vp, _vp, _vp, _sz, _vp, _vp],
        "minite_moe_permute_quant_noalloc": [_vp, _vp, _vp, _i64, _i64, _i32, _i32, _vp, _vp, _vp,
                                             _vp, _vp, _vp, _vp, _vp, _vp, _vp],
        "minite_moe_combine_backward_quant": [_vp, _i64, _i64, _i32, _i32, _vp, _vp, _vp, _vp, _vp,
                                              _vp, _vp, _vp, _sz, _vp, _vp],
        "minite_quantize_tokens_nvfp4": [_vp, _i64, _vp, _vp, _i64, _i64, _i32, _vp, _i64, _vp, _vp,
                                         _vp, _vp, _vp, _sz, _vp, _vp],
        "minite_grouped_gemm_wgrad_nvfp4": [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i64, _i64, _i64,
                                            _vp, _int, _vp, _vp],
        "minite_grouped_gemm_nvfp4": [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i32,
                                      _vp, _int, _vp, _vp],
        "minite_gate_up_swiglu_quant_nvfp4": [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64,
                                              _i64, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp,
                                              _vp],
        "minite_swiglu_weighted_quant": [_vp, _vp, _i64, _i64, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp],
        "minite_swiglu_weighted_quant_keep_h": [_vp, _vp, _i64, _i64, _i32, _vp, _vp, _vp, _vp, _vp,
                                                _vp, _vp, _vp, _vp],
        "minite_swiglu_backward_quant": [_vp, _vp, _vp, _i64, _i64, _i32, _vp, _vp, _vp, _vp, _vp, _vp,
                                         _vp],
        "minite_swiglu_backward_quant_keep": [_vp, _vp, _vp, _i64, _i64, _i32, _vp, _vp, _vp, _vp,
                                              _vp, _vp, _vp, _vp, _vp],
        "minite_moe_combine": [_vp, _vp, _i64, _i64, _i64, _i32, _vp, _vp, _vp],
        "minite_test_convert": [_vp, _i64, _vp, _vp, _vp, _vp],
        "minite_test_div6_exhaustive": [_vp, _vp],
        "minite_test_convert_digest": [ctypes.c_ulonglong, ctypes.c_ulonglong, _vp, _vp],
    }
    for name, args in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = _int
    lib.minite_workspace_bytes.argtypes = [_int, _i64, _i64, _i32, _i32]
    lib.minite_workspace_bytes.restype = _sz
    lib.minite_status_string.argtypes = [_int]
    lib.minite_status_string.restype = ctypes.c_char_p
    lib.minite_version.argtypes = []
    lib.minite_version.restype = ctypes.c_char_p
    lib.minite_set_wait_budget_ns.argtypes = [ctypes.c_uint64]
    lib.minite_set_wait_budget_ns.restype = None
    lib.minite_set_gemm_variant.argtypes = [_int]
    lib.minite_set_gemm_variant.restype = None
    _LIB = lib
    return lib


def _p(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise MiniteError("expected a CUDA tensor")
    return ctypes.c_void_p(t.data_ptr())


def _s(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(rc: int, name: str):
    if rc != 0:
        raise MiniteError(f"{name}: {minite_status_string(rc)} (status {rc})")


def minite_status_string(rc: int) -> str:
    return load().minite_status_string(rc).decode()


def minite_version() -> str:
    return load().minite_version().decode()


def minite_workspace_bytes(op: int, a: int, b: int = 0, E: int = 0, k: int = 0) -> int:
    return int(load().minite_workspace_bytes(op, a, b, E, k))


def minite_set_wait_budget_ns(ns: int):
    load().minite_set_wait_budget_ns(int(ns))


def minite_set_gemm_variant(variant: int):
    """0 automatic, 1 single-CTA grouped-GEMM kernel, 2 CTA-pair kernel."""
    load().minite_set_gemm_variant(int(variant))


def minite_quantize_nvfp4(x, scale_mode, orientation, codes, sf, gscale_out, gscale_in=None,
                          workspace=None, status=None, stream=None):
    """x: bf16 [groups, rows, cols] (or [rows, cols] = one group)."""
    g, r, c = (1,) + tuple(x.shape) if x.dim() == 2 else tuple(x.shape)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().minite_quantize_nvfp4(_p(x), g, r, c, scale_mode, orientation, _p(gscale_in),
                                      _p(codes), _p(sf), _p(gscale_out), _p(workspace), ws_bytes,
                                      _p(status), _s(stream))
    _check(rc, "minite_quantize_nvfp4")


def minite_quantize_nvfp4_dual(x, codes_k, sf_k, codes_n, sf_n, gscale_out, workspace,
                               status=None, stream=None):
    """x: bf16 [groups, rows, cols] (or [rows, cols] = one group); per-group scales."""
    g, r, c = (1,) + tuple(x.shape) if x.dim() == 2 else tuple(x.shape)
    ws_bytes = workspace.numel() * workspace.element_size()
    rc = load().minite_quantize_nvfp4_dual(_p(x), g, r, c, _p(codes_k), _p(sf_k), _p(codes_n),
                                           _p(sf_n), _p(gscale_out), _p(workspace), ws_bytes,
                                           _p(status), _s(stream))
    _check(rc, "minite_quantize_nvfp4_dual")


def quantize_dual(x, stream=None):
    """Weight x ([rows, cols] or [groups, rows, cols]) quantized per group in both
    orientations; returns (forward dict, transposed dict) like quantize()."""
    dev = x.device
    g3 = x if x.dim() == 3 else x.unsqueeze(0)
    G, R, C = g3.shape
    fk = dict(codes=torch.empty((G, R, C // 2), dtype=torch.uint8, device=dev),
              sf=torch.empty((G, sf_bytes((R + 127) // 128 * 128, C)), dtype=torch.uint8, device=dev))
    fn = dict(codes=torch.empty((G, C, R // 2), dtype=torch.uint8, device=dev),
              sf=torch.empty((G, sf_bytes((C + 127) // 128 * 128, R)), dtype=torch.uint8, device=dev))
    g = torch.empty((G,), dtype=torch.float32, device=dev)
    ws = torch.empty(minite_workspace_bytes(OP_QUANTIZE, G), dtype=torch.uint8, device=dev)
    minite_quantize_nvfp4_dual(g3, fk["codes"], fk["sf"], fn["codes"], fn["sf"], g, ws, stream=stream)
    fk["g"] = g
    fn["g"] = g
    if x.dim() == 2:
        for d in (fk, fn):
            d["codes"], d["sf"] = d["codes"][0], d["sf"][0]
    return fk, fn


def minite_moe_permute_quant(x, topk_ids, topk_w, E, codes, sf, row_g, expert_offsets,
                             sf_row_offsets, perm_src, dest_row, perm_w, workspace, status=None,
                             stream=None):
    T, H = x.shape
    k = topk_ids.shape[1]
    ws_bytes = workspace.numel() * workspace.element_size()
    rc = load().minite_moe_permute_quant(_p(x), _p(topk_ids), _p(topk_w), T, H, E, k, _p(codes),
                                         _p(sf), _p(row_g), _p(expert_offsets),
                                         _p(sf_row_offsets), _p(perm_src), _p(dest_row),
                                         _p(perm_w), _p(workspace), ws_bytes, _p(status),
                                         _s(stream))
    _check(rc, "minite_moe_permute_quant")


def minite_moe_permute_quant_noalloc(x, topk_ids, topk_w, E, codes, sf, row_g, expert_offsets,
                                     sf_row_offsets, perm_src, dest_row, perm_w, status=None,
                                     stream=None):
    """As minite_moe_permute_quant, with the library's built-in scratch array
    instead of a caller workspace (for callers that cannot allocate)."""
    T, H = x.shape
    k = topk_ids.shape[1]
    rc = load().minite_moe_permute_quant_noalloc(_p(x), _p(topk_ids), _p(topk_w), T, H, E, k,
                                                 _p(codes), _p(sf), _p(row_g), _p(expert_offsets),
                                                 _p(sf_row_offsets), _p(perm_src), _p(dest_row),
                                                 _p(perm_w), _p(status), _s(stream))
    _check(rc, "minite_moe_permute_quant_noalloc")


def minite_grouped_gemm_nvfp4(a_codes, a_sf, a_g, b_codes, b_sf, b_g, expert_offsets,
                              sf_row_offsets, out, status=None, stream=None):
    M, K2 = a_codes.shape
    E, N, _ = b_codes.shape
    out_dtype = OUT_FP32 if out.dtype == torch.float32 else OUT_BF16
    rc = load().minite_grouped_gemm_nvfp4(_p(a_codes), _p(a_sf), _p(a_g), _p(b_codes), _p(b_sf),
                                          _p(b_g), _p(expert_offsets), _p(sf_row_offsets), M, N,
                                          2 * K2, E, _p(out), out_dtype, _p(status), _s(stream))
    _check(rc, "minite_grouped_gemm_nvfp4")


def minite_gate_up_swiglu_quant_nvfp4(a_codes, a_sf, a_g, b_codes, b_sf, b_g, expert_offsets,
                                      sf_row_offsets, perm_w, h_codes, h_sf, h_g, workspace,
                                      gate_up=None, status=None, stream=None):
    """b_codes [E, 2I, K/2]; h_codes [M, I/2]; workspace uint8 of at least
    minite_workspace_bytes(OP_GATE_UP_SWIGLU, M, I, 0, 0) bytes."""
    M, K2 = a_codes.shape
    E, N, _ = b_codes.shape
    rc = load().minite_gate_up_swiglu_quant_nvfp4(
        _p(a_codes), _p(a_sf), _p(a_g), _p(b_codes), _p(b_sf), _p(b_g), _p(expert_offsets),
        _p(sf_row_offsets), M, N // 2, 2 * K2, E, _p(perm_w), _p(gate_up), _p(h_codes), _p(h_sf),
        _p(h_g), _p(workspace), workspace.numel() * workspace.element_size(), _p(status),
        _s(stream))
    _check(rc, "minite_gate_up_swiglu_quant_nvfp4")


def minite_swiglu_weighted_quant(gate_up, perm_w, E, expert_offsets, sf_row_offsets, codes, sf,
                                 row_g, status=None, stream=None):
    M, I2 = gate_up.shape
    rc = load().minite_swiglu_weighted_quant(_p(gate_up), _p(perm_w), M, I2 // 2, E,
                                             _p(expert_offsets), _p(sf_row_offsets), _p(codes),
                                             _p(sf), _p(row_g), _p(status), _s(stream))
    _check(rc, "minite_swiglu_weighted_quant")


def minite_swiglu_weighted_quant_keep_h(gate_up, perm_w, E, expert_offsets, sf_row_offsets, codes,
                                        sf, row_g, h_out, status=None, stream=None, h_amax=None):
    M, I2 = gate_up.shape
    rc = load().minite_swiglu_weighted_quant_keep_h(_p(gate_up), _p(perm_w), M, I2 // 2, E,
                                                    _p(expert_offsets), _p(sf_row_offsets),
                                                    _p(codes), _p(sf), _p(row_g), _p(h_out),
                                                    _p(h_amax), _p(status), _s(stream))
    _check(rc, "minite_swiglu_weighted_quant_keep_h")


def minite_swiglu_backward_quant(gate_up, dh, perm_w, E, expert_offsets, sf_row_offsets, codes,
                                 sf, row_g, status=None, stream=None):
    M, I2 = gate_up.shape
    rc = load().minite_swiglu_backward_quant(_p(gate_up), _p(dh), _p(perm_w), M, I2 // 2, E,
                                             _p(expert_offsets), _p(sf_row_offsets), _p(codes),
                                             _p(sf), _p(row_g), _p(status), _s(stream))
    _check(rc, "minite_swiglu_backward_quant")


def minite_swiglu_backward_quant_keep(gate_up, dh, perm_w, E, expert_offsets, sf_row_offsets,
                                      codes, sf, row_g, dgu_out, status=None, stream=None,
                                      dgu_amax=None):
    M, I2 = gate_up.shape
    rc = load().minite_swiglu_backward_quant_keep(_p(gate_up), _p(dh), _p(perm_w), M, I2 // 2, E,
                                                  _p(expert_offsets), _p(sf_row_offsets),
                                                  _p(codes), _p(sf), _p(row_g), _p(dgu_out),
                                                  _p(dgu_amax), _p(status), _s(stream))
    _check(rc, "minite_swiglu_backward_quant_keep")


def minite_moe_combine_backward_quant(dy, E, dest_row, expert_offsets, sf_row_offsets, perm_src,
                                      codes, sf, row_g, workspace, status=None, stream=None):
    T, H = dy.shape
    k = dest_row.shape[1]
    ws_bytes = workspace.numel() * workspace.element_size()
    rc = load().minite_moe_combine_backward_quant(_p(dy), T, H, E, k, _p(dest_row),
                                                  _p(expert_offsets), _p(sf_row_offsets),
                                                  _p(perm_src), _p(codes), _p(sf), _p(row_g),
                                                  _p(workspace), ws_bytes, _p(status), _s(stream))
    _check(rc, "minite_moe_combine_backward_quant")


def minite_quantize_tokens_nvfp4(x, row_src, m_cap, E, expert_offsets, k_cap, codes, sf, g, kofs,
                                 workspace, status=None, stream=None, row_amax=None):
    x_rows, C = x.shape
    ws_bytes = workspace.numel() * workspace.element_size()
    rc = load().minite_quantize_tokens_nvfp4(_p(x), x_rows, _p(row_src), _p(row_amax), m_cap, C, E,
                                             _p(expert_offsets), k_cap, _p(codes), _p(sf), _p(g),
                                             _p(kofs), _p(workspace), ws_bytes, _p(status),
                                             _s(stream))
    _check(rc, "minite_quantize_tokens_nvfp4")


def minite_grouped_gemm_wgrad_nvfp4(a, b, out, status=None, stream=None):
    """a, b: ``quantize_tokens`` results over the same routing; out [E, Ma, Nb]."""
    E, M, N = out.shape
    if a["k_cap"] != b["k_cap"]:
        raise MiniteError("minite_grouped_gemm_wgrad_nvfp4: operands with different token capacity")
    out_dtype = OUT_FP32 if out.dtype == torch.float32 else OUT_BF16
    rc = load().minite_grouped_gemm_wgrad_nvfp4(_p(a["codes"]), _p(a["sf"]), _p(a["g"]),
                                                _p(b["codes"]), _p(b["sf"]), _p(b["g"]),
                                                _p(a["kofs"]), E, M, N, a["k_cap"], _p(out),
                                                out_dtype, _p(status), _s(stream))
    _check(rc, "minite_grouped_gemm_wgrad_nvfp4")


def quantize_tokens(x, expert_offsets, E, row_src=None, m_cap=None, stream=None, row_amax=None):
    """Weight-gradient operand of x's permuted rows (x[row_src[m]] or x[m]):
    dict(codes [C, k_cap/2], sf, g [E], kofs [E+1], k_cap) with
    k_cap = m_cap + 256 E rounded up to 256. ``row_amax`` [x_rows]: each row's
    |x| maximum when the producer wrote it (x is then read once)."""
    dev = x.device
    x_rows, C = x.shape
    m_cap = (row_src.numel() if row_src is not None else x_rows) if m_cap is None else m_cap
    k_cap = (m_cap + 256 * E + 255) // 256 * 256
    out = dict(codes=torch.empty((C, k_cap // 2), dtype=torch.uint8, device=dev),
               sf=torch.empty(((C + 127) // 128 * 128) * (k_cap // 16), dtype=torch.uint8, device=dev),
               g=torch.empty(E, dtype=torch.float32, device=dev),
               kofs=torch.empty(E + 1, dtype=torch.int32, device=dev), k_cap=k_cap)
    gathered = row_src is not None and row_amax is None
    ws = torch.empty(max(4, minite_workspace_bytes(OP_QUANTIZE_TOKENS, E, x_rows if gathered else 0)),
                     dtype=torch.uint8, device=dev)
    minite_quantize_tokens_nvfp4(x, row_src, m_cap, E, expert_offsets, k_cap, out["codes"],
                                 out["sf"], out["g"], out["kofs"], ws, stream=stream,
                                 row_amax=row_amax)
    return out


def minite_moe_combine(expert_out, dest_row, y, status=None, stream=None):
    M, N = expert_out.shape
    T, k = dest_row.shape
    rc = load().minite_moe_combine(_p(expert_out), _p(dest_row), T, M, N, k, _p(y), _p(status),
                                   _s(stream))
    _check(rc, "minite_moe_combine")


def minite_test_convert(x, out_e2m1=None, out_e4m3=None, out_exp=None, stream=None):
    rc = load().minite_test_convert(_p(x), x.numel(), _p(out_e2m1), _p(out_e4m3), _p(out_exp),
                                    _s(stream))
    _check(rc, "minite_test_convert")


def minite_test_convert_digest(first_chunk, n_chunks, digests, stream=None):
    """Adds the device converters' digests of chunks [first_chunk, first_chunk
    + n_chunks) of 2^20 float32 bit patterns into digests (int64 [n_chunks, 3])."""
    rc = load().minite_test_convert_digest(first_chunk, n_chunks, _p(digests), _s(stream))
    _check(rc, "minite_test_convert_digest")


def minite_test_div6_exhaustive(counter, stream=None):
    rc = load().minite_test_div6_exhaustive(_p(counter), _s(stream))
    _check(rc, "minite_test_div6_exhaustive")


# ---------------------------------------------------------------- allocation helpers


def _kc(cols: int) -> int:
    return ((cols // 16) + 3) // 4 * 4


def sf_bytes(rows_padded: int, cols: int) -> int:
    return rows_padded * _kc(cols)


def quantize(x, per_group=False, along_rows=False, g_in=None, stream=None):
    """Quantize bf16 x ([rows, cols] or [groups, rows, cols]); returns dict(codes, sf, g)."""
    dev = x.device
    g3 = x if x.dim() == 3 else x.unsqueeze(0)
    G, R, C = g3.shape
    Rq, Cq = (C, R) if along_rows else (R, C)
    codes = torch.empty((G, Rq, Cq // 2), dtype=torch.uint8, device=dev)
    sf = torch.empty((G, sf_bytes((Rq + 127) // 128 * 128, Cq)), dtype=torch.uint8, device=dev)
    g = torch.empty((G,) if per_group else (G * Rq,), dtype=torch.float32, device=dev)
    ws = None
    if per_group and g_in is None:
        ws = torch.empty(minite_workspace_bytes(OP_QUANTIZE, G), dtype=torch.uint8, device=dev)
    minite_quantize_nvfp4(g3, SCALE_PER_GROUP if per_group else SCALE_PER_ROW,
                          ALONG_ROWS if along_rows else ALONG_COLS, codes, sf, g, g_in, ws,
                          stream=stream)
    if x.dim() == 2:
        codes, sf = codes[0], sf[0]
    return dict(codes=codes, sf=sf, g=g)


class MoEMLP:
    """Preallocated device buffers for the expert-MLP forward of one shape
    (T tokens, hidden H, intermediate I, E experts, top-k), so that a step
    allocates nothing and can be captured in a CUDA graph."""

    def __init__(self, T, H, I, E, k, device="cuda"):
        self.T, self.H, self.I, self.E, self.k = T, H, I, E, k
        M = T * k
        self.M = M
        d = torch.device(device)
        u8, f32, i32 = torch.uint8, torch.float32, torch.int32
        sf_rows = M + 128 * E
        self.a_codes = torch.empty((M, H // 2), dtype=u8, device=d)
        self.a_sf = torch.empty(sf_bytes(sf_rows, H), dtype=u8, device=d)
        self.a_g = torch.empty(M, dtype=f32, device=d)
        self.offsets = torch.empty(E + 1, dtype=i32, device=d)
        self.sf_offsets = torch.empty(E + 1, dtype=i32, device=d)
        self.perm_src = torch.empty(M, dtype=i32, device=d)
        self.dest_row = torch.empty((T, k), dtype=i32, device=d)
        self.perm_w = torch.empty(M, dtype=f32, device=d)
        self.ws = torch.empty(minite_workspace_bytes(OP_PERMUTE_QUANT, T, H, E, k), dtype=u8, device=d)
        self.gate_up = torch.empty((M, 2 * I), dtype=torch.bfloat16, device=d)
        self.h_codes = torch.empty((M, I // 2), dtype=u8, device=d)
        self.h_sf = torch.empty(sf_bytes(sf_rows, I), dtype=u8, device=d)
        self.h_g = torch.empty(M, dtype=f32, device=d)
        self.down = torch.empty((M, H), dtype=torch.bfloat16, device=d)
        self.y = torch.empty((T, H), dtype=torch.bfloat16, device=d)
        self.status = torch.zeros(1, dtype=i32, device=d)
        # the fused gate_up + SwiGLU kernel takes I % 128 == 0 and E <= 663
        self.fused_ok = I % 128 == 0 and 128 <= I <= 8192 and E <= 663
        self.sw_ws = torch.empty(max(16, minite_workspace_bytes(OP_GATE_UP_SWIGLU, M, I, 0, 0)),
                                 dtype=u8, device=d) if self.fused_ok else None

    def permute_quant(self, x, topk_ids, topk_w, stream=None):
        minite_moe_permute_quant(x, topk_ids, topk_w, self.E, self.a_codes, self.a_sf, self.a_g,
                                 self.offsets, self.sf_offsets, self.perm_src, self.dest_row,
                                 None if topk_w is None else self.perm_w, self.ws, self.status,
                                 stream)

    def gate_up_swiglu(self, wgu, stream=None, fused=True, keep_gate_up=False):
        """h = weighted SwiGLU of the gate_up GEMM, quantized into h_codes /
        h_sf / h_g: one fused launch (the BF16 gate_up stored only with
        keep_gate_up), or the GEMM into gate_up followed by the SwiGLU."""
        if fused:
            if not self.fused_ok:
                raise MiniteError("the fused gate_up + SwiGLU kernel needs I % 128 == 0, E <= 663")
            minite_gate_up_swiglu_quant_nvfp4(
                self.a_codes, self.a_sf, self.a_g, wgu["codes"], wgu["sf"], wgu["g"],
                self.offsets, self.sf_offsets, self.perm_w, self.h_codes, self.h_sf, self.h_g,
                self.sw_ws, gate_up=self.gate_up if keep_gate_up else None, status=self.status,
                stream=stream)
            return
        minite_grouped_gemm_nvfp4(self.a_codes, self.a_sf, self.a_g, wgu["codes"], wgu["sf"],
                                  wgu["g"], self.offsets, self.sf_offsets, self.gate_up,
                                  self.status, stream)
        minite_swiglu_weighted_quant(self.gate_up, self.perm_w, self.E, self.offsets,
                                     self.sf_offsets, self.h_codes, self.h_sf, self.h_g,
                                     self.status, stream)

    def forward(self, x, topk_ids, topk_w, wgu, wd, stream=None, fused=False, keep_gate_up=True):
        """x [T,H] bf16, topk_ids [T,k] int32, topk_w [T,k] f32; wgu / wd are
        ``quantize(..., per_group=True)`` results of [E,2I,H] and [E,H,I].
        fused: gate_up GEMM, SwiGLU and requantization in one launch."""
        self.permute_quant(x, topk_ids, topk_w, stream)
        self.gate_up_swiglu(wgu, stream, fused=fused, keep_gate_up=keep_gate_up)
        minite_grouped_gemm_nvfp4(self.h_codes, self.h_sf, self.h_g, wd["codes"], wd["sf"],
                                  wd["g"], self.offsets, self.sf_offsets, self.down, self.status,
                                  stream)
        minite_moe_combine(self.down, self.dest_row, self.y, self.status, stream)
        return self.y
