"""Stage-by-stage checks of the expert-MLP forward on sampled tokens, shared
by the GPU tests (the oracle's values go in, the GPU's full-size launches
are checked)."""
import numpy as np
import torch

from _helpers import assert_bf16_within_one_ulp, bf16_dev, u16
from nvfp4_w4a4_moe_permute_gb300 import minite as M
from oracle import nvfp4_moe_oracle as O


def idx(rows):
    return torch.from_numpy(np.ascontiguousarray(rows, dtype=np.int64)).cuda()


def take(t, rows):
    return t.index_select(0, idx(rows))


def _sf_positions(off, sfo, rows, C):
    """Byte offsets, in a per-expert padded scale region, of the scales of
    permuted rows `rows` (one row of C / 16 positions per row)."""
    kc = O.roundup(C // 16, 4)
    e = O.row_experts(off, rows)
    padded_row = np.asarray(sfo, dtype=np.int64)[e] + (rows - np.asarray(off, dtype=np.int64)[e])
    return O.sf_swizzle_offset(padded_row[:, None], np.arange(C // 16)[None, :], kc)


def _assert_rows_codes(codes_dev, g_dev, sf_dev, rows, off, sfo, C, ref_codes, ref_sf, ref_g, what):
    assert np.array_equal(take(codes_dev, rows).cpu().numpy(), ref_codes), f"{what} codes"
    assert np.array_equal(take(g_dev, rows).cpu().numpy().view(np.uint32),
                          np.asarray(ref_g, dtype=np.float32).view(np.uint32)), f"{what} g"
    pos = _sf_positions(off, sfo, rows, C)
    got = take(sf_dev, pos.ravel()).cpu().numpy().reshape(pos.shape)
    assert np.array_equal(got, ref_sf), f"{what} scales"


def check_forward_stagewise(d, tok, wq, mlp, wgu, wd, status):
    """`mlp` holds one forward over the whole batch of `d`, with weights
    `wgu` / `wd` (device) and status `status`. Checks the sampled tokens
    `tok` stage by stage, relaunching the SwiGLU, the down GEMM and the
    combine at full size with the oracle's inputs in the sampled rows."""
    c = d["cfg"]
    T, H, E, I = c["T"], c["H"], c["E"], c["I"]
    full = O.moe_permute(d["topk_ids"], E)
    off, sfo = full["expert_offsets"], full["sf_row_offsets"]
    Mu = int(off[-1])
    # routing metadata of the whole batch
    assert np.array_equal(mlp.offsets.cpu().numpy(), off)
    assert np.array_equal(mlp.sf_offsets.cpu().numpy(), sfo)
    assert np.array_equal(mlp.dest_row.cpu().numpy(), full["dest_row"])
    assert np.array_equal(mlp.perm_src.cpu().numpy()[:Mu], full["perm_src"])

    ref = O.moe_mlp_forward(d["x"][tok], d["topk_ids"][tok], d["topk_w"][tok], E, *wq)
    p = ref["permute"]
    mini = p["dest_row"].ravel()                            # oracle rows, (token, slot) order
    rows = full["dest_row"][tok].ravel()                    # the same pairs in the full batch
    assert (mini >= 0).all() and (rows >= 0).all()

    # permutation + quantization of the sampled rows
    _assert_rows_codes(mlp.a_codes, mlp.a_g, mlp.a_sf, rows, off, sfo, H, p["codes"][mini],
                       p["sf"][mini], p["row_g"][mini], "permuted x")
    assert np.array_equal(take(mlp.perm_w, rows).cpu().numpy().view(np.uint32),
                          p["perm_w"][mini].view(np.uint32))

    # gate_up GEMM rows (from the GPU's own permuted operand, equal to the oracle's above)
    gu_exact, _ = O.grouped_gemm_exact(p["codes"], p["sf"], p["row_g"], wq[0][0], wq[0][1],
                                       wq[0][3], p["expert_offsets"], rows=mini)
    assert_bf16_within_one_ulp(u16(take(mlp.gate_up, rows)), gu_exact, "gate_up rows")

    # SwiGLU + requant: the oracle's BF16 gate_up in the sampled rows, full-size launch
    sw = ref["swiglu"]
    mlp.gate_up.index_copy_(0, idx(rows), bf16_dev(ref["gate_up"][mini]))
    M.minite_swiglu_weighted_quant(mlp.gate_up, mlp.perm_w, E, mlp.offsets, mlp.sf_offsets,
                                   mlp.h_codes, mlp.h_sf, mlp.h_g, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    _assert_rows_codes(mlp.h_codes, mlp.h_g, mlp.h_sf, rows, off, sfo, I, sw["codes"][mini],
                       sw["sf"][mini], sw["row_g"][mini], "SwiGLU")

    # down GEMM rows: the GPU's h operand of the sampled rows now equals the oracle's
    M.minite_grouped_gemm_nvfp4(mlp.h_codes, mlp.h_sf, mlp.h_g, wd["codes"], wd["sf"], wd["g"],
                                mlp.offsets, mlp.sf_offsets, mlp.down, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    d_exact, _ = O.grouped_gemm_exact(sw["codes"], sw["sf"], sw["row_g"], wq[1][0], wq[1][1],
                                      wq[1][3], p["expert_offsets"], rows=mini)
    assert_bf16_within_one_ulp(u16(take(mlp.down, rows)), d_exact, "down rows")

    # combine: the oracle's BF16 down rows of the sampled tokens, full-size launch
    mlp.down.index_copy_(0, idx(rows), bf16_dev(ref["down"][mini]))
    M.minite_moe_combine(mlp.down, mlp.dest_row, mlp.y, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(u16(take(mlp.y, tok)), ref["y"]), "combined y"
    return full
