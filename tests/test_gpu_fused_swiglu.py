"""The fused gate_up GEMM + weighted SwiGLU + NVFP4 requantization
(minite_gate_up_swiglu_quant_nvfp4).

Two bars, both element by element:
  * against the oracle: the BF16 gate_up the fused call keeps is within one
    BF16 ulp of the exact product, and every row whose kept gate_up equals
    the oracle's correctly rounded product (nearly all rows) has codes,
    scales and global scale bit-exact with the oracle's SwiGLU quantization
    of that product (a row where the tensor cores' FP32 sum rounds the other
    way quantizes a different input, so it is not held to the oracle's codes);
  * against the unfused composition on the GPU (minite_grouped_gemm_nvfp4
    into BF16, then minite_swiglu_weighted_quant): the whole code buffer, the
    whole scale buffer (padding rows included, sentinel bytes outside the
    written rows left alone) and the global scales bit-identical.

Expert sizes include 0, 1, 127, 128, 129, 255, 256 and 257 rows, and I takes
values whose tile count per 256-row block (I / 128 = 1, 3, 6) divides the
cluster count or not.
"""
import numpy as np
import pytest
import torch

from _helpers import assert_bf16_within_one_ulp, bf16_dev, np_dev, u16
from nvfp4_w4a4_moe_permute_gb300 import inputs as IN
from nvfp4_w4a4_moe_permute_gb300 import minite as M
from oracle import nvfp4_moe_oracle as O

pytestmark = pytest.mark.gpu

SENTINEL = 0xA5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from nvfp4_w4a4_moe_permute_gb300 import build
    build.build()
    M.load()
    M.minite_set_wait_budget_ns(0)
    M.minite_set_gemm_variant(0)
    yield
    M.minite_set_wait_budget_ns(0)


def routing_with_counts(counts, T, k, rng):
    """topk_ids [T, k] whose expert loads are `counts` (each <= T, sum T*k),
    every token's k experts distinct: the experts' slots, listed expert by
    expert, fill slot 0 of every token, then slot 1, ...; list positions t
    and t + T (same token) are T apart, so they name different experts."""
    counts = np.asarray(counts, dtype=np.int64)
    assert counts.sum() == T * k and counts.max() <= T
    flat = np.repeat(np.arange(len(counts), dtype=np.int32), counts)
    ids = flat.reshape(k, T).T.copy()
    ids = ids[rng.permutation(T)]
    w = rng.random((T, k), dtype=np.float32) + np.float32(0.05)
    w = (w / w.sum(axis=1, keepdims=True)).astype(np.float32)
    return ids, w


def make_case(T, H, I, counts, k, seed):
    rng = np.random.default_rng(seed)
    ids, w = routing_with_counts(counts, T, k, rng)
    E = len(counts)
    return dict(cfg=dict(T=T, H=H, I=I, E=E, k=k), topk_ids=ids, topk_w=w,
                x=IN.f32_to_bf16_bits(rng.standard_normal((T, H), dtype=np.float32)),
                w_gate_up=IN.f32_to_bf16_bits(
                    rng.standard_normal((E, 2 * I, H), dtype=np.float32) * np.float32(0.02)))


def _run_both(d, with_w=True, keep_gate_up=True):
    """Permute once, then the unfused composition and the fused call into
    separate sentinel-filled buffers. Returns (mlp, unfused, fused, wgu)."""
    c = d["cfg"]
    T, H, I, E, k = c["T"], c["H"], c["I"], c["E"], c["k"]
    wgu = M.quantize(bf16_dev(d["w_gate_up"]), per_group=True)
    mlp = M.MoEMLP(T, H, I, E, k)
    mlp.permute_quant(bf16_dev(d["x"]), np_dev(d["topk_ids"]),
                      np_dev(d["topk_w"]) if with_w else None)
    perm_w = mlp.perm_w if with_w else None

    def bufs():
        return dict(codes=torch.full_like(mlp.h_codes, SENTINEL),
                    sf=torch.full_like(mlp.h_sf, SENTINEL),
                    g=torch.full_like(mlp.h_g, float("nan")),
                    gate_up=torch.full_like(mlp.gate_up, float("nan")))

    un, fu = bufs(), bufs()
    M.minite_grouped_gemm_nvfp4(mlp.a_codes, mlp.a_sf, mlp.a_g, wgu["codes"], wgu["sf"], wgu["g"],
                                mlp.offsets, mlp.sf_offsets, un["gate_up"], mlp.status)
    M.minite_swiglu_weighted_quant(un["gate_up"], perm_w, E, mlp.offsets, mlp.sf_offsets,
                                   un["codes"], un["sf"], un["g"], mlp.status)
    M.minite_gate_up_swiglu_quant_nvfp4(mlp.a_codes, mlp.a_sf, mlp.a_g, wgu["codes"], wgu["sf"],
                                        wgu["g"], mlp.offsets, mlp.sf_offsets, perm_w, fu["codes"],
                                        fu["sf"], fu["g"], mlp.sw_ws,
                                        gate_up=fu["gate_up"] if keep_gate_up else None,
                                        status=mlp.status)
    torch.cuda.synchronize()
    assert int(mlp.status.item()) == 0
    return mlp, un, fu, wgu


def _assert_identical(un, fu, Mu, gate_up=True):
    assert torch.equal(fu["codes"], un["codes"]), "h codes (whole buffer)"
    assert torch.equal(fu["sf"], un["sf"]), "h scales (whole buffer)"
    assert np.array_equal(fu["g"][:Mu].cpu().numpy().view(np.uint32),
                          un["g"][:Mu].cpu().numpy().view(np.uint32)), "h global scales"
    if gate_up:
        assert np.array_equal(u16(fu["gate_up"][:Mu]), u16(un["gate_up"][:Mu])), "gate_up"


def _oracle_rows(d, fu, off, sfo, rows, with_w=True):
    """Oracle parity of the fused outputs on permuted rows `rows` of the
    whole batch (oracle permutation of all tokens)."""
    c = d["cfg"]
    E, I = c["E"], c["I"]
    pq = O.moe_permute_quant(d["x"], d["topk_ids"], d["topk_w"] if with_w else None, E)
    assert np.array_equal(pq["expert_offsets"], off)
    wq = O.quantize_weights(d["w_gate_up"])
    gu, _ = O.grouped_gemm_exact(pq["codes"], pq["sf"], pq["row_g"], wq[0], wq[1], wq[3],
                                 pq["expert_offsets"], rows=rows)
    got_gu = u16(fu["gate_up"].index_select(0, torch.from_numpy(rows).cuda()))
    assert_bf16_within_one_ulp(got_gu, gu, "fused gate_up rows")
    gu_bf16 = O.f64_to_bf16(gu)
    same = (got_gu == gu_bf16).all(axis=1)
    # rows whose FP32 tensor-core sum rounds to another BF16 somewhere are rare
    assert same.mean() > 0.9, f"only {same.mean():.3f} of rows with the oracle's gate_up"
    rs = rows[same]
    # the oracle's SwiGLU + quantization of its own gate_up, for those rows
    w = pq["perm_w"] if with_w else None
    sw = O.swiglu_weighted(O.bf16_to_f32(gu_bf16[same]), None if w is None else w[rs])
    codes, sf, g = O.quantize_per_row(sw)
    ridx = torch.from_numpy(rs).cuda()
    assert np.array_equal(fu["codes"].index_select(0, ridx).cpu().numpy(), codes), "codes"
    assert np.array_equal(fu["g"].index_select(0, ridx).cpu().numpy().view(np.uint32),
                          np.asarray(g, dtype=np.float32).view(np.uint32)), "global scales"
    kc = O.roundup(I // 16, 4)
    e = O.row_experts(off, rs)
    prow = np.asarray(sfo, dtype=np.int64)[e] + (rs - np.asarray(off, dtype=np.int64)[e])
    pos = O.sf_swizzle_offset(prow[:, None], np.arange(I // 16)[None, :], kc)
    got_sf = fu["sf"].index_select(0, torch.from_numpy(pos.ravel()).cuda()).cpu().numpy()
    assert np.array_equal(got_sf.reshape(pos.shape), sf), "scales"
    return int(same.sum())


RAGGED = [0, 1, 127, 128, 129, 255, 256, 257, 384, 0, 510, 513]   # 12 experts, 2560 rows
T_RAGGED = sum(RAGGED) // 2


@pytest.mark.parametrize("I", [128, 384, 768])
@pytest.mark.parametrize("with_w", [True, False])
def test_fused_ragged_experts_match_oracle_and_unfused(I, with_w):
    counts = RAGGED
    d = make_case(T_RAGGED, 256, I, counts, 2, seed=100 + I)
    mlp, un, fu, _ = _run_both(d, with_w)
    off = mlp.offsets.cpu().numpy()
    sfo = mlp.sf_offsets.cpu().numpy()
    Mu = int(off[-1])
    assert np.array_equal(np.diff(off), counts)
    _assert_identical(un, fu, Mu)
    n = _oracle_rows(d, fu, off, sfo, np.arange(Mu), with_w)
    assert n > 0


def test_fused_extreme_rows_match_oracle_and_unfused():
    """Tokens of zeros (every gate 0), tokens scaled by 2^12 (gates far
    beyond 2^8) and by 2^-14 (gates below 2^-16) next to ordinary ones: the
    SiLU of such gates is evaluated by the formula, not read from a table."""
    d = make_case(T_RAGGED, 256, 384, RAGGED, 2, seed=21)
    x = IN.bf16_bits_to_f32(d["x"]).copy()
    rng = np.random.default_rng(22)
    tok = rng.permutation(x.shape[0])
    x[tok[:40]] = 0.0
    x[tok[40:80]] *= np.float32(2.0 ** 12)
    x[tok[80:120]] *= np.float32(2.0 ** -14)
    d["x"] = IN.f32_to_bf16_bits(x)
    mlp, un, fu, _ = _run_both(d, True)
    off = mlp.offsets.cpu().numpy()
    sfo = mlp.sf_offsets.cpu().numpy()
    Mu = int(off[-1])
    _assert_identical(un, fu, Mu)
    _oracle_rows(d, fu, off, sfo, np.arange(Mu), True)


def test_fused_without_kept_gate_up_is_identical():
    d = make_case(T_RAGGED, 512, 384, RAGGED, 2, seed=7)
    mlp, un, fu, _ = _run_both(d, True, keep_gate_up=False)
    Mu = int(mlp.offsets[-1].item())
    _assert_identical(un, fu, Mu, gate_up=False)
    # gate_up was not requested: its sentinel is untouched
    assert torch.isnan(fu["gate_up"].float()).all()


def test_fused_repeat_and_graph_replay_are_identical():
    """The workspace is cleared by every call: a second call, and replays of
    a captured call, give the same bytes."""
    d = make_case(T_RAGGED, 256, 768, RAGGED, 2, seed=9)
    mlp, un, fu, wgu = _run_both(d, True)
    Mu = int(mlp.offsets[-1].item())
    first = {k: v.clone() for k, v in fu.items()}
    for key in ("codes", "sf"):
        fu[key].fill_(SENTINEL)

    def call():
        M.minite_gate_up_swiglu_quant_nvfp4(mlp.a_codes, mlp.a_sf, mlp.a_g, wgu["codes"],
                                            wgu["sf"], wgu["g"], mlp.offsets, mlp.sf_offsets,
                                            mlp.perm_w, fu["codes"], fu["sf"], fu["g"], mlp.sw_ws,
                                            gate_up=fu["gate_up"], status=mlp.status)

    call()
    torch.cuda.synchronize()
    _assert_identical(first, fu, Mu)
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        call()
    for _ in range(3):
        for key in ("codes", "sf"):
            fu[key].fill_(SENTINEL)
        graph.replay()
        torch.cuda.synchronize()
        assert int(mlp.status.item()) == 0
        _assert_identical(first, fu, Mu)


@pytest.mark.parametrize("name", ["mlp", "skewed"])
def test_fused_full_size_identical_to_unfused_and_oracle_rows(name):
    """Qwen3-30B-A3B expert MLP (4096 tokens) and the skewed 32768-token
    layer: every row identical to the unfused composition; 256 sampled
    permuted rows plus every row of the smallest and largest non-empty
    expert against the oracle."""
    d = IN.make_moe_inputs(name)
    d.pop("w_down", None)
    d.pop("dy", None)
    mlp, un, fu, _ = _run_both(d, True)
    off = mlp.offsets.cpu().numpy()
    sfo = mlp.sf_offsets.cpu().numpy()
    Mu = int(off[-1])
    _assert_identical(un, fu, Mu)
    counts = np.diff(off)
    nz = np.nonzero(counts)[0]
    e_small, e_large = nz[np.argmin(counts[nz])], nz[np.argmax(counts[nz])]
    rng = np.random.default_rng(13)
    rows = np.unique(np.concatenate([rng.choice(Mu, 256, replace=False),
                                     np.arange(off[e_small], off[e_small + 1]),
                                     np.arange(off[e_large], min(off[e_large + 1],
                                                                 off[e_large] + 512)),
                                     [0, Mu - 1]]))
    _oracle_rows(d, fu, off, sfo, rows.astype(np.int64))


def test_plain_and_fused_gemm_repeat_bit_identical_full_size():
    """Races in a pipeline show up as run-to-run differences: three launches
    of the gate_up GEMM and of the fused kernel on the 4096-token layer give
    the same bytes each time."""
    d = IN.make_moe_inputs("mlp")
    d.pop("w_down", None)
    c = d["cfg"]
    T, H, I, E, k = c["T"], c["H"], c["I"], c["E"], c["k"]
    wgu = M.quantize(bf16_dev(d["w_gate_up"]), per_group=True)
    mlp = M.MoEMLP(T, H, I, E, k)
    mlp.permute_quant(bf16_dev(d["x"]), np_dev(d["topk_ids"]), np_dev(d["topk_w"]))
    Mu = int(mlp.offsets[-1].item())
    plain, fused = [], []
    for _ in range(3):
        M.minite_grouped_gemm_nvfp4(mlp.a_codes, mlp.a_sf, mlp.a_g, wgu["codes"], wgu["sf"],
                                    wgu["g"], mlp.offsets, mlp.sf_offsets, mlp.gate_up, mlp.status)
        torch.cuda.synchronize()
        plain.append(mlp.gate_up[:Mu].clone())
        mlp.gate_up_swiglu(wgu, fused=True, keep_gate_up=True)
        torch.cuda.synchronize()
        fused.append((mlp.gate_up[:Mu].clone(), mlp.h_codes[:Mu].clone(), mlp.h_g[:Mu].clone()))
    assert int(mlp.status.item()) == 0
    for i in (1, 2):
        assert torch.equal(plain[i], plain[0]), "plain GEMM differs between launches"
        for a, b in zip(fused[i], fused[0]):
            assert torch.equal(a, b), "fused kernel differs between launches"
    assert torch.equal(fused[0][0], plain[0]), "fused gate_up differs from the plain GEMM"


def test_fused_rejects_unsupported_shapes():
    d = make_case(64, 256, 192, [64, 64], 2, seed=3)   # I % 128 != 0
    c = d["cfg"]
    mlp = M.MoEMLP(c["T"], c["H"], c["I"], c["E"], c["k"])
    assert not mlp.fused_ok
    wgu = M.quantize(bf16_dev(d["w_gate_up"]), per_group=True)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    with pytest.raises(M.MiniteError):
        M.minite_gate_up_swiglu_quant_nvfp4(mlp.a_codes, mlp.a_sf, mlp.a_g, wgu["codes"], wgu["sf"],
                                            wgu["g"], mlp.offsets, mlp.sf_offsets, None,
                                            mlp.h_codes, mlp.h_sf, mlp.h_g, ws, status=mlp.status)


def test_fused_wait_timeout_sets_status_and_context_survives():
    """Every wait of the fused kernel (pipeline barriers and the row-maximum
    exchange) runs out under a 1 ns budget: the call sets the timeout bit and
    returns, and the next call on the same context gives the right bytes."""
    d = make_case(T_RAGGED, 256, 384, RAGGED, 2, seed=31)
    mlp, un, fu, wgu = _run_both(d, True)
    Mu = int(mlp.offsets[-1].item())
    st = torch.zeros(1, dtype=torch.int32, device="cuda")

    def call():
        M.minite_gate_up_swiglu_quant_nvfp4(mlp.a_codes, mlp.a_sf, mlp.a_g, wgu["codes"],
                                            wgu["sf"], wgu["g"], mlp.offsets, mlp.sf_offsets,
                                            mlp.perm_w, fu["codes"], fu["sf"], fu["g"], mlp.sw_ws,
                                            gate_up=fu["gate_up"], status=st)

    try:
        M.minite_set_wait_budget_ns(1)
        call()
        torch.cuda.synchronize()
    finally:
        M.minite_set_wait_budget_ns(0)
    assert int(st.item()) & (1 << M.ERR_TIMEOUT)
    st.zero_()
    for key in ("codes", "sf"):
        fu[key].fill_(SENTINEL)
    call()
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    _assert_identical(un, fu, Mu)
