"""Parity of the CUDA path (called through the C ABI) with the CPU oracle.

Integer, code, scale and index outputs must match bit for bit. Grouped-GEMM
outputs: FP32 within 2^-20 * sum_k |a_k b_k| of the exact result, BF16
within one BF16 ulp of the correctly rounded exact result. Comparisons of
permuted rows are keyed by (token, slot) through the permutation itself,
which is compared exactly first.
"""
import numpy as np
import pytest
import torch

from _helpers import (assert_bf16_within_one_ulp, assert_fp32_within_bound, bf16_dev,
                      np_dev, u16)
from _stagewise import check_forward_stagewise
from nvfp4_w4a4_moe_permute_gb300 import inputs as IN
from nvfp4_w4a4_moe_permute_gb300 import minite as M
from oracle import nvfp4_moe_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from nvfp4_w4a4_moe_permute_gb300 import build
    build.build()
    M.load()
    M.minite_set_wait_budget_ns(0)
    yield


@pytest.fixture(autouse=True)
def _automatic_gemm_variant():
    yield
    M.minite_set_gemm_variant(0)


VARIANTS = [1, 5, 6]  # single-CTA one- and two-chunk stages, deep-pipeline CTA pair


def _status():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def _rand_bf16(rng, shape, scale_spread=6):
    x = rng.standard_normal(shape).astype(np.float32)
    if len(shape) >= 2:
        x *= np.exp2(rng.integers(-scale_spread, scale_spread + 1, shape[:-1] + (1,))).astype(np.float32)
    return O.f32_to_bf16(x)


# --------------------------------------------------------------------- converters

def _sweep_bits():
    parts = [np.arange(0, 2 ** 32, 257, dtype=np.uint64).astype(np.uint32)]
    # every float32 within +-1024 ulps of each E2M1 midpoint and grid value,
    # and of each E4M3 midpoint and value
    vals = O.e4m3_decode(np.arange(127, dtype=np.uint8)).astype(np.float64)
    pts = np.concatenate([O.E2M1_MAGNITUDES, (O.E2M1_MAGNITUDES[1:] + O.E2M1_MAGNITUDES[:-1]) / 2,
                          vals, (vals[1:] + vals[:-1]) / 2, [448.0, 464.0, 480.0]])
    base = pts.astype(np.float32).view(np.uint32).astype(np.int64)
    near = (base[:, None] + np.arange(-1024, 1025)[None, :]).ravel()
    near = near[(near >= 0) & (near < 2 ** 31)].astype(np.uint32)
    parts.append(near)
    parts.append(near | np.uint32(0x80000000))
    b = np.concatenate(parts)
    f = b.view(np.float32)
    return f[np.isfinite(f)]


def test_converters_bit_exact_over_float32_sweep():
    v = _sweep_bits()
    for lo in range(0, v.size, 1 << 23):
        c = v[lo:lo + (1 << 23)]
        x = np_dev(c)
        e2 = torch.empty(c.size, dtype=torch.uint8, device="cuda")
        e4 = torch.empty(c.size, dtype=torch.uint8, device="cuda")
        ex = torch.empty(c.size, dtype=torch.float32, device="cuda")
        M.minite_test_convert(x, e2, e4, ex)
        torch.cuda.synchronize()
        assert np.array_equal(e2.cpu().numpy(), O.e2m1_rn(c)), "E2M1"
        pos = (c > 0) | ((c == 0) & ~np.signbit(c))  # scales are never -0
        assert np.array_equal(e4.cpu().numpy()[pos], O.e4m3_rn_satfinite(c[pos])), "E4M3"
        got = ex.cpu().numpy().view(np.uint32)
        assert np.array_equal(got, O.exp_spec(c).view(np.uint32)), "exp_spec"


def test_converters_bit_exact_over_every_float32():
    """Every finite float32 input: the kernels' E2M1 and E4M3 converters and
    the specified exponential against the oracle's. The device reduces its
    results per chunk of 2^20 bit patterns to digests; the oracle's digests
    come from a pool of host processes (spawned) over the same chunks. A
    differing chunk is then compared element by element to name the input."""
    import multiprocessing as mp
    import os
    import _digest as DG
    n_chunks = 1 << (32 - DG.CHUNK_BITS)
    dev = torch.zeros((n_chunks, 3), dtype=torch.int64, device="cuda")
    M.minite_test_convert_digest(0, n_chunks, dev)
    procs = max(1, min(os.cpu_count() or 1, 64))
    parts = [list(range(i, n_chunks, procs)) for i in range(procs)]
    with mp.get_context("spawn").Pool(procs) as pool:
        res = pool.map(DG.chunk_digests, parts)
    host = np.zeros((n_chunks, 3), dtype=np.uint64)
    for part, r in zip(parts, res):
        host[part] = np.array(r, dtype=np.uint64)
    got = dev.cpu().numpy().view(np.uint64)
    bad = np.nonzero((got != host).any(axis=1))[0]
    if bad.size:
        c = int(bad[0])
        b = np.arange(c << DG.CHUNK_BITS, (c + 1) << DG.CHUNK_BITS, dtype=np.uint64).astype(np.uint32)
        f = b.view(np.float32)
        f = f[np.isfinite(f)]
        e2 = torch.empty(f.size, dtype=torch.uint8, device="cuda")
        e4 = torch.empty(f.size, dtype=torch.uint8, device="cuda")
        ex = torch.empty(f.size, dtype=torch.float32, device="cuda")
        M.minite_test_convert(np_dev(f), e2, e4, ex)
        torch.cuda.synchronize()
        pos = (f > 0) | ((f == 0) & ~np.signbit(f))
        d2 = np.nonzero(e2.cpu().numpy() != O.e2m1_rn(f))[0]
        d4 = np.nonzero(e4.cpu().numpy()[pos] != O.e4m3_rn_satfinite(f[pos]))[0]
        dx = np.nonzero(ex.cpu().numpy().view(np.uint32) != O.exp_spec(f).view(np.uint32))[0]
        pytest.fail(f"{bad.size} chunks differ; chunk {c}: e2m1 at {f[d2[:3]]}, "
                    f"e4m3 at {f[pos][d4[:3]]}, exp at {f[dx[:3]]}")


def test_division_by_six_is_exact_for_every_nonnegative_float():
    counter = torch.zeros(1, dtype=torch.int64, device="cuda")
    M.minite_test_div6_exhaustive(counter)
    torch.cuda.synchronize()
    assert int(counter.item()) == 0


# --------------------------------------------------------------------- quantize

@pytest.mark.parametrize("rows,cols", [(1, 16), (3, 48), (37, 80), (128, 256), (130, 2048),
                                       (200, 4096), (64, 1536), (129, 768)])
def test_quantize_per_row_bit_exact(rows, cols):
    rng = np.random.default_rng(rows * 7 + cols)
    x = _rand_bf16(rng, (rows, cols))
    x[0, :] = 0  # zero row
    if rows > 2:
        x[1, :] = O.f32_to_bf16(np.full(cols, 1e-40, dtype=np.float32))  # subnormal row
        x[2, 5] = O.f32_to_bf16(np.array([3.0e38], dtype=np.float32))[0]
    q = M.quantize(bf16_dev(x))
    torch.cuda.synchronize()
    codes, sf, g = O.quantize_per_row(O.bf16_to_f32(x))
    assert np.array_equal(q["codes"].cpu().numpy(), codes)
    assert np.array_equal(q["sf"].cpu().numpy(), O.swizzle_sf(sf))
    assert np.array_equal(q["g"].cpu().numpy().view(np.uint32), g.view(np.uint32))


@pytest.mark.parametrize("E,R,C", [(1, 32, 64), (3, 128, 256), (4, 100, 768), (2, 1536, 2048),
                                   (5, 2048, 768)])
def test_quantize_weights_per_expert_bit_exact(E, R, C):
    rng = np.random.default_rng(E * 1000 + R + C)
    w = O.f32_to_bf16((rng.standard_normal((E, R, C)) * 0.02).astype(np.float32))
    q = M.quantize(bf16_dev(w), per_group=True)
    torch.cuda.synchronize()
    codes, _, sw, g = O.quantize_weights(w)
    assert np.array_equal(q["codes"].cpu().numpy(), codes)
    assert np.array_equal(q["sf"].cpu().numpy(), sw)
    assert np.array_equal(q["g"].cpu().numpy().view(np.uint32), g.view(np.uint32))


@pytest.mark.parametrize("E,R,C", [(1, 64, 128), (2, 96, 80), (3, 2048, 768), (1, 48, 200),
                                   (2, 768, 1536)])
def test_quantize_weights_along_rows_bit_exact(E, R, C):
    rng = np.random.default_rng(E * 999 + R + C)
    w = O.f32_to_bf16((rng.standard_normal((E, R, C)) * 0.02).astype(np.float32))
    codes, _, sw, g = O.quantize_weights(w, along_rows=True)
    wd = bf16_dev(w)
    for g_in in (None, np_dev(g)):
        q = M.quantize(wd, per_group=True, along_rows=True, g_in=g_in)
        torch.cuda.synchronize()
        assert np.array_equal(q["codes"].cpu().numpy(), codes)
        assert np.array_equal(q["sf"].cpu().numpy(), sw)
        assert np.array_equal(q["g"].cpu().numpy().view(np.uint32), g.view(np.uint32))


@pytest.mark.parametrize("E,R,C", [(1, 64, 128), (2, 96, 80), (3, 2048, 768), (1, 48, 208),
                                   (2, 144, 1536), (4, 16, 16)])
def test_quantize_weights_both_orientations_in_one_pass_bit_exact(E, R, C):
    rng = np.random.default_rng(E * 77 + R + C)
    w = O.f32_to_bf16((rng.standard_normal((E, R, C)) * 0.02).astype(np.float32))
    w[0, 0, :] = 0  # a zero row in the forward copy, a zero element run in the transposed one
    ck, _, swk, gk = O.quantize_weights(w)
    cn, _, swn, gn = O.quantize_weights(w, along_rows=True)
    fk, fn = M.quantize_dual(bf16_dev(w))
    torch.cuda.synchronize()
    assert np.array_equal(fk["codes"].cpu().numpy(), ck)
    assert np.array_equal(fk["sf"].cpu().numpy(), swk)
    assert np.array_equal(fn["codes"].cpu().numpy(), cn)
    assert np.array_equal(fn["sf"].cpu().numpy(), swn)
    assert np.array_equal(fk["g"].cpu().numpy().view(np.uint32), gk.view(np.uint32))
    assert np.array_equal(gk.view(np.uint32), gn.view(np.uint32))


def test_tensor_wide_policy_depends_on_the_batch_and_per_token_does_not():
    """The comparison policy (one global scale over the whole activation
    tensor, PER_GROUP on a single group) matches the oracle's negative
    control bit-exactly and changes a token's codes when an outlier token
    joins the batch; per-token scaling leaves them unchanged."""
    rng = np.random.default_rng(41)
    x = _rand_bf16(rng, (32, 512))
    # outliers well above every row of x (whose rows carry scales up to 2^6)
    other = O.f32_to_bf16((rng.standard_normal((8, 512)) * 1e5).astype(np.float32))
    assert np.abs(O.bf16_to_f32(other)).max() > 100 * np.abs(O.bf16_to_f32(x)).max()
    both = np.concatenate([other, x])
    tw_alone = M.quantize(bf16_dev(x), per_group=True)
    tw_both = M.quantize(bf16_dev(both), per_group=True)
    pt_alone = M.quantize(bf16_dev(x))
    pt_both = M.quantize(bf16_dev(both))
    torch.cuda.synchronize()
    ref_c, ref_s, _ = O.quantize_tensor_wide_activations(O.bf16_to_f32(x))
    assert np.array_equal(tw_alone["codes"].cpu().numpy(), ref_c)
    assert np.array_equal(tw_alone["sf"].cpu().numpy(), O.swizzle_sf(ref_s))
    assert not np.array_equal(tw_both["codes"].cpu().numpy()[8:], tw_alone["codes"].cpu().numpy())
    assert np.array_equal(pt_both["codes"].cpu().numpy()[8:], pt_alone["codes"].cpu().numpy())
    assert np.array_equal(pt_both["g"].cpu().numpy()[8:].view(np.uint32),
                          pt_alone["g"].cpu().numpy().view(np.uint32))


# --------------------------------------------------------------------- permute

def run_permute(x_u16, ids, w, E):
    T, H = x_u16.shape
    k = ids.shape[1]
    mlp = M.MoEMLP(T, H, 64, E, k)
    status = _status()
    mlp.status = status
    mlp.permute_quant(bf16_dev(x_u16), np_dev(ids), None if w is None else np_dev(w))
    torch.cuda.synchronize()
    return mlp, int(status.item())


def check_permute(mlp, ref, H, check_rows=None):
    off = ref["expert_offsets"]
    Mu = int(off[-1])
    assert np.array_equal(mlp.offsets.cpu().numpy(), off)
    assert np.array_equal(mlp.sf_offsets.cpu().numpy(), ref["sf_row_offsets"])
    assert np.array_equal(mlp.dest_row.cpu().numpy(), ref["dest_row"])
    assert np.array_equal(mlp.perm_src.cpu().numpy()[:Mu], ref["perm_src"])
    if ref["perm_w"] is not None:
        assert np.array_equal(mlp.perm_w.cpu().numpy()[:Mu].view(np.uint32),
                              ref["perm_w"].view(np.uint32))
    rows = np.arange(Mu) if check_rows is None else check_rows
    assert np.array_equal(mlp.a_codes.cpu().numpy()[rows], ref["codes"][rows])
    assert np.array_equal(mlp.a_g.cpu().numpy()[rows].view(np.uint32), ref["row_g"][rows].view(np.uint32))
    n_sf = ref["sf_swizzled"].size
    assert np.array_equal(mlp.a_sf.cpu().numpy()[:n_sf], ref["sf_swizzled"])


def test_permute_tiny_config():
    d = IN.make_moe_inputs("tiny")
    E = d["cfg"]["E"]
    mlp, st = run_permute(d["x"], d["topk_ids"], d["topk_w"], E)
    assert st == 0
    check_permute(mlp, O.moe_permute_quant(d["x"], d["topk_ids"], d["topk_w"], E), d["cfg"]["H"])


@pytest.mark.parametrize("name,T", [("tiny", None), ("skewed", 1500), ("mlp", 300)])
def test_combine_backward_quant_equals_the_permutation_of_dy(name, T):
    """The combine backward with fused quantization, given the forward's
    routing, produces exactly what a fresh permutation of dY produces (codes,
    scales, row_g) and matches the oracle's permutation of dY bit for bit."""
    d = IN.make_moe_inputs(name, T=T, with_weights=False)
    c = d["cfg"]
    T, H, E, k = c["T"], c["H"], c["E"], c["k"]
    rng = np.random.default_rng(17)
    dy = _rand_bf16(rng, (T, H))
    dy[0] = 0
    ids, w = np_dev(d["topk_ids"]), np_dev(d["topk_w"])
    fwd = M.MoEMLP(T, H, 64, E, k)
    fwd.permute_quant(bf16_dev(d["x"]), ids, w)
    ref = M.MoEMLP(T, H, 64, E, k)
    ref.permute_quant(bf16_dev(dy), ids, None)
    Mt = T * k
    codes = torch.zeros((Mt, H // 2), dtype=torch.uint8, device="cuda")
    sf = torch.full((M.sf_bytes(Mt + 128 * E, H),), 0xAB, dtype=torch.uint8, device="cuda")
    g = torch.zeros(Mt, dtype=torch.float32, device="cuda")
    ws = torch.empty(M.minite_workspace_bytes(M.OP_COMBINE_BACKWARD_QUANT, T, H), dtype=torch.uint8,
                     device="cuda")
    st = _status()
    M.minite_moe_combine_backward_quant(bf16_dev(dy), E, fwd.dest_row, fwd.offsets, fwd.sf_offsets,
                                        fwd.perm_src, codes, sf, g, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    Mu = int(fwd.offsets[-1].item())
    assert torch.equal(codes[:Mu], ref.a_codes[:Mu])
    assert torch.equal(g[:Mu], ref.a_g[:Mu])
    p = O.moe_permute_quant(dy, d["topk_ids"], None, E)
    assert np.array_equal(codes.cpu().numpy()[:Mu], p["codes"])
    assert np.array_equal(g.cpu().numpy()[:Mu].view(np.uint32), p["row_g"].view(np.uint32))
    assert np.array_equal(sf.cpu().numpy()[:p["sf_swizzled"].size], p["sf_swizzled"])


def test_combine_backward_quant_rejects_inconsistent_routing_on_the_device():
    T, H, E, k = 64, 128, 2, 2
    rng = np.random.default_rng(3)
    dy = bf16_dev(_rand_bf16(rng, (T, H)))
    dest = torch.arange(T * k, dtype=torch.int32, device="cuda").view(T, k)
    perm_src = (torch.arange(T * k, dtype=torch.int32, device="cuda") // k).contiguous()
    codes = torch.full((T * k, H // 2), 7, dtype=torch.uint8, device="cuda")
    sf = torch.full((M.sf_bytes(T * k + 128 * E, H),), 7, dtype=torch.uint8, device="cuda")
    g = torch.zeros(T * k, dtype=torch.float32, device="cuda")
    ws = torch.empty(M.minite_workspace_bytes(M.OP_COMBINE_BACKWARD_QUANT, T, H), dtype=torch.uint8,
                     device="cuda")
    # offsets that decrease: nothing is written
    st = _status()
    M.minite_moe_combine_backward_quant(dy, E, dest, np_dev(np.array([0, 100, 90], np.int32)),
                                        np_dev(np.array([0, 128, 256], np.int32)), perm_src, codes,
                                        sf, g, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 1 << 1
    assert (codes == 7).all() and (sf == 7).all()
    # consistent offsets covering only 100 rows: the pairs routed past them are skipped
    st.zero_()
    M.minite_moe_combine_backward_quant(dy, E, dest, np_dev(np.array([0, 60, 100], np.int32)),
                                        np_dev(np.array([0, 128, 256], np.int32)), perm_src, codes,
                                        sf, g, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 1 << 1
    assert (codes[100:] == 7).all()
    assert not (codes[:100] == 7).all()


def test_permute_random_shapes_edge_cases():
    rng = np.random.default_rng(42)
    for trial in range(25):
        T = int(rng.integers(1, 301))
        E = int(rng.integers(1, 10))
        k = int(rng.integers(1, 5))
        H = int(rng.choice([64, 128, 192, 320]))
        ids = rng.integers(0, E, (T, k)).astype(np.int32)
        if trial % 5 == 1:
            ids[:] = E - 1  # everything to one expert
        if trial % 5 == 2 and E > 1:
            ids[ids == 0] = 1  # an empty expert
        if trial % 5 == 3:
            ids[rng.random((T, k)) < 0.05] = E + 3  # bad ids: dropped, status bit set
        w = rng.random((T, k)).astype(np.float32)
        x = _rand_bf16(rng, (T, H))
        mlp, st = run_permute(x, ids, w if trial % 2 else None, E)
        bad = ((ids < 0) | (ids >= E)).any()
        assert st == ((1 << M.ERR_BAD_ROUTING) if bad else 0)
        check_permute(mlp, O.moe_permute_quant(x, ids, w if trial % 2 else None, E), H)


def test_permute_qwen3_gate_up_layer_full_size():
    d = IN.make_moe_inputs("gate_up", with_weights=False)
    E = d["cfg"]["E"]
    mlp, st = run_permute(d["x"], d["topk_ids"], d["topk_w"], E)
    assert st == 0
    check_permute(mlp, O.moe_permute_quant(d["x"], d["topk_ids"], d["topk_w"], E), d["cfg"]["H"])


def test_permute_skewed_full_size_sampled_rows():
    d = IN.make_moe_inputs("skewed", with_weights=False)
    E = d["cfg"]["E"]
    mlp, st = run_permute(d["x"], d["topk_ids"], d["topk_w"], E)
    assert st == 0
    ref = O.moe_permute_quant(d["x"], d["topk_ids"], d["topk_w"], E)
    counts = np.diff(ref["expert_offsets"])
    assert (counts == 0).sum() == d["cfg"]["n_empty"]
    rng = np.random.default_rng(0)
    rows = rng.choice(int(ref["expert_offsets"][-1]), 4096, replace=False)
    check_permute(mlp, ref, d["cfg"]["H"], check_rows=np.sort(rows))


# --------------------------------------------------------------------- grouped GEMM

def make_gemm_case(counts, N, K, seed, act_scale=True):
    rng = np.random.default_rng(seed)
    E = len(counts)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    sfo = np.concatenate([[0], np.cumsum((np.array(counts) + 127) // 128 * 128)]).astype(np.int32)
    Mu = int(off[-1])
    x = _rand_bf16(rng, (max(Mu, 1), K))
    codes, sf, g = O.quantize_per_row(O.bf16_to_f32(x))
    a_sw = O.place_sf_per_expert(sf[:Mu], off, sfo)
    w = O.f32_to_bf16((rng.standard_normal((E, N, K)) * 0.02).astype(np.float32))
    bc, bsf, bsw, bg = O.quantize_weights(w)
    return dict(E=E, N=N, K=K, off=off, sfo=sfo, Mu=Mu, codes=codes, sf=sf, g=g, a_sw=a_sw,
                bc=bc, bsf=bsf, bsw=bsw, bg=bg)


def run_gemm(c, out_dtype, M_total=None):
    Mt = M_total or max(c["Mu"], 1)
    a_codes = torch.zeros((Mt, c["K"] // 2), dtype=torch.uint8, device="cuda")
    a_codes[:c["codes"].shape[0]] = np_dev(c["codes"][:Mt])
    a_sf = torch.zeros((Mt + 128 * c["E"]) * (c["K"] // 16), dtype=torch.uint8, device="cuda")
    a_sf[:c["a_sw"].size] = np_dev(c["a_sw"])
    a_g = torch.ones(Mt, dtype=torch.float32, device="cuda")
    a_g[:c["g"].shape[0]] = np_dev(c["g"][:Mt])
    out = torch.full((Mt, c["N"]), float("nan"), dtype=out_dtype, device="cuda")
    st = _status()
    M.minite_grouped_gemm_nvfp4(a_codes, a_sf, a_g, np_dev(c["bc"]), np_dev(c["bsw"]),
                                np_dev(c["bg"]), np_dev(c["off"]), np_dev(c["sfo"]), out, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return out


def check_gemm(c, out, rows=None):
    rows = np.arange(c["Mu"]) if rows is None else rows
    y, bound = O.grouped_gemm_exact(c["codes"], c["sf"], c["g"], c["bc"], c["bsf"], c["bg"],
                                    c["off"], rows=rows)
    if out.dtype == torch.float32:
        assert_fp32_within_bound(out.cpu().numpy()[rows], y, bound, "fp32 out")
    else:
        assert_bf16_within_one_ulp(u16(out)[rows], y, "bf16 out")


GEMM_CASES = [
    ([5], 32, 64), ([128], 128, 256), ([1, 0, 300, 17], 160, 320), ([0, 0, 0, 9], 384, 512),
    ([129, 127], 256, 2048), ([3, 200, 1, 0, 64], 96, 768), ([257], 128, 128), ([40] * 9, 64, 192),
    ([70, 300], 256, 1280),
]


@pytest.mark.parametrize("counts,N,K", GEMM_CASES)
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("variant", VARIANTS)
def test_grouped_gemm_small(counts, N, K, dtype, variant):
    M.minite_set_gemm_variant(variant)
    c = make_gemm_case(counts, N, K, seed=sum(counts) + N + K)
    out = run_gemm(c, dtype)
    check_gemm(c, out)
    # rows of no expert (beyond offsets[E]) are not written
    if out.shape[0] > c["Mu"]:
        assert torch.isnan(out[c["Mu"]:].float()).all()


@pytest.mark.parametrize("variant", VARIANTS)
def test_grouped_gemm_rows_beyond_used_are_untouched(variant):
    M.minite_set_gemm_variant(variant)
    c = make_gemm_case([10, 20], 128, 256, seed=3)
    out = run_gemm(c, torch.float32, M_total=100)
    check_gemm(c, out)
    assert torch.isnan(out[30:]).all()


@pytest.mark.parametrize("variant", VARIANTS)
def test_grouped_gemm_one_hot_weights_reproduce_dequantized_activations(variant):
    M.minite_set_gemm_variant(variant)
    rng = np.random.default_rng(9)
    Mu, K, N = 200, 256, 32
    x = _rand_bf16(rng, (Mu, K))
    codes, sf, g = O.quantize_per_row(O.bf16_to_f32(x))
    cols = rng.choice(K, N, replace=False)
    w = np.zeros((1, N, K), dtype=np.float32)
    w[0, np.arange(N), cols] = 6.0
    bc, bsf, bsw, bg = O.quantize_weights(O.f32_to_bf16(w))
    off = np.array([0, Mu], dtype=np.int32)
    c = dict(E=1, N=N, K=K, off=off, sfo=np.array([0, 256], dtype=np.int32), Mu=Mu, codes=codes,
             sf=sf, g=g, a_sw=O.place_sf_per_expert(sf, off, np.array([0, 256])), bc=bc,
             bsf=bsf, bsw=bsw, bg=bg)
    out = run_gemm(c, torch.float32).cpu().numpy()
    xh = O.dequantize(codes, sf, g)
    # one nonzero product per output: exact up to the final fp32 scaling
    ref = (6.0 * xh[:, cols]).astype(np.float32).astype(np.float64)
    assert np.allclose(out, ref, rtol=2.0 ** -22, atol=0)


@pytest.mark.parametrize("variant", VARIANTS)
def test_grouped_gemm_dense_config_bf16_and_fp32(variant):
    M.minite_set_gemm_variant(variant)
    d = IN.make_dense_inputs()
    Mr, N, K = d["cfg"]["M"], d["cfg"]["N"], d["cfg"]["K"]
    codes, sf, g = O.quantize_per_row(O.bf16_to_f32(d["a"]))
    bc, bsf, bsw, bg = O.quantize_weights(d["w"][None])
    off = np.array([0, Mr], dtype=np.int32)
    sfo = np.array([0, Mr], dtype=np.int32)
    c = dict(E=1, N=N, K=K, off=off, sfo=sfo, Mu=Mr, codes=codes, sf=sf, g=g,
             a_sw=O.swizzle_sf(sf), bc=bc, bsf=bsf, bsw=bsw, bg=bg)
    # the GPU quantizer reproduces the operands bit for bit
    qa = M.quantize(bf16_dev(d["a"]))
    torch.cuda.synchronize()
    assert np.array_equal(qa["codes"].cpu().numpy(), codes)
    rng = np.random.default_rng(1)
    rows = np.sort(np.concatenate([rng.choice(Mr, 1024, replace=False), [0, Mr - 1]]))
    for dt in (torch.float32, torch.bfloat16):
        out = run_gemm(c, dt)
        check_gemm(c, out, rows=np.unique(rows))


@pytest.mark.parametrize("variant", VARIANTS)
def test_grouped_gemm_batch_invariance(variant):
    """A token's output row is bitwise identical whatever else is routed to its
    expert (more rows, fewer rows, other experts)."""
    M.minite_set_gemm_variant(variant)
    base = make_gemm_case([70, 150, 33], 128, 512, seed=11)
    out0 = run_gemm(base, torch.float32).cpu().numpy()
    rng = np.random.default_rng(12)
    extra = _rand_bf16(rng, (300, 512))
    ec, esf, eg = O.quantize_per_row(O.bf16_to_f32(extra))
    # expert 1 gets 300 more rows appended after its own; experts 0 and 2 unchanged
    off0 = base["off"]
    order = np.concatenate([np.arange(0, off0[2]), -1 - np.arange(300), np.arange(off0[2], off0[3])])
    codes = np.concatenate([base["codes"][:off0[2]], ec, base["codes"][off0[2]:off0[3]]])
    sf = np.concatenate([base["sf"][:off0[2]], esf, base["sf"][off0[2]:off0[3]]])
    g = np.concatenate([base["g"][:off0[2]], eg, base["g"][off0[2]:off0[3]]])
    counts = [70, 450, 33]
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    sfo = np.concatenate([[0], np.cumsum((np.array(counts) + 127) // 128 * 128)]).astype(np.int32)
    c = dict(base, off=off, sfo=sfo, Mu=553, codes=codes, sf=sf, g=g,
             a_sw=O.place_sf_per_expert(sf, off, sfo))
    out1 = run_gemm(c, torch.float32).cpu().numpy()
    keep = order >= 0
    assert np.array_equal(out1[keep].view(np.uint32), out0[order[keep]].view(np.uint32))
    # and alone: expert 1's first 5 rows routed with nothing else
    c2 = dict(base, off=np.array([0, 0, 5, 5], dtype=np.int32),
              sfo=np.array([0, 0, 128, 128], dtype=np.int32), Mu=5, codes=base["codes"][70:75],
              sf=base["sf"][70:75], g=base["g"][70:75],
              a_sw=O.place_sf_per_expert(base["sf"][70:75], np.array([0, 0, 5, 5]), np.array([0, 0, 128, 128])))
    out2 = run_gemm(c2, torch.float32).cpu().numpy()
    assert np.array_equal(out2[:5].view(np.uint32), out0[70:75].view(np.uint32))


def test_grouped_gemm_kernels_agree_bitwise():
    """All grouped-GEMM kernels use the same K order per row, so their
    outputs are identical."""
    c = make_gemm_case([300, 0, 1, 700, 129], 384, 1024, seed=31)
    outs = []
    for v in VARIANTS:
        M.minite_set_gemm_variant(v)
        outs.append(run_gemm(c, torch.float32).cpu().numpy().view(np.uint32))
    for o in outs[1:]:
        assert np.array_equal(outs[0], o)


@pytest.mark.parametrize("counts,N,K", [
    ([300, 0, 33, 129, 64, 1], 512, 256),
    # 401 experts: the CTA-pair kernel's output staging no longer fits beside
    # the per-expert tables, so every row takes the plain (transposed) stores
    ([0] * 200 + [97] + [0] * 199 + [260], 256, 128),
])
def test_grouped_gemm_bf16_store_paths_agree_bitwise(counts, N, K):
    """BF16 output of the CTA-pair kernel: whole 32-row boxes by TMA stores,
    an expert's last rows by plain stores of four-lane transposed chunks. Both
    agree bit for bit with the single-CTA kernel and within one BF16 ulp with
    the exact product, and rows past the last expert stay untouched."""
    c = make_gemm_case(counts, N, K, seed=sum(counts) + len(counts))
    outs = []
    for v in (1, 6):
        M.minite_set_gemm_variant(v)
        out = run_gemm(c, torch.bfloat16, M_total=c["Mu"] + 40)
        check_gemm(c, out)
        assert torch.isnan(out[c["Mu"]:].float()).all()
        outs.append(u16(out))
    assert np.array_equal(outs[0], outs[1])


@pytest.mark.parametrize("variant", VARIANTS)
def test_grouped_gemm_inconsistent_offsets_are_reported_not_executed(variant):
    M.minite_set_gemm_variant(variant)
    c = make_gemm_case([10, 20], 128, 256, seed=5)
    c["off"] = np.array([0, 25, 20], dtype=np.int32)  # decreasing
    Mt = 30
    out = torch.full((Mt, 128), float("nan"), dtype=torch.float32, device="cuda")
    st = _status()
    M.minite_grouped_gemm_nvfp4(np_dev(c["codes"]), np_dev(np.resize(c["a_sw"], (Mt + 256) * 16)),
                                np_dev(c["g"]), np_dev(c["bc"]), np_dev(c["bsw"]), np_dev(c["bg"]),
                                np_dev(c["off"]), np_dev(c["sfo"]), out, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 1 << 1
    assert torch.isnan(out).all()


# --------------------------------------------------------------------- SwiGLU, combine

@pytest.mark.parametrize("counts,I", [([3, 0, 130, 1], 64), ([256, 17], 768), ([1], 128),
                                      ([100] * 5, 1536), ([5, 130], 512), ([33], 1024),
                                      ([40, 0, 7], 2048)])
def test_swiglu_weighted_quant_bit_exact(counts, I):
    rng = np.random.default_rng(len(counts) * 31 + I)
    E = len(counts)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    sfo = np.concatenate([[0], np.cumsum((np.array(counts) + 127) // 128 * 128)]).astype(np.int32)
    Mu = int(off[-1])
    Mt = Mu + 7
    gu = O.f32_to_bf16((rng.standard_normal((Mt, 2 * I)) * 3).astype(np.float32))
    gu[0, :I] = O.f32_to_bf16(np.linspace(-120, 120, I).astype(np.float32))  # clamp region
    # gates on both sides of every tabulation edge: zeros, subnormals, |g| near
    # 2^-24 and 2^8, large magnitudes
    special = np.array([0.0, -0.0, 1e-40, -1e-40, 2.0 ** -25, -(2.0 ** -24), 2.0 ** -24,
                        -(2.0 ** -25), 255.0, -255.0, 256.0, -256.0, 300.0, -300.0, 3e4, -3e4],
                       dtype=np.float32)
    gu[1 % Mt, :I] = O.f32_to_bf16(np.resize(special, I))
    pw = rng.random(Mt).astype(np.float32)
    for weights in (pw, None):
        ref = O.swiglu_weighted_quant(gu, weights, off, sfo)
        codes = torch.zeros((Mt, I // 2), dtype=torch.uint8, device="cuda")
        sf = torch.full(((Mt + 128 * E) * (I // 16),), 0xAB, dtype=torch.uint8, device="cuda")
        g = torch.zeros(Mt, dtype=torch.float32, device="cuda")
        st = _status()
        M.minite_swiglu_weighted_quant(bf16_dev(gu), None if weights is None else np_dev(weights),
                                       E, np_dev(off), np_dev(sfo), codes, sf, g, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert np.array_equal(codes.cpu().numpy()[:Mu], ref["codes"])
        assert np.array_equal(sf.cpu().numpy()[:ref["sf_swizzled"].size], ref["sf_swizzled"])
        assert np.array_equal(g.cpu().numpy()[:Mu].view(np.uint32), ref["row_g"].view(np.uint32))


@pytest.mark.parametrize("counts,I", [([3, 0, 130, 1], 64), ([256, 17], 768), ([1], 128),
                                      ([100] * 5, 1536), ([5, 130], 512), ([33], 1024),
                                      ([40, 0, 7], 2048), ([300, 212], 768)])
def test_swiglu_backward_quant_bit_exact(counts, I):
    rng = np.random.default_rng(len(counts) * 37 + I + 1)
    E = len(counts)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    sfo = np.concatenate([[0], np.cumsum((np.array(counts) + 127) // 128 * 128)]).astype(np.int32)
    Mu = int(off[-1])
    Mt = Mu + 5
    gu = O.f32_to_bf16((rng.standard_normal((Mt, 2 * I)) * 3).astype(np.float32))
    dh = _rand_bf16(rng, (Mt, I), scale_spread=10)
    gu[0, :I] = O.f32_to_bf16(np.linspace(-120, 120, I).astype(np.float32))  # clamp region
    special = np.array([0.0, -0.0, 1e-40, -1e-40, 2.0 ** -25, -(2.0 ** -24), 2.0 ** -24,
                        -(2.0 ** -25), 255.0, -255.0, 256.0, -256.0, 300.0, -300.0, 3e4, -3e4],
                       dtype=np.float32)
    gu[1 % Mt, :I] = O.f32_to_bf16(np.resize(special, I))
    dh[2 % Mt] = 0  # zero gradient row: global scale 1, all codes and scales 0
    dh[3 % Mt, ::7] = O.f32_to_bf16(np.array([1.0e30], dtype=np.float32))[0]  # huge, finite
    pw = rng.random(Mt).astype(np.float32)
    for weights in (pw, None):
        ref = O.swiglu_backward_quant(gu, dh, weights, off, sfo)
        codes = torch.zeros((Mt, I), dtype=torch.uint8, device="cuda")
        sf = torch.full(((Mt + 128 * E) * (2 * I // 16),), 0xAB, dtype=torch.uint8, device="cuda")
        g = torch.zeros(Mt, dtype=torch.float32, device="cuda")
        st = _status()
        M.minite_swiglu_backward_quant(bf16_dev(gu), bf16_dev(dh),
                                       None if weights is None else np_dev(weights),
                                       E, np_dev(off), np_dev(sfo), codes, sf, g, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert np.array_equal(codes.cpu().numpy()[:Mu], ref["codes"])
        assert np.array_equal(sf.cpu().numpy()[:ref["sf_swizzled"].size], ref["sf_swizzled"])
        assert np.array_equal(g.cpu().numpy()[:Mu].view(np.uint32), ref["row_g"].view(np.uint32))
        assert (codes.cpu().numpy()[Mu:] == 0).all()  # rows past the last expert untouched


def test_swiglu_backward_inconsistent_offsets_are_reported_not_executed():
    I, E = 128, 2
    gu = torch.zeros((40, 2 * I), dtype=torch.bfloat16, device="cuda")
    dh = torch.ones((40, I), dtype=torch.bfloat16, device="cuda")
    off = np.array([0, 30, 20], dtype=np.int32)  # decreasing
    sfo = np.array([0, 128, 128], dtype=np.int32)
    codes = torch.full((40, I), 7, dtype=torch.uint8, device="cuda")
    sf = torch.full((512 * 16,), 7, dtype=torch.uint8, device="cuda")
    g = torch.zeros(40, dtype=torch.float32, device="cuda")
    st = _status()
    M.minite_swiglu_backward_quant(gu, dh, None, E, np_dev(off), np_dev(sfo), codes, sf, g, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 1 << 1
    assert (codes == 7).all() and (sf == 7).all()


@pytest.mark.parametrize("T,k,N", [(1, 1, 8), (64, 2, 64), (300, 8, 2048), (33, 5, 136)])
def test_combine_bit_exact(T, k, N):
    rng = np.random.default_rng(T * k + N)
    Mr = T * k
    D = O.f32_to_bf16(rng.standard_normal((Mr, N)).astype(np.float32))
    dest = rng.permutation(Mr).reshape(T, k).astype(np.int32)
    if T > 2:
        dest[1, 0] = -1
    y = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
    st = _status()
    M.minite_moe_combine(bf16_dev(D), np_dev(dest), y, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert np.array_equal(u16(y), O.moe_combine(D, dest))


# --------------------------------------------------------------------- whole MLP

def _weights(d):
    return (M.quantize(bf16_dev(d["w_gate_up"]), per_group=True),
            M.quantize(bf16_dev(d["w_down"]), per_group=True))


def test_mlp_tiny_stagewise_and_end_to_end():
    """The tiny configuration through every stage, all 64 tokens: permutation
    bit-exact, both GEMMs within one BF16 ulp of the exact product, SwiGLU
    codes and the combine bit-exact (each stage given the oracle's input)."""
    d = IN.make_moe_inputs("tiny")
    c = d["cfg"]
    T, H, E, k, I = c["T"], c["H"], c["E"], c["k"], c["I"]
    wgu, wd = _weights(d)
    mlp = M.MoEMLP(T, H, I, E, k)
    mlp.forward(bf16_dev(d["x"]), np_dev(d["topk_ids"]), np_dev(d["topk_w"]), wgu, wd)
    torch.cuda.synchronize()
    assert int(mlp.status.item()) == 0
    wq = (O.quantize_weights(d["w_gate_up"]), O.quantize_weights(d["w_down"]))
    ref = O.moe_mlp_forward(d["x"], d["topk_ids"], d["topk_w"], E, *wq)
    check_permute(mlp, ref["permute"], H)
    check_forward_stagewise(d, np.arange(T), wq, mlp, wgu, wd, mlp.status)


def _dev_rows(a, rows, dtype=None):
    """Device copy of oracle array `a` in a zeroed buffer of `rows` rows (the
    rows past a's are the unused capacity a stage's buffers have)."""
    out = np.zeros((rows,) + a.shape[1:], dtype=a.dtype if dtype is None else dtype)
    out[:a.shape[0]] = a
    return bf16_dev(out) if out.dtype == np.uint16 else np_dev(out)


@pytest.mark.parametrize("name,T", [("tiny", None), ("mlp", 256)])
def test_backward_chain_stagewise(name, T):
    """The NVFP4 backward of the expert MLP, stage by stage: permute+quant of
    dY, down dgrad GEMM (W_down quantized along N), SwiGLU backward with
    per-row requantization, gate_up dgrad GEMM (W_gate_up quantized along N),
    combine of dX. The oracle runs the whole chain from the layer's inputs;
    a GPU stage whose input is an earlier stage's result takes the oracle's
    value of it (uploaded), so no expected value depends on GPU output.
    Codes, scales and the combine bit-exact, GEMM outputs within one BF16 ulp
    of the exact result."""
    d = IN.make_moe_inputs(name, T=T)
    c = d["cfg"]
    T, H, E, k, I = c["T"], c["H"], c["E"], c["k"], c["I"]
    rng = np.random.default_rng(9)
    dy = O.f32_to_bf16(rng.standard_normal((T, H)).astype(np.float32))
    # the oracle's chain
    fwd = O.moe_mlp_forward(d["x"], d["topk_ids"], d["topk_w"], E,
                            O.quantize_weights(d["w_gate_up"]), O.quantize_weights(d["w_down"]))
    pf = fwd["permute"]
    p = O.moe_permute_quant(dy, d["topk_ids"], None, E)
    off, sfo = p["expert_offsets"], p["sf_row_offsets"]
    assert np.array_equal(off, pf["expert_offsets"])
    Mu = int(off[-1])
    qdT = O.quantize_weights(d["w_down"], along_rows=True)
    dh_exact, _ = O.grouped_gemm_exact(p["codes"], p["sf"], p["row_g"], qdT[0], qdT[1], qdT[3], off)
    dh_o = O.f64_to_bf16(dh_exact)
    sb = O.swiglu_backward_quant(fwd["gate_up"], dh_o, pf["perm_w"], off, sfo)
    qguT = O.quantize_weights(d["w_gate_up"], along_rows=True)
    dx_exact, _ = O.grouped_gemm_exact(sb["codes"], sb["sf"], sb["row_g"], qguT[0], qguT[1],
                                       qguT[3], off)
    dxp_o = O.f64_to_bf16(dx_exact)
    dx_o = O.moe_combine(dxp_o, pf["dest_row"])

    # the GPU's stages
    ids = np_dev(d["topk_ids"])
    _, wdT = M.quantize_dual(bf16_dev(d["w_down"]))
    _, wguT = M.quantize_dual(bf16_dev(d["w_gate_up"]))
    bwd = M.MoEMLP(T, H, I, E, k)
    bwd.permute_quant(bf16_dev(dy), ids, None)
    Mt = T * k
    st = _status()
    dh = torch.empty((Mt, I), dtype=torch.bfloat16, device="cuda")
    M.minite_grouped_gemm_nvfp4(bwd.a_codes, bwd.a_sf, bwd.a_g, wdT["codes"], wdT["sf"], wdT["g"],
                                bwd.offsets, bwd.sf_offsets, dh, st)
    off_d, sfo_d = np_dev(off), np_dev(sfo)
    dgu_codes = torch.zeros((Mt, I), dtype=torch.uint8, device="cuda")
    dgu_sf = torch.full((M.sf_bytes(Mt + 128 * E, 2 * I),), 0xAB, dtype=torch.uint8, device="cuda")
    dgu_g = torch.zeros(Mt, dtype=torch.float32, device="cuda")
    M.minite_swiglu_backward_quant(_dev_rows(fwd["gate_up"], Mt), _dev_rows(dh_o, Mt),
                                   _dev_rows(pf["perm_w"], Mt), E, off_d, sfo_d, dgu_codes, dgu_sf,
                                   dgu_g, st)
    dx_perm = torch.empty((Mt, H), dtype=torch.bfloat16, device="cuda")
    M.minite_grouped_gemm_nvfp4(dgu_codes, dgu_sf, dgu_g, wguT["codes"], wguT["sf"], wguT["g"],
                                off_d, sfo_d, dx_perm, st)
    dx = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    M.minite_moe_combine(_dev_rows(dxp_o, Mt), np_dev(pf["dest_row"]), dx, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and int(bwd.status.item()) == 0

    check_permute(bwd, p, H)
    assert_bf16_within_one_ulp(u16(dh)[:Mu], dh_exact, "dh")
    assert np.array_equal(dgu_codes.cpu().numpy()[:Mu], sb["codes"])
    assert np.array_equal(dgu_sf.cpu().numpy()[:sb["sf_swizzled"].size], sb["sf_swizzled"])
    assert np.array_equal(dgu_g.cpu().numpy()[:Mu].view(np.uint32), sb["row_g"].view(np.uint32))
    assert_bf16_within_one_ulp(u16(dx_perm)[:Mu], dx_exact, "dx_perm")
    assert np.array_equal(u16(dx), dx_o)


# --------------------------------------------------------------------- weight gradient

def check_token_operand(q, ref, C):
    """A GPU token-axis operand against the oracle's: K offsets, codes and
    global scales equal; every scale byte up to column kofs[E] / 16 equal
    (rows past C zero), read at the layout's offsets."""
    K = int(ref["kofs"][-1])
    assert np.array_equal(q["kofs"].cpu().numpy(), ref["kofs"])
    assert np.array_equal(q["codes"].cpu().numpy()[:, :K // 2], ref["codes"])
    rp = (C + 127) // 128 * 128
    r, col = np.meshgrid(np.arange(rp), np.arange(K // 16), indexing="ij")
    want = np.zeros((rp, K // 16), dtype=np.uint8)
    want[:C] = ref["sf"]
    got = q["sf"].cpu().numpy()[O.sf_swizzle_offset(r, col, q["k_cap"] // 16)]
    assert np.array_equal(got, want)
    assert np.array_equal(q["g"].cpu().numpy().view(np.uint32), ref["g"].view(np.uint32))


@pytest.mark.parametrize("counts,C,gather", [([3, 0, 260, 17], 48, True), ([1], 16, False),
                                              ([700, 5, 0, 0, 129], 256, True),
                                              ([64, 64], 2048, False), ([300, 1000], 768, True)])
@pytest.mark.parametrize("given_amax", [False, True])
def test_quantize_tokens_bit_exact(counts, C, gather, given_amax):
    """Token-axis operand against the oracle, the experts' maxima taken from
    the rows themselves or from caller-given per-row maxima (as the SwiGLU
    entries that keep BF16 output write them)."""
    rng = np.random.default_rng(sum(counts) + C)
    E = len(counts)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    Mu = int(off[-1])
    if gather:  # permuted row m is source row src[m] of a smaller matrix
        T = max(1, Mu // 3)
        x = _rand_bf16(rng, (T, C))
        src = rng.integers(0, T, Mu + 5).astype(np.int32)
        rows = O.bf16_to_f32(x)[src[:Mu]]
        xd = bf16_dev(x)
        ra = xd.float().abs().amax(dim=1) if given_amax else None
        q = M.quantize_tokens(xd, np_dev(off), E, row_src=np_dev(src), row_amax=ra)
    else:
        x = _rand_bf16(rng, (Mu + 7, C))
        x[:, 3] = 0  # a zero channel
        rows = O.bf16_to_f32(x)[:Mu]
        xd = bf16_dev(x)
        ra = xd.float().abs().amax(dim=1) if given_amax else None
        q = M.quantize_tokens(xd, np_dev(off), E, row_amax=ra)
    torch.cuda.synchronize()
    check_token_operand(q, O.quantize_tokens_per_expert(rows, off), C)


@pytest.mark.parametrize("counts,Ma,Nb", [([3, 0, 260, 17], 128, 256), ([1000, 40], 256, 96),
                                          ([600], 2048, 768), ([5, 300, 2, 0, 90, 1], 160, 32)])
def test_wgrad_gemm_within_bound(counts, Ma, Nb):
    rng = np.random.default_rng(7 * sum(counts) + Ma)
    E = len(counts)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    Mu = int(off[-1])
    xa = _rand_bf16(rng, (Mu, Ma))
    xb = _rand_bf16(rng, (Mu, Nb))
    qa = M.quantize_tokens(bf16_dev(xa), np_dev(off), E)
    qb = M.quantize_tokens(bf16_dev(xb), np_dev(off), E)
    outs = {}
    for dt in (torch.float32, torch.bfloat16):
        out = torch.full((E, Ma, Nb), float("nan"), dtype=dt, device="cuda")
        st = _status()
        M.minite_grouped_gemm_wgrad_nvfp4(qa, qb, out, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        outs[dt] = out
    ra = O.quantize_tokens_per_expert(O.bf16_to_f32(xa), off)
    rb = O.quantize_tokens_per_expert(O.bf16_to_f32(xb), off)
    check_token_operand(qa, ra, Ma)
    check_token_operand(qb, rb, Nb)
    y, bound = O.wgrad_exact(ra, rb)
    for e in range(E):
        if counts[e] == 0:
            assert torch.isnan(outs[torch.float32][e]).all()  # experts without tokens: untouched
            continue
        assert_fp32_within_bound(outs[torch.float32][e].cpu().numpy(), y[e], bound[e], f"dW[{e}]")
        assert_bf16_within_one_ulp(u16(outs[torch.bfloat16][e]), y[e], f"dW[{e}] bf16")


def _small_moe(seed, T, H, I, E, k):
    rng = np.random.default_rng(seed)
    logits = rng.standard_normal((T, E))
    ids = np.argsort(-logits, axis=1)[:, :k].astype(np.int32)
    w = rng.random((T, k)).astype(np.float32)
    return dict(x=O.f32_to_bf16(rng.standard_normal((T, H)).astype(np.float32)), ids=ids, w=w,
                wgu=O.f32_to_bf16((rng.standard_normal((E, 2 * I, H)) * 0.02).astype(np.float32)),
                wd=O.f32_to_bf16((rng.standard_normal((E, H, I)) * 0.02).astype(np.float32)),
                dy=O.f32_to_bf16(rng.standard_normal((T, H)).astype(np.float32)))


@pytest.mark.parametrize("T,H,I,E,k", [(64, 64, 64, 4, 2), (600, 256, 128, 4, 2),
                                       (900, 128, 64, 8, 3)])
def test_weight_gradients_stagewise(T, H, I, E, k):
    """Both weight gradients of the expert MLP, stage by stage: the forward
    keeps BF16 h, the SwiGLU backward keeps BF16 [dg | du]; dW_down sums
    dY x h and dW_gate_up sums [dg | du] x x over each expert's tokens, from
    token-axis NVFP4 operands. Operands bit-exact, gradients within
    2^-20 sum|ab| of the exact result."""
    d = _small_moe(T + H, T, H, I, E, k)
    # the oracle's chain from the layer's inputs
    fwd = O.moe_mlp_forward(d["x"], d["ids"], d["w"], E, O.quantize_weights(d["wgu"]),
                            O.quantize_weights(d["wd"]))
    pf = fwd["permute"]
    off, src, perm_w = pf["expert_offsets"], pf["perm_src"], pf["perm_w"]
    Mu = int(off[-1])
    gu_f = O.bf16_to_f32(fwd["gate_up"])
    h_o = O.f32_to_bf16(O.swiglu_weighted(gu_f, perm_w))
    p_dy = O.moe_permute_quant(d["dy"], d["ids"], None, E)
    qdT = O.quantize_weights(d["wd"], along_rows=True)
    dh_exact, _ = O.grouped_gemm_exact(p_dy["codes"], p_dy["sf"], p_dy["row_g"], qdT[0], qdT[1],
                                       qdT[3], off)
    dh_o = O.f64_to_bf16(dh_exact)
    dgu_o = O.f32_to_bf16(O.swiglu_backward(gu_f, O.bf16_to_f32(dh_o), perm_w))
    r_dy = O.quantize_tokens_per_expert(O.bf16_to_f32(d["dy"])[src], off)
    r_h = O.quantize_tokens_per_expert(O.bf16_to_f32(h_o), off)
    r_dgu = O.quantize_tokens_per_expert(O.bf16_to_f32(dgu_o), off)
    r_x = O.quantize_tokens_per_expert(O.bf16_to_f32(d["x"])[src], off)

    # the GPU's stages; a stage whose input is an earlier stage's result takes
    # the oracle's value of it
    dev = "cuda"
    x, ids, w, dy = bf16_dev(d["x"]), np_dev(d["ids"]), np_dev(d["w"]), bf16_dev(d["dy"])
    mlp = M.MoEMLP(T, H, I, E, k)
    Mt = T * k
    st = _status()
    mlp.permute_quant(x, ids, w)
    gu_in, pw_in = _dev_rows(fwd["gate_up"], Mt), _dev_rows(perm_w, Mt)
    h = torch.zeros((Mt, I), dtype=torch.bfloat16, device=dev)
    h_amax = torch.full((Mt,), float("nan"), dtype=torch.float32, device=dev)
    M.minite_swiglu_weighted_quant_keep_h(gu_in, pw_in, E, mlp.offsets, mlp.sf_offsets,
                                          mlp.h_codes, mlp.h_sf, mlp.h_g, h, st, h_amax=h_amax)
    dgu_codes = torch.empty((Mt, I), dtype=torch.uint8, device=dev)
    dgu_sf = torch.empty((M.sf_bytes(Mt + 128 * E, 2 * I),), dtype=torch.uint8, device=dev)
    dgu_g = torch.empty(Mt, dtype=torch.float32, device=dev)
    dgu = torch.zeros((Mt, 2 * I), dtype=torch.bfloat16, device=dev)
    dgu_amax = torch.full((Mt,), float("nan"), dtype=torch.float32, device=dev)
    M.minite_swiglu_backward_quant_keep(gu_in, _dev_rows(dh_o, Mt), pw_in, E, mlp.offsets,
                                        mlp.sf_offsets, dgu_codes, dgu_sf, dgu_g, dgu, st,
                                        dgu_amax=dgu_amax)
    q_dy = M.quantize_tokens(dy, mlp.offsets, E, row_src=mlp.perm_src, m_cap=Mt)
    q_h = M.quantize_tokens(h, mlp.offsets, E, m_cap=Mt, row_amax=h_amax)
    q_dgu = M.quantize_tokens(dgu, mlp.offsets, E, m_cap=Mt, row_amax=dgu_amax)
    q_x = M.quantize_tokens(x, mlp.offsets, E, row_src=mlp.perm_src, m_cap=Mt)
    dWd = torch.full((E, H, I), float("nan"), dtype=torch.float32, device=dev)
    dWgu = torch.full((E, 2 * I, H), float("nan"), dtype=torch.float32, device=dev)
    M.minite_grouped_gemm_wgrad_nvfp4(q_dy, q_h, dWd, st)
    M.minite_grouped_gemm_wgrad_nvfp4(q_dgu, q_x, dWgu, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and int(mlp.status.item()) == 0

    assert np.array_equal(mlp.offsets.cpu().numpy(), off)
    assert np.array_equal(mlp.perm_src.cpu().numpy()[:Mu], src)
    # the kept BF16 tensors are the roundings of what the stages quantize
    assert np.array_equal(u16(h)[:Mu], h_o)
    assert np.array_equal(u16(dgu)[:Mu], dgu_o)
    # the row maxima written beside them: max |row| of the kept rows, rows past Mu untouched
    for amax, kept in ((h_amax, h_o), (dgu_amax, dgu_o)):
        a_ = amax.cpu().numpy()
        assert np.array_equal(a_[:Mu], np.abs(O.bf16_to_f32(kept)).max(axis=1))
        assert np.isnan(a_[Mu:]).all()
    for q, r, C in ((q_dy, r_dy, H), (q_h, r_h, I), (q_dgu, r_dgu, 2 * I), (q_x, r_x, H)):
        check_token_operand(q, r, C)
    for out, ra, rb in ((dWd, r_dy, r_h), (dWgu, r_dgu, r_x)):
        y, bound = O.wgrad_exact(ra, rb)
        got = out.cpu().numpy()
        for e in range(E):
            if off[e + 1] == off[e]:
                continue
            assert_fp32_within_bound(got[e], y[e], bound[e], f"dW[{e}]")


def test_wgrad_gemm_rejects_bad_token_offsets():
    rng = np.random.default_rng(8)
    off = np.array([0, 100, 300], np.int32)
    xa = _rand_bf16(rng, (300, 128))
    qa = M.quantize_tokens(bf16_dev(xa), np_dev(off), 2)
    qa["kofs"] = np_dev(np.array([0, 200, 512], np.int32))  # 200: not a multiple of 256
    out = torch.full((2, 128, 128), float("nan"), dtype=torch.float32, device="cuda")
    st = _status()
    M.minite_grouped_gemm_wgrad_nvfp4(qa, qa, out, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 1 << 1
    assert torch.isnan(out).all()


@pytest.mark.parametrize("I", [64, 768, 2048])
def test_swiglu_keep_h_stores_rounded_h_its_row_maxima_and_the_same_codes(I):
    rng = np.random.default_rng(I)
    counts = [5, 130, 0, 40]
    E = len(counts)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    sfo = np.concatenate([[0], np.cumsum((np.array(counts) + 127) // 128 * 128)]).astype(np.int32)
    Mu = int(off[-1])
    Mt = Mu + 3
    gu = O.f32_to_bf16((rng.standard_normal((Mt, 2 * I)) * 3).astype(np.float32))
    pw = rng.random(Mt).astype(np.float32)
    res = []
    for keep in (False, True):
        codes = torch.zeros((Mt, I // 2), dtype=torch.uint8, device="cuda")
        sf = torch.zeros(((Mt + 128 * E) * (I // 16),), dtype=torch.uint8, device="cuda")
        g = torch.zeros(Mt, dtype=torch.float32, device="cuda")
        h = torch.zeros((Mt, I), dtype=torch.bfloat16, device="cuda")
        h_amax = torch.full((Mt,), float("nan"), dtype=torch.float32, device="cuda")
        st = _status()
        if keep:
            M.minite_swiglu_weighted_quant_keep_h(bf16_dev(gu), np_dev(pw), E, np_dev(off),
                                                  np_dev(sfo), codes, sf, g, h, st, h_amax=h_amax)
        else:
            M.minite_swiglu_weighted_quant(bf16_dev(gu), np_dev(pw), E, np_dev(off), np_dev(sfo),
                                           codes, sf, g, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        res.append((codes, sf, g, h, h_amax))
    for a, b in zip(res[0][:3], res[1][:3]):
        assert torch.equal(a, b)
    ref = O.f32_to_bf16(O.swiglu_weighted(O.bf16_to_f32(gu[:Mu]), pw[:Mu]))
    assert np.array_equal(u16(res[1][3])[:Mu], ref)
    assert (u16(res[1][3])[Mu:] == 0).all()
    # each kept row's |h| maximum; rows past the routed ones untouched
    amax = res[1][4].cpu().numpy()
    assert np.array_equal(amax[:Mu], np.abs(O.bf16_to_f32(ref)).max(axis=1))
    assert np.isnan(amax[Mu:]).all()


# --------------------------------------------------------------------- failure detection

@pytest.mark.parametrize("variant", VARIANTS)
def test_gemm_wait_timeout_sets_status_and_context_survives(variant):
    M.minite_set_gemm_variant(variant)
    c = make_gemm_case([600, 300], 256, 2048, seed=21)
    Mt = c["Mu"]
    args = [np_dev(c["codes"]), np_dev(np.concatenate([c["a_sw"], np.zeros(256 * 128, np.uint8)])),
            np_dev(c["g"]), np_dev(c["bc"]), np_dev(c["bsw"]), np_dev(c["bg"]), np_dev(c["off"]),
            np_dev(c["sfo"])]
    out = torch.zeros((Mt, 256), dtype=torch.float32, device="cuda")
    st = _status()
    try:
        M.minite_set_wait_budget_ns(1)
        M.minite_grouped_gemm_nvfp4(*args, out, st)
        torch.cuda.synchronize()
    finally:
        M.minite_set_wait_budget_ns(0)
    assert int(st.item()) & (1 << M.ERR_TIMEOUT)
    st.zero_()
    M.minite_grouped_gemm_nvfp4(*args, out, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    check_gemm(c, out)
