"""Full-size parity of the expert-MLP path, stage by stage, on sampled rows.

The GPU runs each configuration at its full size, in the launch
configuration the benchmark times. The oracle cannot afford every row at
these sizes, but per-token scaling makes each permuted row's result depend
on that row's inputs alone, so it runs on sampled tokens (or rows) and the
GPU's rows of those tokens are located through the oracle's own permutation
of the whole batch.

Every stage is held to its own bar: routing metadata, codes, scales and the
combine bit for bit; grouped-GEMM outputs within one BF16 ulp of the
correctly rounded exact product. A stage whose input is an earlier stage's
result takes, for the sampled rows, the oracle's value of that input
(written into the GPU's full-size buffer before the stage is launched again
at full size); rows that are not sampled keep the GPU's own values and are
not checked. No expected value passes through the GPU.
"""
import numpy as np
import pytest
import torch

from _helpers import assert_bf16_within_one_ulp, bf16_dev, np_dev, u16
from _stagewise import check_forward_stagewise, take
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
    M.minite_set_gemm_variant(0)
    yield


_INPUTS = {}
_WQ = {}


def _inputs(name):
    if name not in _INPUTS:
        _INPUTS[name] = IN.make_moe_inputs(name)
    return _INPUTS[name]


def _oracle_weights(name):
    """The oracle's quantization of both weights (codes, sf, sf_swizzled, g)."""
    if name not in _WQ:
        d = _inputs(name)
        _WQ[name] = (O.quantize_weights(d["w_gate_up"]), O.quantize_weights(d["w_down"]))
    return _WQ[name]


def test_gate_up_layer_full_size_rows_within_one_ulp():
    """Qwen3-30B-A3B gate_up layer (4096 tokens, 128 experts, top-8): the
    whole permutation bit-exact, and 2048 sampled permuted rows plus every
    row of the smallest and the largest non-empty expert within one BF16 ulp
    of the exact product."""
    d = _inputs("gate_up")
    c = d["cfg"]
    T, H, E, k, I = c["T"], c["H"], c["E"], c["k"], c["I"]
    wgu = M.quantize(bf16_dev(d["w_gate_up"]), per_group=True)
    mlp = M.MoEMLP(T, H, I, E, k)
    mlp.permute_quant(bf16_dev(d["x"]), np_dev(d["topk_ids"]), np_dev(d["topk_w"]))
    M.minite_grouped_gemm_nvfp4(mlp.a_codes, mlp.a_sf, mlp.a_g, wgu["codes"], wgu["sf"], wgu["g"],
                                mlp.offsets, mlp.sf_offsets, mlp.gate_up, mlp.status)
    torch.cuda.synchronize()
    assert int(mlp.status.item()) == 0
    ref = O.moe_permute_quant(d["x"], d["topk_ids"], d["topk_w"], E)
    off = ref["expert_offsets"]
    Mu = int(off[-1])
    assert np.array_equal(mlp.offsets.cpu().numpy(), off)
    assert np.array_equal(mlp.a_codes.cpu().numpy()[:Mu], ref["codes"])
    counts = np.diff(off)
    nz = np.nonzero(counts)[0]
    e_small = nz[np.argmin(counts[nz])]
    e_large = nz[np.argmax(counts[nz])]
    rng = np.random.default_rng(3)
    rows = np.unique(np.concatenate([rng.choice(Mu, 2048, replace=False),
                                     np.arange(off[e_small], off[e_small + 1]),
                                     np.arange(off[e_large], off[e_large + 1]), [0, Mu - 1]]))
    wq = _oracle_weights("gate_up")[0]
    y, _ = O.grouped_gemm_exact(ref["codes"], ref["sf"], ref["row_g"], wq[0], wq[1], wq[3], off,
                                rows=rows)
    assert_bf16_within_one_ulp(u16(take(mlp.gate_up, rows)), y, "gate_up rows")


def test_mlp_forward_full_size_stagewise_on_sampled_tokens():
    """Full Qwen3-30B-A3B expert-MLP forward (4096 tokens): 64 sampled
    tokens (512 permuted rows) through every stage."""
    d = _inputs("mlp")
    c = d["cfg"]
    T, H, E, k, I = c["T"], c["H"], c["E"], c["k"], c["I"]
    wgu = M.quantize(bf16_dev(d["w_gate_up"]), per_group=True)
    wd = M.quantize(bf16_dev(d["w_down"]), per_group=True)
    mlp = M.MoEMLP(T, H, I, E, k)
    mlp.forward(bf16_dev(d["x"]), np_dev(d["topk_ids"]), np_dev(d["topk_w"]), wgu, wd)
    torch.cuda.synchronize()
    assert int(mlp.status.item()) == 0
    rng = np.random.default_rng(5)
    tok = np.sort(rng.choice(T, 64, replace=False))
    check_forward_stagewise(d, tok, _oracle_weights("mlp"), mlp, wgu, wd, mlp.status)


def test_benchmarked_step_full_size_stagewise_on_sampled_tokens():
    """The step the benchmark times: the skewed 32768-token layer (weight
    quantization, permutation, both GEMMs, SwiGLU, combine, the combine
    backward with dY quantization and the down projection's dgrad GEMM),
    captured as one CUDA graph and replayed. 48 sampled tokens (384 permuted
    rows) through every forward stage, then their dgrad rows
    dH = dY_hat W_down_hat within one BF16 ulp of the exact product."""
    import bench
    d = _inputs("skewed")
    c = d["cfg"]
    T, E = c["T"], c["E"]
    dev = torch.device("cuda", 0)
    step = bench.Step(d, dev)
    s = torch.cuda.current_stream(dev)
    step.run(s)
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(s)
    with torch.cuda.graph(graph, stream=cap):
        step.run(torch.cuda.current_stream(dev))
    s.wait_stream(cap)
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    wq = _oracle_weights("skewed")
    rng = np.random.default_rng(11)
    tok = np.sort(rng.choice(T, 48, replace=False))
    # the dgrad rows first (the forward checks below relaunch stages in place)
    pq = O.moe_permute_quant(d["dy"][tok], d["topk_ids"][tok], None, E)
    wdT = O.quantize_weights(d["w_down"], along_rows=True)
    dh_s, _ = O.grouped_gemm_exact(pq["codes"], pq["sf"], pq["row_g"], wdT[0], wdT[1], wdT[3],
                                   pq["expert_offsets"])
    full = O.moe_permute(d["topk_ids"], E)
    gpu_rows = full["dest_row"][tok].ravel()
    mini_rows = pq["dest_row"].ravel()
    assert (gpu_rows >= 0).all() and (mini_rows >= 0).all()
    assert_bf16_within_one_ulp(u16(take(step.dh, gpu_rows)), dh_s[mini_rows], "dH rows")
    check_forward_stagewise(d, tok, wq, step.mlp, step.wgu, step.wd, step.status)
