"""The allocation-free permutation entry point.

Some callers cannot allocate device memory where they run the permutation
(a fixed memory plan, a plugin that only receives its inputs and outputs, a
loop that must not enter the allocator). minite_moe_permute_quant_noalloc
serves them with a scratch array built into the library. Its results must be
identical to the workspace entry point's, call after call, since every call
reuses the same array. This file is collected last so that a failure here
leaves every other test already run.
"""
import ctypes

import numpy as np
import pytest
import torch

from nvfp4_w4a4_moe_permute_gb300 import inputs as IN
from nvfp4_w4a4_moe_permute_gb300 import minite as M

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from nvfp4_w4a4_moe_permute_gb300 import build
    build.build()
    M.load()
    yield


def _outputs(T, H, E, k, dev):
    M_ = T * k
    kc = (H // 16 + 3) // 4 * 4
    return dict(
        codes=torch.full((M_, H // 2), 0x5A, dtype=torch.uint8, device=dev),
        sf=torch.full(((M_ + 128 * E) * kc,), 0x5A, dtype=torch.uint8, device=dev),
        row_g=torch.full((M_,), -1.0, dtype=torch.float32, device=dev),
        offsets=torch.full((E + 1,), -7, dtype=torch.int32, device=dev),
        sf_offsets=torch.full((E + 1,), -7, dtype=torch.int32, device=dev),
        perm_src=torch.full((M_,), -7, dtype=torch.int32, device=dev),
        dest_row=torch.full((T, k), -7, dtype=torch.int32, device=dev),
        perm_w=torch.full((M_,), -1.0, dtype=torch.float32, device=dev),
        status=torch.zeros(1, dtype=torch.int32, device=dev),
    )


def _run(fn_name, x, ids, w, E, out, ws=None):
    args = [x, ids, w, E, out["codes"], out["sf"], out["row_g"], out["offsets"], out["sf_offsets"],
            out["perm_src"], out["dest_row"], out["perm_w"]]
    if ws is not None:
        M.minite_moe_permute_quant(*args, ws, out["status"])
    else:
        M.minite_moe_permute_quant_noalloc(*args, out["status"])


def test_noalloc_permute_matches_workspace_entry_point_on_consecutive_calls():
    dev = torch.device("cuda:0")
    for call, (name, T) in enumerate([("gate_up", 4096), ("tiny", None), ("gate_up", 1000)]):
        d = IN.make_moe_inputs(name, seed=call, T=T, with_weights=False)
        c = d["cfg"]
        T, H, E, k = c["T"], c["H"], c["E"], c["k"]
        x = torch.from_numpy(d["x"].view(np.int16)).view(torch.bfloat16).to(dev)
        ids = torch.from_numpy(d["topk_ids"]).to(dev)
        w = torch.from_numpy(d["topk_w"]).to(dev)
        ref = _outputs(T, H, E, k, dev)
        ws = torch.empty(M.minite_workspace_bytes(M.OP_PERMUTE_QUANT, T, H, E, k),
                         dtype=torch.uint8, device=dev)
        _run("ws", x, ids, w, E, ref, ws)
        got = _outputs(T, H, E, k, dev)
        _run("noalloc", x, ids, w, E, got)
        torch.cuda.synchronize()
        for key in ref:
            assert torch.equal(ref[key], got[key]), f"call {call}: {key} differs"
        assert int(got["status"].item()) == 0


def test_noalloc_repeat_of_the_same_shape_with_new_routing():
    """Two calls in a row with the same shape (100000 tokens over 128
    experts, so the per-chunk histograms take about 0.8 MiB of the array)
    but different routing and inputs: anything the first call left in the
    shared array that the second call failed to rewrite would show here,
    since the shapes do not change. Outputs start from sentinels each time."""
    dev = torch.device("cuda:0")
    T, H, E, k = 100000, 64, 128, 8
    assert (1 << 19) < 4 * E * -(-T // (512 // k)) < (2 << 20)
    for seed in (21, 22):
        rng = np.random.default_rng(seed)
        x = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).to(dev).to(torch.bfloat16)
        ids_np, w_np = IN.topk_softmax_routing(rng.standard_normal((T, E)).astype(np.float32), k)
        ids = torch.from_numpy(ids_np).to(dev)
        w = torch.from_numpy(w_np).to(dev)
        ref = _outputs(T, H, E, k, dev)
        ws = torch.empty(M.minite_workspace_bytes(M.OP_PERMUTE_QUANT, T, H, E, k),
                         dtype=torch.uint8, device=dev)
        _run("ws", x, ids, w, E, ref, ws)
        got = _outputs(T, H, E, k, dev)
        _run("noalloc", x, ids, w, E, got)
        torch.cuda.synchronize()
        for key in ref:
            assert torch.equal(ref[key], got[key]), f"seed {seed}: {key} differs"
        assert int(got["status"].item()) == 0


def test_noalloc_scatters_scales_directly_when_token_order_staging_does_not_fit():
    """T * (H/16 + 4) bytes of token-order scales exceed the 2 MiB array here,
    so the allocation-free entry writes each token's scales straight to its
    rows; the results must still equal the workspace entry point's."""
    dev = torch.device("cuda:0")
    T, H, E, k = 20000, 2048, 8, 2
    rng = np.random.default_rng(5)
    xf = rng.standard_normal((T, H)).astype(np.float32)
    x = torch.from_numpy(xf).to(dev).to(torch.bfloat16)
    ids = torch.from_numpy(np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)).to(dev)
    w = torch.from_numpy(rng.random((T, k)).astype(np.float32)).to(dev)
    assert M.minite_workspace_bytes(M.OP_PERMUTE_QUANT, T, H, E, k) > (2 << 20)
    ref = _outputs(T, H, E, k, dev)
    ws = torch.empty(M.minite_workspace_bytes(M.OP_PERMUTE_QUANT, T, H, E, k),
                     dtype=torch.uint8, device=dev)
    _run("ws", x, ids, w, E, ref, ws)
    got = _outputs(T, H, E, k, dev)
    _run("noalloc", x, ids, w, E, got)
    torch.cuda.synchronize()
    for key in ref:
        assert torch.equal(ref[key], got[key]), f"{key} differs"
    assert int(got["status"].item()) == 0


def test_noalloc_rejects_problems_beyond_its_scratch():
    lib = M.load()
    fake = ctypes.c_void_p(4096)  # never dereferenced: the size check comes first
    T, H, E, k = 65536, 2048, 1024, 8
    assert M.minite_workspace_bytes(M.OP_PERMUTE_QUANT, T, H, E, k) > (2 << 20)
    rc = lib.minite_moe_permute_quant_noalloc(fake, fake, None, T, H, E, k, fake, fake, fake, fake,
                                              fake, fake, fake, None, None, None)
    assert rc == 6
    assert "scratch" in M.minite_status_string(rc)
