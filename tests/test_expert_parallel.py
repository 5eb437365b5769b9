"""Expert parallelism on CPU: world-size-2 and -3 gloo ranks, each holding a
share of the batch's tokens and a range of the experts, exchange NVFP4 rows
with ``ep.dispatch`` and send the experts' outputs back with ``ep.combine``.

The expert computation itself is the oracle's (the GPU kernels need a GPU);
what is under test is the exchange: the rows a rank receives for its
experts must be bit-identical to the single-rank permutation's rows of
those experts (codes, scales, global scales, routing weights), and every
rank's combined output must be bit-identical to the single-rank oracle
chain's output for its tokens.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.abspath(os.path.join(os.path.dirname(__file__), ".."))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _token_range(T, world, rank):
    return rank * T // world, (rank + 1) * T // world


def _rank(rank, world, port, case, T, q):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    from nvfp4_w4a4_moe_permute_gb300 import ep
    from nvfp4_w4a4_moe_permute_gb300 import inputs as IN
    from oracle import nvfp4_moe_oracle as O
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        d = IN.make_moe_inputs(case, T=T)
        c = d["cfg"]
        E, H = c["E"], c["H"]
        t0, t1 = _token_range(c["T"], world, rank)
        pq = O.moe_permute_quant(d["x"][t0:t1], d["topk_ids"][t0:t1], d["topk_w"][t0:t1], E)
        n = lambda a: torch.from_numpy(np.ascontiguousarray(a))  # noqa: E731
        got = ep.dispatch(n(pq["codes"]), n(pq["sf_swizzled"]), n(pq["row_g"]), n(pq["perm_w"]),
                          n(pq["expert_offsets"]), n(pq["sf_row_offsets"]), H)
        e0, e1 = got["experts"]
        loff = got["expert_offsets"].numpy().astype(np.int64)
        lsfo = got["sf_row_offsets"].numpy().astype(np.int64)
        codes = got["codes"].numpy()
        g = got["row_g"].numpy()
        pw = got["perm_w"].numpy()
        # row-major scales of the received rows, read back from their local regions
        kc = (H // 16 + 3) // 4 * 4
        sf = np.zeros((codes.shape[0], H // 16), dtype=np.uint8)
        buf = got["sf_swizzled"].numpy()
        for e in range(e1 - e0):
            a, b = loff[e], loff[e + 1]
            if b > a:
                sf[a:b] = O.unswizzle_sf(buf[lsfo[e] * kc:], b - a, H // 16)
        # the experts' computation (oracle) on the received rows
        wgu = O.quantize_weights(d["w_gate_up"][e0:e1])
        wd = O.quantize_weights(d["w_down"][e0:e1])
        gu, _ = O.grouped_gemm_exact(codes, sf, g, wgu[0], wgu[1], wgu[3], loff)
        sw = O.swiglu_weighted_quant(O.f64_to_bf16(gu), pw, loff, lsfo)
        dn, _ = O.grouped_gemm_exact(sw["codes"], sw["sf"], sw["row_g"], wd[0], wd[1], wd[3], loff)
        back = ep.combine(n(O.f64_to_bf16(dn)).view(torch.int16).view(torch.bfloat16), got["plan"])
        back_u16 = back.view(torch.int16).numpy().view(np.uint16)
        y = O.moe_combine(back_u16, pq["dest_row"])
        q.put((rank, dict(experts=(e0, e1), codes=codes, sf=sf, g=g, pw=pw, loff=loff, y=y,
                          sent_rows=int(pq["expert_offsets"][-1]), back_rows=back_u16.shape[0])))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,case,T", [(2, "tiny", None), (3, "tiny", 61), (2, "tiny", 7)])
def test_dispatch_and_combine_match_the_single_rank_chain(world, case, T):
    sys.path.insert(0, ROOT)
    from nvfp4_w4a4_moe_permute_gb300 import inputs as IN
    from oracle import nvfp4_moe_oracle as O
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, case, T, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=300) for _ in range(world))
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    # the single-rank reference: every token, every expert
    d = IN.make_moe_inputs(case, T=T)
    c = d["cfg"]
    E = c["E"]
    full = O.moe_permute_quant(d["x"], d["topk_ids"], d["topk_w"], E)
    ref = O.moe_mlp_forward(d["x"], d["topk_ids"], d["topk_w"], E,
                            O.quantize_weights(d["w_gate_up"]), O.quantize_weights(d["w_down"]))
    off = full["expert_offsets"]
    covered = []
    for r in range(world):
        got = res[r]
        e0, e1 = got["experts"]
        covered += list(range(e0, e1))
        rows = np.arange(off[e0], off[e1])
        # received rows == the single-rank permutation's rows of these experts
        assert np.array_equal(got["loff"], off[e0:e1 + 1] - off[e0])
        assert np.array_equal(got["codes"], full["codes"][rows])
        assert np.array_equal(got["sf"], full["sf"][rows])
        assert np.array_equal(got["g"].view(np.uint32), full["row_g"][rows].view(np.uint32))
        assert np.array_equal(got["pw"].view(np.uint32), full["perm_w"][rows].view(np.uint32))
        # every row a rank sent came back
        assert got["back_rows"] == got["sent_rows"]
        # and its tokens' outputs equal the single-rank chain's, bit for bit
        t0, t1 = _token_range(c["T"], world, r)
        assert np.array_equal(got["y"], ref["y"][t0:t1])
    assert covered == list(range(E))


def test_expert_ranges_cover_the_experts_evenly():
    sys.path.insert(0, ROOT)
    from nvfp4_w4a4_moe_permute_gb300 import ep
    for E, world in [(128, 8), (5, 2), (4, 3), (3, 4)]:
        r = ep.expert_ranges(E, world)
        assert r[0][0] == 0 and r[-1][1] == E
        assert all(a1 == b0 for (_, a1), (b0, _) in zip(r, r[1:]))
        sizes = [b - a for a, b in r]
        assert max(sizes) - min(sizes) <= 1


def test_record_bytes_per_row_are_nvfp4_not_bf16():
    """A dispatched row carries H/2 code bytes, H/16 scale bytes, its global
    scale and its routing weight: 1160 bytes at H = 2048 against 4096 for a
    BF16 row."""
    H = 2048
    assert H // 2 + H // 16 + 4 + 4 == 1160
    assert 2 * H / (H // 2 + H // 16 + 8) > 3.5
