"""Expert parallelism for the W4A4 MoE expert MLP: the all-to-all exchange of
NVFP4 rows between ranks that own disjoint ranges of experts.

The miniTE report (summary page, section "Respect the timing boundaries")
quotes learner timings on 8 GPUs that include communication; sharding the
experts over ranks puts an all-to-all of the permuted rows on the path.
Per-token activation scaling (section "Follow the numerical execution path")
makes a permuted row's E2M1 codes, E4M3 block scales and FP32 global scale a
function of its token alone, so a row is quantized where its token lives
and travels in NVFP4: H/2 + H/16 + 8 bytes per row (codes, scales, global
scale, routing weight) instead of the 2H bytes of a BF16 row, 3.5x less at
H = 2048. The receiving rank does not requantize: its GEMM inputs are
bit-identical to those a single rank holding every token would build for
the same experts, and so are the outputs that travel back.

Layout (a reading; the pages give none):
  * rank r owns experts [e0(r), e1(r)) of a near-even split
    (``expert_ranges``); a sender's permuted rows are sorted by expert, so
    the rows bound for one rank form one contiguous range;
  * received rows are ordered by (expert, source rank, the source's order).
    When the batch is split over ranks by token (rank r holds tokens
    [r*T/R, (r+1)*T/R)) this is the single-rank order (expert, token, slot);
  * scales travel row-major (16-element blocks along the row) and are
    placed in the receiving rank's own per-expert 128-row padded regions of
    512-byte atoms, the layout every GEMM operand here uses.

The functions take torch tensors and use torch.distributed collectives
(NCCL on GPUs, gloo in the CPU tests). They only move bytes: slicing, the
two all-to-alls and the index gathers between the swizzled scale layout
and row-major order; no arithmetic of the method happens here. The split
sizes are read on the host (one small device-to-host copy per exchange).
Not measured on hardware: every run of this build has one GPU.
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def expert_ranges(E: int, world: int):
    """[(e0, e1)] per rank: E experts split as evenly as possible, the first
    E % world ranks taking one more."""
    base, rem = divmod(E, world)
    out, e = [], 0
    for r in range(world):
        n = base + (1 if r < rem else 0)
        out.append((e, e + n))
        e += n
    return out


def _kc(cols16: int) -> int:
    return (cols16 + 3) // 4 * 4


def sf_byte_offsets(padded_rows: torch.Tensor, cols16: int) -> torch.Tensor:
    """Byte offsets [n, cols16] of the scale of (padded row, block column) in
    the 128-row x 4-column atom layout: atom (row / 128) * (kc / 4) + col / 4
    of 512 bytes, then (row % 32) * 16 + ((row % 128) / 32) * 4 + col % 4,
    with kc = cols16 rounded up to 4."""
    kc = _kc(cols16)
    r = padded_rows.to(torch.int64)[:, None]
    c = torch.arange(cols16, dtype=torch.int64, device=padded_rows.device)[None, :]
    return (((r // 128) * (kc // 4) + c // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4
            + c % 4)


def _padded_rows(rows: torch.Tensor, expert_offsets: torch.Tensor,
                 sf_row_offsets: torch.Tensor) -> torch.Tensor:
    """Row of each permuted row inside the per-expert padded scale regions."""
    e = torch.searchsorted(expert_offsets, rows, right=True) - 1
    return sf_row_offsets[e] + (rows - expert_offsets[e])


def _bytes(t: torch.Tensor) -> torch.Tensor:
    return t.contiguous().view(torch.uint8).reshape(t.shape[0], -1)


def dispatch(codes, sf_swizzled, row_g, perm_w, expert_offsets, sf_row_offsets, H: int,
             group=None):
    """Send this rank's permuted NVFP4 rows to the ranks owning their experts.

    codes uint8 [M, H/2], sf_swizzled uint8 (per-expert padded regions),
    row_g float32 [M], perm_w float32 [M] or None, expert_offsets / sf_row_offsets
    int32 [E+1] (as the permutation produces them; rows at or beyond
    expert_offsets[E] are unused). Returns the rows of this rank's experts:
    dict(codes, sf_swizzled, row_g, perm_w, expert_offsets, sf_row_offsets,
    experts=(e0, e1), plan) with the offsets local to [e0, e1) and the
    scale capacity (rows + 128 * local experts) * kc bytes; `plan` is what
    ``combine`` needs to send the experts' outputs back."""
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    dev = codes.device
    off = expert_offsets.to(torch.int64).cpu()
    sfo = sf_row_offsets.to(torch.int64).cpu()
    E = off.numel() - 1
    ranges = expert_ranges(E, world)
    e0, e1 = ranges[rank]
    El = e1 - e0
    C16 = H // 16
    # rows per destination rank, and per (destination) expert
    send_rows = [int(off[b] - off[a]) for a, b in ranges]
    counts = (off[1:] - off[:-1]).to(torch.int64)
    recv_counts = torch.empty(world * El, dtype=torch.int64)
    dist.all_to_all_single(recv_counts, counts, output_split_sizes=[El] * world,
                           input_split_sizes=[b - a for a, b in ranges], group=group)
    recv_counts = recv_counts.view(world, El)
    recv_rows = [int(v) for v in recv_counts.sum(dim=1).tolist()]
    # one record per row: codes | row-major scales | global scale | routing weight
    Mu = int(off[E])
    if perm_w is None:  # rows without routing weights (the permutation of dY)
        perm_w = torch.zeros(Mu, dtype=torch.float32, device=dev)
    rows = torch.arange(Mu, dtype=torch.int64)
    pos = sf_byte_offsets(_padded_rows(rows, off, sfo), C16).to(dev)
    sf_rows = sf_swizzled.reshape(-1)[pos.reshape(-1)].reshape(Mu, C16)
    rec = torch.cat([codes[:Mu].reshape(Mu, H // 2), sf_rows, _bytes(row_g[:Mu].reshape(Mu, 1)),
                     _bytes(perm_w[:Mu].reshape(Mu, 1))], dim=1).contiguous()
    RB = rec.shape[1]
    got = torch.empty((sum(recv_rows), RB), dtype=torch.uint8, device=dev)
    dist.all_to_all_single(got.view(-1), rec.view(-1),
                           output_split_sizes=[n * RB for n in recv_rows],
                           input_split_sizes=[n * RB for n in send_rows], group=group)
    # received blocks by source; order them by (expert, source, source order)
    block0 = torch.cumsum(torch.tensor([0] + recv_rows[:-1], dtype=torch.int64), 0)
    within = torch.cumsum(torch.cat([torch.zeros(world, 1, dtype=torch.int64), recv_counts], 1),
                          1)[:, :-1]
    pieces = []
    for e in range(El):
        for q in range(world):
            n = int(recv_counts[q, e])
            if n:
                s = int(block0[q] + within[q, e])
                pieces.append(torch.arange(s, s + n, dtype=torch.int64))
    order = torch.cat(pieces) if pieces else torch.zeros(0, dtype=torch.int64)
    local = got[order.to(dev)]
    lcount = recv_counts.sum(dim=0)
    loff = torch.cat([torch.zeros(1, dtype=torch.int64), torch.cumsum(lcount, 0)])
    lsfo = torch.cat([torch.zeros(1, dtype=torch.int64), torch.cumsum((lcount + 127) // 128 * 128, 0)])
    Ml = int(loff[-1])
    kc = _kc(C16)
    sf_out = torch.zeros((Ml + 128 * El) * kc, dtype=torch.uint8, device=dev)
    if Ml:
        lpos = sf_byte_offsets(_padded_rows(torch.arange(Ml, dtype=torch.int64), loff, lsfo), C16)
        sf_out[lpos.to(dev).reshape(-1)] = local[:, H // 2:H // 2 + C16].reshape(-1)
    b0 = H // 2 + C16
    return dict(
        codes=local[:, :H // 2].contiguous(),
        sf_swizzled=sf_out,
        row_g=local[:, b0:b0 + 4].contiguous().view(torch.float32).reshape(-1),
        perm_w=local[:, b0 + 4:b0 + 8].contiguous().view(torch.float32).reshape(-1),
        expert_offsets=loff.to(torch.int32).to(dev),
        sf_row_offsets=lsfo.to(torch.int32).to(dev),
        experts=(e0, e1),
        plan=dict(order=order, send_rows=send_rows, recv_rows=recv_rows, group=group),
    )


def combine(expert_out, plan):
    """Send the outputs of this rank's expert rows (in ``dispatch``'s local
    order, [M_local, N] of any dtype) back to the ranks their tokens live
    on. Returns [M, N] of the same dtype: this rank's own permuted rows (the
    order of the permutation it dispatched), ready for the combine into
    token order. The rows travel as raw bytes."""
    group = plan["group"]
    order = plan["order"].to(expert_out.device)
    # back to the received order (blocks by source rank)
    back = torch.empty_like(expert_out)
    back[order] = expert_out
    src = _bytes(back) if back.shape[0] else back.reshape(0, 0).to(torch.uint8)
    rb = expert_out.shape[1] * expert_out.element_size()
    out = torch.empty((sum(plan["send_rows"]), rb), dtype=torch.uint8, device=back.device)
    dist.all_to_all_single(out.view(-1), src.contiguous().view(-1),
                           output_split_sizes=[n * rb for n in plan["send_rows"]],
                           input_split_sizes=[n * rb for n in plan["recv_rows"]], group=group)
    return out.view(expert_out.dtype).reshape(-1, expert_out.shape[1])
