"""Lane sharding across ranks, on CPU with the gloo backend (world sizes 2 and 4).

Each rank verifies a contiguous lane range of one round with the CPU oracle,
using lane_base = its first lane; the gathered results must equal the oracle
on the unsplit round.  The max-over-ranks reduction of step times that the
benchmark uses is checked as well.
"""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from speculative_decoding_verify_bf16_gb300.sharding import lane_range, shard_rows


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _round():
    import workloads
    return workloads.make_custom_round(5, "cpu", lanes=9, vocab=300, kmax=6, dtype="bf16",
                                       sampled="mixed")


def _oracle(r, lanes=None, lane_base=0, rows=None):
    import oracle
    bits = lambda t: t.view(torch.int16).numpy().view(np.uint16)
    tgt = oracle.decode_bf16(bits(r.target))
    drf = oracle.decode_bf16(bits(r.draft)) if r.draft is not None else None
    return tgt, drf


def _worker(rank, world, port, out_path):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
    import oracle
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r = _round()
    tgt, drf = _oracle(r)
    lo, hi = lane_range(r.lanes, world, rank)
    row_lo, row_hi, offs = shard_rows(r.row_offsets.tolist(), lo, hi)
    res = oracle.verify_round(tgt[row_lo:row_hi], drf[row_lo:row_hi] if drf is not None else None,
                              r.draft_tokens.numpy()[row_lo:row_hi], r.draft_lens.numpy()[lo:hi], offs,
                              r.temperatures.numpy()[lo:hi], seed=r.seed, lane_base=lo)
    # gather committed counts (lanes) and tokens (rows), padded to the largest part
    committed = torch.full((r.lanes,), -9, dtype=torch.int32)
    tokens = torch.full((r.rows,), -9, dtype=torch.int32)
    committed[lo:hi] = torch.from_numpy(res.committed)
    tokens[row_lo:row_hi] = torch.from_numpy(res.out_tokens)
    parts_c = [torch.empty_like(committed) for _ in range(world)]
    parts_t = [torch.empty_like(tokens) for _ in range(world)]
    dist.all_gather(parts_c, committed)
    dist.all_gather(parts_t, tokens)
    # each rank contributes a step time; the benchmark takes the maximum
    t = torch.tensor([1.5 + rank], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    if rank == 0:
        c = torch.stack(parts_c).max(0).values
        tok = torch.stack(parts_t).max(0).values
        torch.save({"committed": c, "tokens": tok, "tmax": t.item()}, out_path)
    dist.barrier()
    dist.destroy_process_group()


def test_lane_range_partitions():
    for lanes in [0, 1, 7, 8, 9, 128]:
        for world in [1, 2, 3, 8]:
            ranges = [lane_range(lanes, world, r) for r in range(world)]
            assert ranges[0][0] == 0 and ranges[-1][1] == lanes
            assert all(a[1] == b[0] for a, b in zip(ranges, ranges[1:]))
            sizes = [h - l for l, h in ranges]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        lane_range(4, 2, 2)


@pytest.mark.parametrize("world", [2, 4])
def test_gloo_ranks_reproduce_the_unsplit_round(tmp_path, world):
    """9 lanes over 2 ranks (5 + 4) or 4 ranks (3 + 2 + 2 + 2)."""
    import oracle
    out = str(tmp_path / "gathered.pt")
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    got = torch.load(out)
    r = _round()
    tgt, drf = _oracle(r)
    full = oracle.verify_round(tgt, drf, r.draft_tokens.numpy(), r.draft_lens.numpy(),
                               r.row_offsets.numpy(), r.temperatures.numpy(), seed=r.seed)
    assert np.array_equal(got["committed"].numpy(), full.committed)
    assert np.array_equal(got["tokens"].numpy(), full.out_tokens)
    assert got["tmax"] == 1.5 + (world - 1)
