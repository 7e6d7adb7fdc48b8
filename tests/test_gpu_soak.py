"""Determinism under load: every workload's CUDA graph (hundreds of launches
overlapping through programmatic dependent launch) is replayed for a few
seconds, and every replay must reproduce the first replay's outputs bit for
bit with every lane status OK.  Races in the ring or the exchange barriers
show up here as sporadic differences or time-outs."""

import time

import pytest
import torch

import bench
import workloads

import speculative_decoding_verify_bf16_gb300 as sv

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)
SECONDS_PER_WORKLOAD = 2.0


@pytest.mark.parametrize("name", workloads.WORKLOADS)
def test_graph_replays_are_deterministic(name):
    sv.build_library()
    sv.load_library()
    stream = torch.cuda.Stream()
    b = bench.Bench(name, 1, DEV, 0)
    with torch.cuda.stream(stream):
        for i in range(len(b.sets)):
            b.step(i, stream)
    torch.cuda.synchronize()
    steps = 10 if b.has_state else 200
    g = b.capture(steps, stream)
    with torch.cuda.stream(stream):
        g.replay()
    stream.synchronize()
    ref = [{k: v.clone() for k, v in o.items()} for o in b.outs]
    for o in ref:
        assert (o["status"] == 0).all()
    t0, reps = time.time(), 0
    while time.time() - t0 < SECONDS_PER_WORKLOAD:
        with torch.cuda.stream(stream):
            g.replay()
        stream.synchronize()
        reps += 1
        for j, (o, r) in enumerate(zip(b.outs, ref)):
            for k in ("committed", "out_tokens", "status"):
                assert torch.equal(o[k], r[k]), (name, reps, j, k)
    assert reps > 0
    if b.has_state:
        # the sets share one recurrent state: it holds what the graph's last
        # commit wrote, staged column committed - 1 of that step's set
        j = (steps - 1) % len(b.sets)
        s, o = b.sets[j], b.outs[j]
        for lane in (0, s.lanes // 2, s.lanes - 1):
            c = int(o["committed"][lane])
            assert torch.equal(s.live[lane], s.staged[lane, c - 1]), (lane, c)
