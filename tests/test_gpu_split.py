"""GPU parity of the work-list form of the verify kernel (a workspace given):
against the oracle, against the cluster form, and the workspace protocol
(counters zero before a launch and after it, one workspace shared by
back-to-back launches)."""

import numpy as np
import pytest
import torch

import workloads
import speculative_decoding_verify_bf16_gb300 as sv
from gpu_harness import compare, run_gpu, run_oracle, workspace_counters, workspace_for
from test_gpu_verify import SMALL_CASES

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    sv.build_library()
    sv.load_library()


def _run_split(r, **kw):
    ws = workspace_for(r)
    g = run_gpu(r, workspace=ws, **kw)
    assert int(workspace_counters(ws, r.lanes).count_nonzero()) == 0, "a launch leaves its counters zero"
    return g


@pytest.mark.parametrize("stats", [True, False], ids=["stats", "nostats"])
@pytest.mark.parametrize("case", SMALL_CASES, ids=lambda c: f"V{c[0]}-k{c[1]}-B{c[2]}-{c[3]}-{c[4]}")
def test_small_shapes_match_oracle(case, stats):
    vocab, kmax, lanes, dtype, sampled, fixed_k, seed = case
    r = workloads.make_custom_round(seed, DEV, lanes=lanes, vocab=vocab, kmax=kmax, dtype=dtype,
                                    sampled=sampled, fixed_k=fixed_k)
    compare(r, _run_split(r, stats=stats), run_oracle(r), check_stats=stats)


@pytest.mark.parametrize("launch", ["stats", "bench"])
@pytest.mark.parametrize("name", workloads.WORKLOADS)
def test_named_workloads_full_size(name, launch):
    """Every workload at full size through the work-list form, with row_stats
    and as the bench launches it (no row_stats, metadata before the wait)."""
    r = workloads.make_round(name, seed=7, device=DEV)
    bench_launch = launch == "bench"
    g = _run_split(r, stats=not bench_launch, meta_before_wait=bench_launch)
    counts = compare(r, g, run_oracle(r), check_stats=not bench_launch)
    print(name, launch, counts)


@pytest.mark.parametrize("sampled", ["none", "mixed", "all"])
def test_split_and_cluster_forms_agree(sampled):
    """Greedy lanes are bit-identical between the two forms (argmax does not
    depend on how the vocabulary is split); every lane matches the oracle."""
    r = workloads.make_custom_round(44, DEV, lanes=13, vocab=70001, kmax=7, dtype="bf16", sampled=sampled)
    orc = run_oracle(r)
    a = run_gpu(r)
    b = _run_split(r)
    compare(r, a, orc)
    compare(r, b, orc)
    greedy = r.temperatures.cpu().numpy() <= 0
    np.testing.assert_array_equal(a["committed"][greedy], b["committed"][greedy])
    np.testing.assert_array_equal(a["argmax"], b["argmax"])
    np.testing.assert_array_equal(a["max_logit"], b["max_logit"])
    np.testing.assert_array_equal(a["lane_status"], b["lane_status"])


@pytest.mark.parametrize("chunk_kb,grid", [("8", "0"), ("24", "0"), ("8", "1"), ("16", "7"), ("24", "3")])
def test_chunk_and_grid_overrides_change_nothing(monkeypatch, chunk_kb, grid):
    """Other chunk sizes and CTA counts (one CTA doing everything included)
    give the same greedy results and match the oracle."""
    r = workloads.make_custom_round(45, DEV, lanes=9, vocab=40000, kmax=6, dtype="bf16", sampled="mixed")
    ref = _run_split(r)
    monkeypatch.setenv("SPEC_SPLIT_CHUNK_KB", chunk_kb)
    monkeypatch.setenv("SPEC_SPLIT_GRID", grid)
    g = _run_split(r)
    compare(r, g, run_oracle(r))
    greedy = r.temperatures.cpu().numpy() <= 0
    np.testing.assert_array_equal(ref["committed"][greedy], g["committed"][greedy])
    np.testing.assert_array_equal(ref["argmax"], g["argmax"])


@pytest.mark.parametrize("stats", [True, False], ids=["stats", "nostats"])
def test_nonfinite_rows_and_statuses(stats):
    r = workloads.make_custom_round(3, DEV, lanes=5, vocab=20000, kmax=3, dtype="bf16", sampled="all",
                                    fixed_k=True)
    off = r.row_offsets.cpu().numpy()
    r.target[off[1] + 2, 7] = float("nan")
    r.target[off[2] + 0, 19997] = float("inf")
    r.target[off[3] + 1, :] = float("-inf")
    r.draft[off[4] + 0, 10000] = float("nan")
    r.draft[off[0] + 3, 5] = float("nan")  # a lane's last drafter row: never read
    g = _run_split(r, stats=stats)
    assert g["lane_status"].tolist() == [0, 4, 4, 4, 4]
    compare(r, g, run_oracle(r), check_stats=stats)
    r = workloads.make_custom_round(4, DEV, lanes=4, vocab=64, kmax=3, dtype="bf16", sampled="none", fixed_k=True)
    off = r.row_offsets.cpu().numpy()
    r.draft_tokens[off[1] + 1] = 64
    r.draft_tokens[off[2]] = -3
    g = _run_split(r)
    assert g["lane_status"].tolist() == [0, 5, 5, 0]
    compare(r, g, run_oracle(r))
    r.draft_lens[3] = 2
    g = _run_split(r)
    assert g["lane_status"].tolist() == [0, 5, 5, 6] and g["committed"][3] == 0
    r = workloads.make_custom_round(4, DEV, lanes=2, vocab=100, kmax=16, fixed_k=True, sampled="none")
    g = _run_split(r)
    assert g["lane_status"].tolist() == [2, 2] and (g["out_tokens"] == -1).all()
    r = workloads.make_custom_round(5, DEV, lanes=3, vocab=64, kmax=3, dtype="bf16", sampled="all", fixed_k=True)
    r.temperatures[0] = 0.0
    r.draft = None
    g = _run_split(r)
    assert g["lane_status"].tolist() == [0, 1, 1]


def test_negative_infinity_and_long_runs_of_it():
    r = workloads.make_custom_round(6, DEV, lanes=3, vocab=30000, kmax=4, dtype="bf16", sampled="all", fixed_k=True)
    r.target[:, :17000] = float("-inf")
    r.draft[:, :9000] = float("-inf")
    orc = run_oracle(r)
    compare(r, _run_split(r, stats=True), orc)
    compare(r, _run_split(r, stats=False), orc, check_stats=False)


def test_identical_draft_and_target_accepts_everything():
    r = workloads.make_custom_round(7, DEV, lanes=8, vocab=5000, kmax=6, dtype="bf16", sampled="all", fixed_k=True)
    r.draft = r.target.clone()
    g = _run_split(r)
    assert (g["committed"] == 7).all()
    compare(r, g, run_oracle(r))


@pytest.mark.parametrize("vocab", [1_000_003, 262144])
def test_draws_over_many_chunks(vocab):
    """Flat rows (small spread, no spike) put the draw's crossing anywhere in
    the row, across many pass-2 chunks; bf16 and fp32."""
    for seed, dtype in ((1, "bf16"), (2, "f32")):
        r = workloads.make_custom_round(800 + seed, DEV, lanes=5, vocab=vocab, kmax=3, dtype=dtype, sampled="all",
                                        fixed_k=True, sigma=0.5, spike=0.0, alpha=0.3)
        orc = run_oracle(r)
        compare(r, _run_split(r, stats=False), orc, check_stats=False)
        compare(r, _run_split(r, stats=True), orc, check_stats=True)


@pytest.mark.parametrize("meta_early", [False, True], ids=["meta-after-wait", "meta-before-wait"])
def test_back_to_back_graph_launches_share_one_workspace(meta_early):
    """40 launches captured in one CUDA graph, all with the same workspace (each
    launch must leave its counters zero for the next): every launch gives the
    first one's results, equal to the oracle's, and the counters end zero."""
    r = workloads.make_custom_round(78, DEV, lanes=12, vocab=151936, kmax=5, dtype="bf16", sampled="mixed",
                                    fixed_k=True)
    ws = workspace_for(r)
    n = 40
    outs = [(torch.zeros(r.lanes, dtype=torch.int32, device=DEV), torch.zeros(r.rows, dtype=torch.int32, device=DEV),
             torch.zeros(r.lanes, dtype=torch.int32, device=DEV)) for _ in range(n)]
    stream = torch.cuda.Stream()

    def launch(o):
        sv.spec_verify_accept(r.target, r.draft, r.draft_tokens, r.draft_lens, r.row_offsets, r.temperatures,
                              r.seed, o[0], o[1], o[2], stream=torch.cuda.current_stream(),
                              meta_before_wait=meta_early, workspace=ws)

    with torch.cuda.stream(stream):
        launch(outs[0])
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            for o in outs:
                launch(o)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert int(workspace_counters(ws, r.lanes).count_nonzero()) == 0
    first = {"committed": outs[0][0].cpu().numpy(), "out_tokens": outs[0][1].cpu().numpy(),
             "lane_status": outs[0][2].cpu().numpy()}
    compare(r, first, run_oracle(r), check_stats=False)
    for o in outs[1:]:
        assert torch.equal(o[0], outs[0][0]) and torch.equal(o[1], outs[0][1]) and torch.equal(o[2], outs[0][2])


def test_a_wait_that_never_completes_reports_a_timeout():
    """SPEC_VERIFY_TEST_WITHHOLD_COPY: the last pass-1 chunk is announced but
    never copied; its group's wait gives up after 2 s, every lane reports
    SPEC_ERR_TIMEOUT with nothing committed, the workspace's counters end zero,
    and the next launch with the same workspace matches the oracle."""
    import time

    r = workloads.make_custom_round(81, DEV, lanes=4, vocab=200000, kmax=3, dtype="bf16", sampled="mixed",
                                    fixed_k=True)
    ws = workspace_for(r)
    committed = torch.full((r.lanes,), -7, dtype=torch.int32, device=DEV)
    out = torch.full((r.rows,), -7, dtype=torch.int32, device=DEV)
    status = torch.full((r.lanes,), -7, dtype=torch.int32, device=DEV)
    torch.cuda.synchronize()
    t0 = time.time()
    sv.spec_verify_accept(r.target, r.draft, r.draft_tokens, r.draft_lens, r.row_offsets, r.temperatures, r.seed,
                          committed, out, status, test_flags=sv.SPEC_VERIFY_TEST_WITHHOLD_COPY, workspace=ws)
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    assert (status.cpu() == sv.SPEC_ERR_TIMEOUT).all(), status
    assert (committed.cpu() == 0).all() and (out.cpu() == -1).all()
    assert 1.5 < elapsed < 60, elapsed
    assert int(workspace_counters(ws, r.lanes).count_nonzero()) == 0
    g = run_gpu(r, workspace=ws)
    compare(r, g, run_oracle(r))
    assert int(workspace_counters(ws, r.lanes).count_nonzero()) == 0


def test_workspace_errors_and_the_lane_limit():
    r = workloads.make_custom_round(9, DEV, lanes=4, vocab=1000, kmax=3, dtype="bf16", sampled="mixed", fixed_k=True)
    small = torch.zeros(256, dtype=torch.uint8, device=DEV)
    with pytest.raises(sv.SpecError) as e:
        run_gpu(r, workspace=small)
    assert e.value.code == sv.SPEC_ERR_INVALID_ARG
    # more lanes than the work-list form takes: the cluster form runs instead
    r = workloads.make_custom_round(10, DEV, lanes=2100, vocab=300, kmax=2, dtype="bf16", sampled="mixed")
    ws = workspace_for(r)
    compare(r, run_gpu(r, workspace=ws), run_oracle(r))


def test_lane_shards_reproduce_the_unsplit_round():
    from speculative_decoding_verify_bf16_gb300.sharding import lane_range, shard_rows

    r = workloads.make_custom_round(92, DEV, lanes=11, vocab=50000, kmax=6, dtype="bf16", sampled="mixed")
    full = _run_split(r)
    for rank in range(3):
        lo, hi = lane_range(r.lanes, 3, rank)
        row_lo, row_hi, offs = shard_rows(r.row_offsets.tolist(), lo, hi)
        c = torch.zeros(hi - lo, dtype=torch.int32, device=DEV)
        o = torch.zeros(row_hi - row_lo, dtype=torch.int32, device=DEV)
        st = torch.zeros(hi - lo, dtype=torch.int32, device=DEV)
        ws = sv.new_workspace(hi - lo, row_hi - row_lo, r.vocab, r.target.dtype, r.target.device)
        sv.spec_verify_accept(r.target[row_lo:row_hi], r.draft[row_lo:row_hi],
                              r.draft_tokens[row_lo:row_hi].contiguous(), r.draft_lens[lo:hi].contiguous(),
                              torch.tensor(offs, dtype=torch.int32, device=DEV),
                              r.temperatures[lo:hi].contiguous(), r.seed, c, o, st, lane_base=lo, workspace=ws)
        torch.cuda.synchronize()
        assert np.array_equal(c.cpu().numpy(), full["committed"][lo:hi])
        assert np.array_equal(o.cpu().numpy(), full["out_tokens"][row_lo:row_hi])
