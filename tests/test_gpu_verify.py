"""GPU parity: the fused verify kernel against the CPU oracle, through the C ABI."""

import numpy as np
import pytest
import torch

import oracle
import workloads
import speculative_decoding_verify_bf16_gb300 as sv
from gpu_harness import compare, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    sv.build_library()
    sv.load_library()


# V spans tiny vocabularies (one CTA, ragged tails shorter than a vector),
# several slices per lane, and a vocabulary that does not divide into vectors.
SMALL_CASES = [
    # (vocab, kmax, lanes, dtype, sampled, fixed_k, seed)
    (1, 3, 3, "bf16", "none", False, 1),
    (7, 4, 3, "bf16", "mixed", False, 2),
    (8, 7, 17, "bf16", "mixed", False, 3),
    (9, 2, 5, "f32", "mixed", False, 4),
    (1023, 7, 17, "bf16", "all", False, 5),
    (4097, 5, 3, "f32", "all", False, 6),
    (4097, 15, 2, "bf16", "mixed", True, 7),
    (40000, 7, 9, "bf16", "mixed", False, 8),
    (65537, 3, 1, "bf16", "all", True, 9),
    (151936, 7, 3, "bf16", "mixed", False, 10),
    (262144, 2, 2, "bf16", "all", True, 11),
    (32000, 0, 6, "bf16", "mixed", True, 12),
    (5000, 7, 33, "f32", "none", False, 13),
]


@pytest.mark.parametrize("stats", [True, False], ids=["stats", "nostats"])
@pytest.mark.parametrize("case", SMALL_CASES, ids=lambda c: f"V{c[0]}-k{c[1]}-B{c[2]}-{c[3]}-{c[4]}")
def test_small_shapes_match_oracle(case, stats):
    """Without row_stats, sampled rows take the sweep that needs no exact max."""
    vocab, kmax, lanes, dtype, sampled, fixed_k, seed = case
    r = workloads.make_custom_round(seed, DEV, lanes=lanes, vocab=vocab, kmax=kmax, dtype=dtype,
                                    sampled=sampled, fixed_k=fixed_k)
    gpu = run_gpu(r, stats=stats)
    orc = run_oracle(r)
    compare(r, gpu, orc, check_stats=stats)


@pytest.mark.parametrize("ld_extra", [8, 5, 64])
def test_padded_rows_match_oracle(ld_extra):
    """Row stride ld > V: padding (huge values) must never be read.

    ld_extra = 5 makes rows misaligned, which takes the element-wise path.
    """
    vocab = 3001
    r = workloads.make_custom_round(21, DEV, lanes=7, vocab=vocab, kmax=5, dtype="bf16",
                                    sampled="mixed", ld=vocab + ld_extra)
    assert r.target.stride(0) == vocab + ld_extra
    compare(r, run_gpu(r), run_oracle(r))


def test_misaligned_base_takes_elementwise_path():
    vocab = 20000
    r = workloads.make_custom_round(22, DEV, lanes=5, vocab=vocab, kmax=4, dtype="bf16", sampled="mixed")
    # shift both logits arrays by one element: base addresses no longer 16-byte aligned
    for name in ("target", "draft"):
        t = getattr(r, name)
        buf = torch.empty(t.numel() + 1, dtype=t.dtype, device=t.device)
        buf[1:] = t.reshape(-1)
        setattr(r, name, buf[1:].view(t.shape))
    assert r.target.data_ptr() % 16 != 0
    compare(r, run_gpu(r), run_oracle(r))


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_many_seeds_mixed(seed):
    r = workloads.make_custom_round(100 + seed, DEV, lanes=64, vocab=12000, kmax=7, dtype="bf16",
                                    sampled="mixed")
    counts = compare(r, run_gpu(r), run_oracle(r))
    print(counts)


@pytest.mark.parametrize("launch", ["stats", "bench"])
@pytest.mark.parametrize("name", workloads.WORKLOADS)
def test_named_workloads_full_size(name, launch):
    """Every workload at its full size, lane by lane against the oracle, in two
    launches: with row_stats (the exact sweep, whose per-row statistics are
    compared too), and exactly as bench.py times it -- no row_stats (sampled
    rows take the sweep that keeps no exact max) and the lane metadata read
    before the wait for the previous kernel."""
    r = workloads.make_round(name, seed=7, device=DEV)
    if name == workloads.RAGGED_MIXED_B128:
        assert sv.spec_row_budget(workloads.RAGGED_DRAFT_TOKENS, workloads.RAGGED_ROW_BUDGET,
                                  r.lanes) == workloads.RAGGED_DRAFT_TOKENS
        assert r.rows <= workloads.RAGGED_ROW_BUDGET
    bench_launch = launch == "bench"
    gpu = run_gpu(r, stats=not bench_launch, meta_before_wait=bench_launch)
    orc = run_oracle(r)
    counts = compare(r, gpu, orc, check_stats=not bench_launch)
    print(name, launch, counts)
    assert (gpu["committed"] >= 1).all()
    assert (gpu["committed"] <= r.draft_lens.cpu().numpy() + 1).all()


def test_round_uniforms_match_the_oracle_generator():
    seed = 0x0123456789ABCDEF
    u = sv.spec_round_uniforms(seed, 40, 16).cpu().numpy()
    for b in range(40):
        for j in range(16):
            ua, us = oracle.round_uniforms(seed, b, j)
            assert u[b, j, 0] == ua and u[b, j, 1] == us, (b, j)
    # large lane ids and seeds exercise the high counter and key words
    u = sv.spec_round_uniforms(2 ** 64 - 1, 3, 2, lane_base=2 ** 32 - 5).cpu().numpy()
    assert u[2, 1, 0] == oracle.round_uniforms(2 ** 64 - 1, 2 ** 32 - 3, 1)[0]
    assert u[2, 1, 1] == oracle.round_uniforms(2 ** 64 - 1, 2 ** 32 - 3, 1)[1]


def test_greedy_equals_plain_argmax_decode_on_the_gpu():
    """Rounds through the GPU kernel emit the plain argmax stream of a toy model."""
    from oracle_checks import ToyLM

    vocab, k = 300, 5
    lm = ToyLM(vocab, seed=13)
    context = [1, 2]
    plain = [lm.next_token(context)]
    while len(plain) < 80:
        plain.append(lm.next_token(context + plain))
    rng = np.random.default_rng(1)
    consumed, anchor, emitted = list(context), plain[0], [plain[0]]
    while len(emitted) < 60:
        pos = len(emitted) - 1
        drafts = [plain[pos + 1 + i] if rng.random() < 0.7 else int(rng.integers(vocab)) for i in range(k)]
        cols = [anchor] + drafts
        rows = np.stack([lm.logits(consumed + cols[:j + 1]) for j in range(k + 1)])
        target = torch.tensor(rows, dtype=torch.float32, device=DEV)
        r = workloads.RoundInputs("toy", vocab, 1, k + 1, "f32", target, None,
                                  torch.tensor(drafts + [-1], dtype=torch.int32, device=DEV),
                                  torch.tensor([k], dtype=torch.int32, device=DEV),
                                  torch.tensor([0, k + 1], dtype=torch.int32, device=DEV),
                                  torch.zeros(1, dtype=torch.float32, device=DEV), 0)
        g = run_gpu(r)
        c = int(g["committed"][0])
        toks = g["out_tokens"][:c].tolist()
        consumed += cols[:c]
        anchor = toks[-1]
        emitted += toks
    assert emitted[:60] == plain[:60]


def test_sampled_marginals_on_the_gpu():
    """Emitted tokens follow p: chi-square over many lanes sharing one set of rows."""
    from scipy import stats

    rng = np.random.default_rng(5)
    vocab, k, temp, lanes = 6, 2, 0.9, 40000
    t_rows = rng.normal(size=(k + 1, vocab)) * 1.2
    d_rows = t_rows + rng.normal(size=(k + 1, vocab))
    t_rows = np.asarray(t_rows, np.float32).astype(np.float64)
    d_rows = np.asarray(d_rows, np.float32).astype(np.float64)
    p = [np.exp(x / temp) / np.exp(x / temp).sum() for x in t_rows]
    q = [np.exp(x / temp) / np.exp(x / temp).sum() for x in d_rows]
    d1 = rng.choice(vocab, size=lanes, p=q[0])
    d2 = rng.choice(vocab, size=lanes, p=q[1])
    tok = np.full((lanes, k + 1), -1)
    tok[:, 0], tok[:, 1] = d1, d2
    f = lambda a, dt: torch.tensor(a, dtype=dt, device=DEV)
    r = workloads.RoundInputs("mc", vocab, lanes, lanes * (k + 1), "f32",
                              f(np.tile(t_rows, (lanes, 1)), torch.float32),
                              f(np.tile(d_rows, (lanes, 1)), torch.float32),
                              f(tok.reshape(-1), torch.int32), f(np.full(lanes, k), torch.int32),
                              f(np.arange(lanes + 1) * (k + 1), torch.int32),
                              f(np.full(lanes, temp), torch.float32), 99)
    g = run_gpu(r, stats=False)
    out = g["out_tokens"].reshape(lanes, k + 1)
    assert (g["lane_status"] == 0).all()
    t1 = np.bincount(out[:, 0], minlength=vocab)
    assert stats.chisquare(t1, p[0] * lanes).pvalue > 1e-4
    acc = g["committed"] >= 2
    t2 = np.bincount(out[acc, 1], minlength=vocab)
    assert stats.chisquare(t2, p[1] * acc.sum()).pvalue > 1e-4
    acc2 = g["committed"] >= 3
    t3 = np.bincount(out[acc2, 2], minlength=vocab)
    assert stats.chisquare(t3, p[2] * acc2.sum()).pvalue > 1e-4


def _tiny_round(vocab=64, k=3, lanes=4, temp=0.0, seed=3):
    return workloads.make_custom_round(seed, DEV, lanes=lanes, vocab=vocab, kmax=k, dtype="bf16",
                                       sampled="none" if temp <= 0 else "all", fixed_k=True)


@pytest.mark.parametrize("stats", [True, False], ids=["stats", "nostats"])
@pytest.mark.parametrize("vocab", [64, 20000])
def test_nonfinite_rows_fail_only_their_lane(stats, vocab):
    r = _tiny_round(vocab=vocab, lanes=5, temp=1.0)
    off = r.row_offsets.cpu().numpy()
    r.target[off[1] + 2, 7] = float("nan")
    r.target[off[2] + 0, vocab - 3] = float("inf")
    r.target[off[3] + 1, :] = float("-inf")
    r.draft[off[4] + 0, vocab // 2] = float("nan")  # a drafter row that is read
    r.draft[off[0] + 3, 5] = float("nan")          # the lane's last drafter row: never read
    gpu, orc = run_gpu(r, stats=stats), run_oracle(r)
    assert gpu["lane_status"].tolist() == [0, 4, 4, 4, 4]
    compare(r, gpu, orc, check_stats=stats)


@pytest.mark.parametrize("stats", [True, False], ids=["stats", "nostats"])
def test_negative_infinity_logits_are_allowed(stats):
    r = _tiny_round(lanes=4, temp=0.0)
    r.target[:, ::3] = float("-inf")
    compare(r, run_gpu(r, stats=stats), run_oracle(r), check_stats=stats)
    r = _tiny_round(lanes=4, temp=1.0)
    r.target[:, ::3] = float("-inf")
    r.draft[:, 1::4] = float("-inf")
    compare(r, run_gpu(r, stats=stats), run_oracle(r), check_stats=stats)
    # a sampled lane whose rows start with a long run of -inf (no reference for a while)
    r = _tiny_round(vocab=30000, lanes=3, temp=0.8)
    r.target[:, :17000] = float("-inf")
    r.draft[:, :9000] = float("-inf")
    compare(r, run_gpu(r, stats=stats), run_oracle(r), check_stats=stats)


@pytest.mark.parametrize("temp", [0.02, 0.3, 5.0])
def test_rising_and_widely_spread_rows_without_row_stats(temp):
    """Rows whose logits rise along the vocabulary (every group exceeds the
    reference the sum was taken against) or spread over thousands of log2
    units at low temperature: the sampled sweep that skips the exact max must
    still match the oracle."""
    lanes, k, vocab = 6, 4, 40000
    r = workloads.make_custom_round(91, DEV, lanes=lanes, vocab=vocab, kmax=k, dtype="bf16", sampled="all",
                                    fixed_k=True)
    rise = torch.linspace(-30.0, 30.0, vocab, device=DEV)
    for b in range(0, lanes, 2):   # even lanes: rising rows, odd lanes: very wide noise
        rows = slice(b * (k + 1), (b + 1) * (k + 1))
        r.target[rows] = (rise + r.target[rows].float() * 0.1).to(r.target.dtype)
        r.draft[rows] = (rise + r.draft[rows].float() * 0.1).to(r.draft.dtype)
    for b in range(1, lanes, 2):
        rows = slice(b * (k + 1), (b + 1) * (k + 1))
        r.target[rows] = (r.target[rows].float() * 40.0).to(r.target.dtype)
        r.draft[rows] = (r.target[rows].float() + 0.1 * torch.randn_like(r.draft[rows].float())).to(r.draft.dtype)
    # drafts at the drafter's mode, so that p(d) and q(d) stay far from fp64 underflow
    pos = torch.arange(r.rows, device=DEV) % (k + 1) < k
    r.draft_tokens[pos] = r.draft.float().argmax(dim=1).to(torch.int32)[pos]
    r.temperatures.fill_(temp)
    orc = run_oracle(r)
    compare(r, run_gpu(r, stats=False), orc, check_stats=False)
    compare(r, run_gpu(r, stats=True), orc, check_stats=True)


def test_token_range_layout_and_unsupported_statuses():
    r = _tiny_round(lanes=4, temp=0.0)
    off = r.row_offsets.cpu().numpy()
    r.draft_tokens[off[1] + 1] = 64          # == V
    r.draft_tokens[off[2]] = -3
    gpu, orc = run_gpu(r), run_oracle(r)
    assert gpu["lane_status"].tolist() == [0, 5, 5, 0]
    compare(r, gpu, orc)
    # draft_lens disagree with the offsets: layout error, nothing written
    r = _tiny_round(lanes=4, temp=0.0)
    r.draft_lens[3] = 2
    gpu = run_gpu(r)
    assert gpu["lane_status"].tolist() == [0, 0, 0, 6]
    assert gpu["committed"][3] == 0
    # more drafts than the kernel supports
    r = workloads.make_custom_round(4, DEV, lanes=2, vocab=100, kmax=16, fixed_k=True, sampled="none")
    gpu = run_gpu(r)
    assert gpu["lane_status"].tolist() == [2, 2]
    assert (gpu["out_tokens"] == -1).all()


def test_sampled_lane_without_draft_logits_is_an_argument_error():
    r = _tiny_round(lanes=3, temp=1.0)
    r.temperatures[0] = 0.0
    r.draft = None
    gpu = run_gpu(r)
    assert gpu["lane_status"].tolist() == [0, 1, 1]


def test_host_argument_errors():
    r = _tiny_round()
    c = torch.zeros(4, dtype=torch.int32, device=DEV)
    o = torch.zeros(r.rows, dtype=torch.int32, device=DEV)
    with pytest.raises(sv.SpecError) as e:
        sv.spec_verify_accept(r.target, None, r.draft_tokens, r.draft_lens, r.row_offsets,
                              r.temperatures, 1, c, o, rows=2)  # rows < lanes
    assert e.value.code == sv.SPEC_ERR_INVALID_ARG


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_vocabulary_of_a_million(dtype):
    """V = 1,000,003 (odd, past every benchmarked size): 62,504-element slices
    at 16 CTAs per lane, a ragged tail in every row, greedy and sampled lanes."""
    r = workloads.make_custom_round(61, DEV, lanes=3, vocab=1_000_003, kmax=5, dtype=dtype, sampled="mixed")
    orc = run_oracle(r)
    compare(r, run_gpu(r), orc)
    compare(r, run_gpu(r, stats=False), orc, check_stats=False)


@pytest.mark.parametrize("vocab", [20000, 200000], ids=["per-group-issue", "single-issuer"])
@pytest.mark.parametrize("sampled", ["none", "mixed"])
def test_a_wait_that_never_completes_reports_a_timeout(vocab, sampled):
    """With SPEC_VERIFY_TEST_WITHHOLD_COPY each CTA's producer skips its last
    bulk copy: the consumers' wait for it runs out after the kernel's 2 s
    limit, every lane reports SPEC_ERR_TIMEOUT with nothing committed, the
    launch returns, and the next launch on the same context matches the oracle."""
    import time

    r = workloads.make_custom_round(81, DEV, lanes=4, vocab=vocab, kmax=3, dtype="bf16", sampled=sampled,
                                    fixed_k=True)
    committed = torch.full((r.lanes,), -7, dtype=torch.int32, device=DEV)
    out = torch.full((r.rows,), -7, dtype=torch.int32, device=DEV)
    status = torch.full((r.lanes,), -7, dtype=torch.int32, device=DEV)
    torch.cuda.synchronize()
    t0 = time.time()
    sv.spec_verify_accept(r.target, r.draft, r.draft_tokens, r.draft_lens, r.row_offsets, r.temperatures,
                          r.seed, committed, out, status, test_flags=sv.SPEC_VERIFY_TEST_WITHHOLD_COPY)
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    assert (status.cpu() == sv.SPEC_ERR_TIMEOUT).all(), status
    assert (committed.cpu() == 0).all()
    assert 1.5 < elapsed < 60, elapsed
    compare(r, run_gpu(r), run_oracle(r))


def test_identical_draft_and_target_accepts_everything():
    """q == p: every ratio is 1 > u, so every sampled lane commits k + 1."""
    r = _tiny_round(vocab=5000, k=6, lanes=8, temp=0.8)
    r.draft = r.target.clone()
    gpu, orc = run_gpu(r), run_oracle(r)
    assert (gpu["committed"] == 7).all()
    compare(r, gpu, orc)


@pytest.mark.parametrize("cluster,vocab", [("1", 262144), ("2", 151936), ("4", 262144), ("3", 99991)])
def test_draws_deep_in_long_segments(monkeypatch, cluster, vocab):
    """Small clusters on large vocabularies give every warp a pass-2 segment of
    many 256-element rounds (up to 52).  The warp that holds the crossing finds
    its round from the round sums kept in the sum phase and re-reads only that
    round; over many seeds the crossings fall in every part of the segments.
    Drawn tokens must match the oracle's inverse-CDF draws."""
    monkeypatch.setenv("SPEC_VERIFY_CLUSTER", cluster)
    for seed in range(3):
        r = workloads.make_custom_round(700 + seed, DEV, lanes=6, vocab=vocab, kmax=3, dtype="bf16", sampled="all",
                                        fixed_k=True, sigma=0.5, spike=0.0, alpha=0.3)
        orc = run_oracle(r)
        compare(r, run_gpu(r, stats=False), orc, check_stats=False)
        compare(r, run_gpu(r, stats=True), orc, check_stats=True)


def test_results_do_not_depend_on_the_cluster_shape(monkeypatch):
    r = workloads.make_custom_round(31, DEV, lanes=6, vocab=70000, kmax=7, dtype="bf16", sampled="mixed")
    ref = run_gpu(r)
    orc = run_oracle(r)
    for c in ("1", "2", "4", "8", "16"):
        monkeypatch.setenv("SPEC_VERIFY_CLUSTER", c)
        for slot_kb in ("32", "4"):
            monkeypatch.setenv("SPEC_VERIFY_SLOT_KB", slot_kb)
            g = run_gpu(r)
            compare(r, g, orc)
            # greedy lanes are bit-identical across shapes
            greedy = (r.temperatures.cpu().numpy() <= 0)
            assert (g["committed"][greedy] == ref["committed"][greedy]).all()


@pytest.mark.parametrize("lanes,vocab,kmax", [(300, 3000, 7), (9, 40000, 7), (200, 20000, 3)])
def test_longest_first_lane_order_changes_nothing(monkeypatch, lanes, vocab, kmax):
    """With more lanes than resident clusters the kernel maps clusters to lanes
    in order of decreasing cost (300 lanes of V=3000 do so by themselves);
    forcing that order on or off must give bit-identical outputs, equal to the
    oracle's."""
    r = workloads.make_custom_round(41 + lanes, DEV, lanes=lanes, vocab=vocab, kmax=kmax, dtype="bf16",
                                    sampled="mixed")
    orc = run_oracle(r)
    runs = {}
    for order in ("0", "1"):
        monkeypatch.setenv("SPEC_VERIFY_ORDER", order)
        runs[order] = run_gpu(r)
        compare(r, runs[order], orc)
    # the order is also computed before the wait for the previous kernel
    runs["early"] = run_gpu(r, meta_before_wait=True)
    for key in ("committed", "out_tokens", "lane_status"):
        np.testing.assert_array_equal(runs["0"][key], runs["1"][key], err_msg=key)
        np.testing.assert_array_equal(runs["1"][key], runs["early"][key], err_msg=key)


@pytest.mark.parametrize("sampled,dtype", [("mixed", "bf16"), ("none", "bf16"), ("all", "f32")])
def test_every_kernel_build_matches_the_oracle(monkeypatch, sampled, dtype):
    """The kernel is built three times: 16 consumer warps in groups of 4 (rounds
    without drafter logits), 20 in groups of 4, and 20 in groups of 5 (rounds
    with them, chosen by shape).  Forcing each build on each kind of round must
    match the oracle; greedy lanes are bit-identical across builds (the argmax
    does not depend on how the warps split the slice)."""
    r = workloads.make_custom_round(58, DEV, lanes=11, vocab=50021, kmax=7, dtype=dtype, sampled=sampled)
    orc = run_oracle(r)
    runs = {}
    for build, warps in (("0", 16), ("1", 20), ("2", 20)):
        monkeypatch.setenv("SPEC_VERIFY_BUILD", build)
        shape = sv.spec_verify_launch_shape(r.lanes, r.rows, r.vocab, r.target.dtype)
        assert shape["threads"] == (warps + 2) * 32
        runs[build] = run_gpu(r)
        compare(r, runs[build], orc)
    greedy = r.temperatures.cpu().numpy() <= 0
    for build in ("1", "2"):
        np.testing.assert_array_equal(runs["0"]["committed"][greedy], runs[build]["committed"][greedy])


def test_rounds_choose_their_kernel_build_by_shape():
    """Whole-row slices in one slot with two slots per group take the groups-of-5
    build: the 8-lane sampled round, and the 8-lane greedy round (its slots are
    above the parallel-issue size).  Row slices streamed in several chunks take
    the groups-of-4 build with drafter logits (the 128-lane ragged round) and the
    16-warp build without (the 64-lane greedy round), as does the 1-lane round of
    4 KB rows when the small-round kernel is switched off; with it, that round
    runs one CTA per lane."""
    s8 = sv.spec_verify_launch_shape(8, 64, 151936, torch.bfloat16, with_draft=True)
    g8 = sv.spec_verify_launch_shape(8, 64, 151936, torch.bfloat16, with_draft=False)
    s128 = sv.spec_verify_launch_shape(128, 563, 262144, torch.bfloat16, with_draft=True)
    g64 = sv.spec_verify_launch_shape(64, 256, 151936, torch.bfloat16, with_draft=False)
    g1 = sv.spec_verify_launch_shape(1, 4, 1024, torch.float32, with_draft=False)
    assert s8["threads"] == g8["threads"] == s128["threads"] == 22 * 32
    assert g64["threads"] == 18 * 32
    # rows of at most 16 KB without drafter logits: the small-round kernel, one CTA of 16 warps per lane
    assert (g1["cluster_ctas"], g1["threads"], g1["smem_bytes"]) == (1, 16 * 32, 0)
    # groups of five: eight 25 KB slots (over 200 KB); groups of four would hold five
    for s in (s8, g8):
        assert s["slice"] * 2 <= 40 * 1024 and s["smem_bytes"] > 8 * s["slice"] * 2
    assert s128["slice"] * 2 > 40 * 1024 and g64["slice"] * 2 > 40 * 1024


@pytest.mark.parametrize("cluster,ring_kb,slot_kb", [("4", "75", "32"), ("12", "75", "32"), ("16", "88", "32"),
                                                      ("8", "40", "8"), ("2", "100", "32")])
@pytest.mark.parametrize("meta_early", [False, True], ids=["meta-after-wait", "meta-before-wait"])
def test_back_to_back_graph_launches_are_identical(monkeypatch, cluster, ring_kb, slot_kb, meta_early):
    """50 launches captured in one CUDA graph (the kernels overlap through
    programmatic dependent launch), each into its own outputs: every launch
    must give the same results, equal to the oracle's.  Ring shapes that would
    leave an odd number of slots are included on purpose; so is the launch
    that reads the lane metadata before waiting for the previous kernel."""
    monkeypatch.setenv("SPEC_VERIFY_CLUSTER", cluster)
    monkeypatch.setenv("SPEC_VERIFY_RING_KB", ring_kb)
    monkeypatch.setenv("SPEC_VERIFY_SLOT_KB", slot_kb)
    r = workloads.make_custom_round(77, DEV, lanes=12, vocab=151936, kmax=5, dtype="bf16",
                                    sampled="mixed", fixed_k=True)
    n = 50
    outs = [(torch.zeros(r.lanes, dtype=torch.int32, device=DEV),
             torch.zeros(r.rows, dtype=torch.int32, device=DEV),
             torch.zeros(r.lanes, dtype=torch.int32, device=DEV)) for _ in range(n)]
    stream = torch.cuda.Stream()

    def launch(o):
        sv.spec_verify_accept(r.target, r.draft, r.draft_tokens, r.draft_lens, r.row_offsets,
                              r.temperatures, r.seed, o[0], o[1], o[2], stream=torch.cuda.current_stream(),
                              meta_before_wait=meta_early)

    with torch.cuda.stream(stream):
        launch(outs[0])  # sets kernel attributes before capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            for o in outs:
                launch(o)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    orc = run_oracle(r)
    first = {"committed": outs[0][0].cpu().numpy(), "out_tokens": outs[0][1].cpu().numpy(),
             "lane_status": outs[0][2].cpu().numpy()}
    compare(r, first, orc, check_stats=False)
    for o in outs[1:]:
        assert torch.equal(o[0], outs[0][0]) and torch.equal(o[1], outs[0][1]) and torch.equal(o[2], outs[0][2])


def test_lane_shards_reproduce_the_unsplit_round():
    """Verifying lanes [lo, hi) on their own with lane_base = lo gives exactly
    the results those lanes get in the whole round (what a lane-sharded
    multi-GPU run relies on)."""
    from speculative_decoding_verify_bf16_gb300.sharding import lane_range, shard_rows

    r = workloads.make_custom_round(91, DEV, lanes=11, vocab=50000, kmax=6, dtype="bf16", sampled="mixed")
    full = run_gpu(r)
    for rank in range(3):
        lo, hi = lane_range(r.lanes, 3, rank)
        row_lo, row_hi, offs = shard_rows(r.row_offsets.tolist(), lo, hi)
        c = torch.zeros(hi - lo, dtype=torch.int32, device=DEV)
        o = torch.zeros(row_hi - row_lo, dtype=torch.int32, device=DEV)
        st = torch.zeros(hi - lo, dtype=torch.int32, device=DEV)
        sv.spec_verify_accept(r.target[row_lo:row_hi], r.draft[row_lo:row_hi],
                              r.draft_tokens[row_lo:row_hi].contiguous(), r.draft_lens[lo:hi].contiguous(),
                              torch.tensor(offs, dtype=torch.int32, device=DEV),
                              r.temperatures[lo:hi].contiguous(), r.seed, c, o, st, lane_base=lo)
        torch.cuda.synchronize()
        assert np.array_equal(c.cpu().numpy(), full["committed"][lo:hi])
        assert np.array_equal(o.cpu().numpy(), full["out_tokens"][row_lo:row_hi])


def _run_both_kernels(monkeypatch, r, stats):
    small = run_gpu(r, stats=stats)
    monkeypatch.setenv("SPEC_VERIFY_SMALL", "0")
    cluster = run_gpu(r, stats=stats)
    monkeypatch.delenv("SPEC_VERIFY_SMALL")
    for key in small:
        a, b = np.asarray(small[key]), np.asarray(cluster[key])
        if a.dtype.kind == "f":
            a, b = a.view(np.uint32 if a.itemsize == 4 else np.uint64), b.view(np.uint32 if b.itemsize == 4 else np.uint64)
        np.testing.assert_array_equal(a, b, err_msg=key)
    return small


@pytest.mark.parametrize("stats", [True, False], ids=["stats", "nostats"])
@pytest.mark.parametrize("dtype,vocab", [("bf16", 1), ("bf16", 7), ("f32", 8), ("f32", 9), ("bf16", 1023),
                                         ("f32", 1024), ("f32", 4096), ("bf16", 4097), ("bf16", 8192)])
def test_small_round_kernel_equals_the_cluster_kernel(monkeypatch, dtype, vocab, stats):
    """Greedy rounds of rows up to 16 KB run one CTA per lane (one warp per
    row, plain loads, batches reduced as trees): every output, row statistics
    included, has the cluster kernel's bits, and both match the oracle -- 1 to
    16 rows a lane, ties within a batch and across batches, and ragged tails
    included."""
    r = workloads.make_custom_round(70 + vocab, DEV, lanes=23, vocab=vocab, kmax=15, dtype=dtype, sampled="none")
    # ties: copies of each row's max a few elements later and a third of the
    # row away, in another lane's vectors or batch (the lowest index must win)
    if vocab > 16:
        t = r.target.float()
        a = t.argmax(dim=1)
        rows = torch.arange(r.rows, device=DEV)
        r.target[rows, (a + 5) % vocab] = r.target[rows, a]
        r.target[rows, (a + vocab // 3) % vocab] = r.target[rows, a]
    shape = sv.spec_verify_launch_shape(r.lanes, r.rows, r.vocab, r.target.dtype)
    assert (shape["cluster_ctas"], shape["threads"]) == (1, 16 * 32)
    compare(r, _run_both_kernels(monkeypatch, r, stats), run_oracle(r), check_stats=stats)


@pytest.mark.parametrize("layout", ["aligned", "padded", "misaligned"])
def test_small_round_kernel_statuses_and_layouts(monkeypatch, layout):
    """NaN, +inf and all -inf rows, draft tokens out of range, offsets that
    disagree with the draft lengths, more drafts than supported and a sampled
    lane without drafter logits: the small-round kernel reports what the
    cluster kernel reports, on aligned, padded (element-wise) and misaligned rows."""
    vocab = 1000
    ld = vocab + 5 if layout == "padded" else None
    r = workloads.make_custom_round(77, DEV, lanes=10, vocab=vocab, kmax=6, dtype="bf16", sampled="none",
                                    fixed_k=True, ld=ld)
    if layout == "misaligned":
        t = r.target
        buf = torch.empty(t.numel() + 1, dtype=t.dtype, device=t.device)
        buf[1:] = t.reshape(-1)
        r.target = buf[1:].view(t.shape)
        assert r.target.data_ptr() % 16 != 0
    off = r.row_offsets.cpu().numpy()
    r.target[off[1] + 2, 7] = float("nan")
    r.target[off[2] + 0, vocab - 3] = float("inf")
    r.target[off[3] + 1, :vocab] = float("-inf")
    r.target[off[4]:off[5], ::3] = float("-inf")   # allowed
    r.draft_tokens[off[5] + 1] = vocab
    r.draft_tokens[off[6]] = -1
    r.temperatures[7] = 0.9                         # sampled, but no drafter logits
    r.draft_lens[8] = 3                             # disagrees with the offsets
    gpu = _run_both_kernels(monkeypatch, r, True)
    assert gpu["lane_status"].tolist() == [0, 4, 4, 4, 0, 5, 5, 1, 6, 0]
    compare(r, gpu, run_oracle(r))
    r = workloads.make_custom_round(78, DEV, lanes=3, vocab=100, kmax=16, fixed_k=True, sampled="none")
    gpu = _run_both_kernels(monkeypatch, r, False)
    assert gpu["lane_status"].tolist() == [2, 2, 2] and (gpu["out_tokens"] == -1).all()
