"""Acceptance counts, the miss back-off and the n-gram drafter on the GPU
against the oracle (integers: exact)."""

import numpy as np
import pytest
import torch

import oracle
import oracle_checks as oc
import workloads
from conftest import read_golden
from gpu_harness import run_gpu
from oracle import backoff as ob
from oracle import metrics as om

import speculative_decoding_verify_bf16_gb300 as sv

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


def _row(c):
    return [c.rounds, c.proposed, c.accepted] + list(c.slot_reached) + list(c.slot_kept)


def _i32(a):
    return torch.tensor(np.asarray(a, np.int32), device=DEV)


def test_counts_of_verify_rounds_match_the_oracle():
    """Several verify rounds of mixed lanes, counted on the GPU per batch and per
    lane, equal the oracle's counts of the same outputs."""
    lanes = 24
    batch = sv.new_accept_counts(1, DEV)
    per_lane = sv.new_accept_counts(lanes, DEV)
    orc_batch = om.AcceptCounts()
    orc_lane = [om.AcceptCounts() for _ in range(lanes)]
    for seed in range(6):
        r = workloads.make_custom_round(300 + seed, DEV, lanes=lanes, vocab=20000, kmax=7, dtype="bf16",
                                        sampled="mixed")
        g = run_gpu(r, stats=False)
        committed = _i32(g["committed"])
        status = _i32(g["lane_status"])
        sv.spec_accept_counts_update(committed, r.draft_lens, status, batch)
        sv.spec_accept_counts_update(committed, r.draft_lens, status, per_lane, per_lane=True)
        k = r.draft_lens.cpu().numpy()
        om.count_verify_outputs(orc_batch, g["committed"], k, g["lane_status"])
        for b in range(lanes):
            om.count_verify_outputs(orc_lane[b], g["committed"][b:b + 1], k[b:b + 1], g["lane_status"][b:b + 1])
    torch.cuda.synchronize()
    assert batch[0].tolist() == _row(orc_batch)
    for b in range(lanes):
        assert per_lane[b].tolist() == _row(orc_lane[b]), b
    # the per-lane counts add up to the batch's
    assert per_lane.sum(0).tolist() == batch[0].tolist()


def test_counts_skip_failed_and_impossible_lanes():
    rng = np.random.default_rng(3)
    lanes = 5000
    k = rng.integers(-2, 18, lanes)
    committed = rng.integers(-1, 20, lanes)
    status = np.where(rng.random(lanes) < 0.1, oracle.STATUS_NONFINITE, 0)
    for st in (status, None):
        counts = sv.new_accept_counts(1, DEV)
        sv.spec_accept_counts_update(_i32(committed), _i32(k), None if st is None else _i32(st), counts)
        torch.cuda.synchronize()
        want = om.count_verify_outputs(om.AcceptCounts(), committed, k, st)
        assert counts[0].tolist() == _row(want)
        assert want.rounds > 1000


def test_worked_example_through_the_device_counts():
    ks, ns = [], []
    for k, n, times in read_golden("acceptance_rounds_worked_example.txt"):
        ks += [k] * times
        ns += [n] * times
    counts = sv.new_accept_counts(1, DEV)
    sv.spec_accept_counts_update(_i32(np.array(ns) + 1), _i32(ks), None, counts)
    torch.cuda.synchronize()
    c = sv.accept_counts_view(counts[0])
    assert (c["rounds"], c["proposed"], c["accepted"]) == (43, 171, 84)
    r = sv.spec_accept_rates_from_counts(counts[0])
    g = oc._golden_rates()
    oc._printed(r["accepted_per_proposed"], g["accepted_per_proposed"])
    oc._printed(r["tokens_per_round"], g["tokens_per_round"])
    for j in range(4):
        oc._printed(r["by_slot"][j], g[f"by_slot_{j + 1}"])
        oc._printed(r["given_previous"][j], g[f"given_previous_{j + 1}"])
    oc._printed(r["implied_alpha"], g["implied_alpha"])


@pytest.mark.parametrize("lanes,draft_tokens,p_keep", [(64, 3, 0.15), (3000, 5, 0.4), (7, 8, 0.02)])
def test_backoff_matches_the_oracle_pass_by_pass(lanes, draft_tokens, p_keep):
    """Random rounds: lanes that may guess sometimes have no guess, some rounds
    nobody guesses, some lanes fail; states and next draft lengths equal the
    oracle's after every pass."""
    rng = np.random.default_rng(lanes)
    states = sv.new_backoff_states(lanes, DEV)
    orc = [ob.BackoffState() for _ in range(lanes)]
    nxt = torch.full((lanes,), draft_tokens, dtype=torch.int32, device=DEV)
    may = np.full(lanes, draft_tokens)
    waited = 0
    for it in range(2000):
        prop = may.copy()
        prop[rng.random(lanes) < 0.1] = 0           # the drafter found nothing
        if rng.random() < 0.05:
            prop[:] = 0                             # a round in which nobody guesses
        kept = np.where(rng.random(lanes) < p_keep, rng.integers(1, draft_tokens + 1, lanes), 0)
        kept = np.minimum(kept, prop)
        committed = kept + 1
        status = np.where(rng.random(lanes) < 0.02, oracle.STATUS_NONFINITE, 0)
        kept_orc = np.where(status == 0, kept, 0)
        sv.spec_backoff_step(states, _i32(prop), _i32(committed), _i32(status), draft_tokens, nxt)
        ob.step(orc, prop.tolist(), kept_orc.tolist())
        may = np.array(ob.next_draft_lens(orc, draft_tokens))
        if it % 50 == 49 or it == 1999:
            got = states.cpu().numpy()
            want = np.array([[s.misses, s.backoff, s.wait] for s in orc])
            np.testing.assert_array_equal(got[:, :3], want, err_msg=f"pass {it}")
        np.testing.assert_array_equal(nxt.cpu().numpy(), may, err_msg=f"pass {it}")
        waited += int((may == 0).sum())
    assert waited > 0  # waits happened


def test_round_control_argument_errors():
    lib = sv.load_library()
    assert lib.spec_accept_counts_update(None, None, None, -1, None, 0, None) == sv.SPEC_ERR_INVALID_ARG
    assert lib.spec_accept_counts_update(None, None, None, 4, None, 0, None) == sv.SPEC_ERR_INVALID_ARG
    assert lib.spec_accept_counts_update(None, None, None, 0, None, 2, None) == sv.SPEC_ERR_INVALID_ARG
    assert lib.spec_accept_counts_update(None, None, None, 0, None, 0, None) == sv.SPEC_OK
    assert lib.spec_backoff_init(None, 3, None) == sv.SPEC_ERR_INVALID_ARG
    assert lib.spec_backoff_step(None, None, None, None, 3, 2, None, None) == sv.SPEC_ERR_INVALID_ARG
    st = sv.new_backoff_states(2, DEV)
    z = torch.zeros(2, dtype=torch.int32, device=DEV)
    with pytest.raises(sv.SpecError):
        sv.spec_backoff_step(st, z, z, None, 16, z)


# ---------------------------------------------------------------------------
# copy-from-the-conversation drafter
# ---------------------------------------------------------------------------
def _ngram_case(rng, lanes, max_len, vocab):
    lens = rng.integers(0, max_len + 1, lanes)
    hists = [[int(x) for x in rng.integers(0, vocab, n)] for n in lens]
    # plant recurrences so that long matches exist
    for h in hists:
        if len(h) > 12 and rng.random() < 0.7:
            m = int(rng.integers(1, 8))
            src = int(rng.integers(0, len(h) - m - 1))
            h[-m:] = h[src:src + m]
    offs = np.concatenate([[0], np.cumsum([len(h) for h in hists])]).astype(np.int64)
    flat = np.array([t for h in hists for t in h] or [0], np.int32)
    return hists, torch.tensor(flat, device=DEV), torch.tensor(offs, device=DEV)


@pytest.mark.parametrize("lanes,max_len,vocab,k,mmin,mmax", [(200, 60, 4, 3, 1, 4), (37, 3000, 50, 8, 2, 6),
                                                            (5, 100000, 1000, 15, 1, 16), (64, 10, 2, 1, 3, 3)])
def test_ngram_drafts_match_the_oracle(lanes, max_len, vocab, k, mmin, mmax):
    from oracle import ngram as ong
    rng = np.random.default_rng(lanes * 7 + k)
    hists, flat, offs = _ngram_case(rng, lanes, max_len, vocab)
    drafts = torch.full((lanes, k + 2), -5, dtype=torch.int32, device=DEV)
    lens = torch.full((lanes,), -5, dtype=torch.int32, device=DEV)
    sv.spec_ngram_draft(flat, offs, k, drafts, lens, match_min=mmin, match_max=mmax)
    torch.cuda.synchronize()
    d, l = drafts.cpu().numpy(), lens.cpu().numpy()
    found = 0
    for b, h in enumerate(hists):
        want = ong.ngram_draft(h, k, mmin, mmax)[0]
        assert l[b] == len(want), (b, l[b], want)
        assert d[b, :len(want)].tolist() == want, b
        assert (d[b, len(want):] == -5).all()  # slots past the drafts are untouched
        found += len(want) > 0
    assert found > 0


def test_ngram_argument_errors():
    lib = sv.load_library()
    z64 = torch.zeros(3, dtype=torch.int64, device=DEV)
    z32 = torch.zeros(8, dtype=torch.int32, device=DEV)
    for k, stride, mmin, mmax in [(16, 16, 1, 4), (3, 2, 1, 4), (3, 3, 0, 4), (3, 3, 3, 2), (3, 3, 1, 17)]:
        assert lib.spec_ngram_draft(z32.data_ptr(), z64.data_ptr(), 2, k, mmin, mmax, z32.data_ptr(), stride,
                                    z32.data_ptr(), None) == sv.SPEC_ERR_INVALID_ARG
    assert lib.spec_ngram_draft(None, None, 2, 3, 1, 4, None, 3, None, None) == sv.SPEC_ERR_INVALID_ARG
    assert lib.spec_ngram_draft(None, None, 0, 3, 1, 4, None, 3, None, None) == sv.SPEC_OK


# ---------------------------------------------------------------------------
# per-row presence / frequency penalties
# ---------------------------------------------------------------------------
def _penalty_lists(rng, r, max_hist):
    V = r.vocab
    toks, counts, offs = [], [], [0]
    dt = r.draft_tokens.cpu().numpy()
    off = r.row_offsets.cpu().numpy()
    for b in range(r.lanes):
        n = int(rng.integers(0, max_hist + 1))
        pool = set(int(x) for x in rng.integers(0, V, n))
        # some drafts of the lane are in the history too, and the row argmaxes
        for j in range(int(off[b + 1] - off[b]) - 1):
            if rng.random() < 0.5:
                pool.add(int(dt[off[b] + j]))
        pool.add(int(r.target[off[b]].float().argmax()))
        t = sorted(pool)
        toks += t
        counts += [int(c) for c in rng.integers(1, 4, len(t))]
        offs.append(len(toks))
    to = lambda a, d: torch.tensor(np.asarray(a), dtype=d, device=DEV)
    return to(toks or [0], torch.int32), to(counts or [1], torch.int32), to(offs, torch.int64)


@pytest.mark.parametrize("dtype,sampled,seed", [("bf16", "mixed", 1), ("f32", "mixed", 2), ("bf16", "none", 3),
                                                ("bf16", "all", 4)])
def test_penalties_match_the_oracle_and_feed_the_verify(dtype, sampled, seed):
    from gpu_harness import compare, logits_to_numpy, run_oracle
    from oracle import penalties as opn
    rng = np.random.default_rng(seed)
    r = workloads.make_custom_round(600 + seed, DEV, lanes=19, vocab=30011, kmax=7, dtype=dtype, sampled=sampled)
    # repeated drafts within a lane
    dt = r.draft_tokens.clone()
    off = r.row_offsets.cpu().numpy()
    for b in range(0, r.lanes, 3):
        if off[b + 1] - off[b] > 2:
            dt[off[b] + 1] = dt[off[b]]
    r.draft_tokens = dt
    toks, counts, offs = _penalty_lists(rng, r, 200)
    pres = torch.tensor(rng.uniform(0, 2, r.lanes), dtype=torch.float32, device=DEV)
    freq = torch.tensor(rng.uniform(0, 1, r.lanes), dtype=torch.float32, device=DEV)
    pres[0], freq[0] = 0.0, 0.0
    before = logits_to_numpy(r.target, r.vocab)
    sv.spec_apply_penalties(r.target, r.row_offsets, r.draft_tokens, r.draft_lens, toks, counts, offs, pres, freq)
    torch.cuda.synchronize()
    got = logits_to_numpy(r.target, r.vocab)
    want = opn.apply_penalties(before, dtype, r.draft_tokens.cpu().numpy(), r.draft_lens.cpu().numpy(), off,
                               toks.cpu().numpy(), counts.cpu().numpy(), offs.cpu().numpy(),
                               pres.cpu().numpy(), freq.cpu().numpy())
    np.testing.assert_array_equal(got, want)
    assert (got != before).sum() > r.lanes
    # the verify on the penalised logits against the oracle's verify on its own penalised copy
    compare(r, run_gpu(r), run_oracle(r))


def test_penalty_lists_that_break_the_contract_are_reported_and_left_alone():
    """The history list of a lane must hold distinct ids in ascending order with
    counts >= 1.  A repeated id (two threads would update one logit), an id out
    of order (the search for drafts would miss it) or a count of 0 is reported
    per lane as SPEC_ERR_INVALID_ARG and that lane's logits stay as they were;
    lanes with valid lists are penalised exactly as the oracle says, and a lane
    whose offsets disagree with its draft length gets SPEC_ERR_LAYOUT."""
    from gpu_harness import logits_to_numpy
    from oracle import penalties as opn
    rng = np.random.default_rng(17)
    r = workloads.make_custom_round(617, DEV, lanes=6, vocab=5003, kmax=5, dtype="bf16", sampled="mixed",
                                    fixed_k=True)
    lists = []
    for b in range(r.lanes):
        ids = np.sort(rng.choice(r.vocab, size=40, replace=False)).astype(np.int32)
        cnt = rng.integers(1, 4, size=40).astype(np.int32)
        lists.append([ids, cnt])
    lists[1][0][7] = lists[1][0][6]                      # a repeated id
    lists[2][0][[3, 4]] = lists[2][0][[4, 3]]            # two ids out of order
    lists[3][1][10] = 0                                  # a count of 0
    toks = torch.tensor(np.concatenate([l[0] for l in lists]), dtype=torch.int32, device=DEV)
    counts = torch.tensor(np.concatenate([l[1] for l in lists]), dtype=torch.int32, device=DEV)
    offs = torch.tensor(np.arange(r.lanes + 1) * 40, dtype=torch.int64, device=DEV)
    lens = r.draft_lens.clone()
    lens[5] = 3                                          # offsets disagree with the draft length
    pres = torch.full((r.lanes,), 0.75, dtype=torch.float32, device=DEV)
    freq = torch.full((r.lanes,), 0.5, dtype=torch.float32, device=DEV)
    status = torch.full((r.lanes,), -7, dtype=torch.int32, device=DEV)
    before = logits_to_numpy(r.target, r.vocab)
    sv.spec_apply_penalties(r.target, r.row_offsets, r.draft_tokens, lens, toks, counts, offs, pres, freq,
                            lane_status=status)
    torch.cuda.synchronize()
    got = logits_to_numpy(r.target, r.vocab)
    assert status.cpu().tolist() == [0, sv.SPEC_ERR_INVALID_ARG, sv.SPEC_ERR_INVALID_ARG, sv.SPEC_ERR_INVALID_ARG,
                                     0, sv.SPEC_ERR_LAYOUT]
    off = r.row_offsets.cpu().numpy()
    want = opn.apply_penalties(before, "bf16", r.draft_tokens.cpu().numpy(), r.draft_lens.cpu().numpy(), off,
                               toks.cpu().numpy(), counts.cpu().numpy(), offs.cpu().numpy(), pres.cpu().numpy(),
                               freq.cpu().numpy())
    for b in range(r.lanes):
        rows = slice(off[b], off[b + 1])
        if b in (0, 4):
            np.testing.assert_array_equal(got[rows], want[rows])
            assert (got[rows] != before[rows]).any()
        else:
            np.testing.assert_array_equal(got[rows], before[rows])


def test_penalties_argument_errors():
    lib = sv.load_library()
    assert lib.spec_apply_penalties(None, 1, 10, 10, -1, *([None] * 10)) == sv.SPEC_ERR_INVALID_ARG
    assert lib.spec_apply_penalties(None, 1, 10, 10, 2, *([None] * 10)) == sv.SPEC_ERR_INVALID_ARG
    assert lib.spec_apply_penalties(None, 1, 9, 10, 0, *([None] * 10)) == sv.SPEC_ERR_INVALID_ARG
    assert lib.spec_apply_penalties(None, 7, 10, 10, 0, *([None] * 10)) == sv.SPEC_ERR_INVALID_ARG
    assert lib.spec_apply_penalties(None, 1, 10, 10, 0, *([None] * 10)) == sv.SPEC_OK


def test_mean_committed_count_follows_the_closed_form():
    """Greedy rounds whose drafts equal the row argmax independently with
    probability alpha (a uniform token otherwise, which matches with
    probability 1/V): the committed count is a truncated geometric variable,
    E[c] = (1 - a^(k+1)) / (1 - a) with a = alpha + (1 - alpha) / V
    (strata2signal "Tokens a round" gives the closed form for independent
    guesses).  The device's mean over 2048 lanes must lie within four
    standard errors of it, and the alpha implied by the device counts within
    four standard errors of a."""
    lanes, k, vocab, alpha = 2048, 7, 1000, 0.8
    r = workloads.make_custom_round(555, DEV, lanes=lanes, vocab=vocab, kmax=k, dtype="bf16", sampled="none",
                                    fixed_k=True, alpha=alpha)
    g = run_gpu(r, stats=False)
    assert (g["lane_status"] == 0).all()
    a = alpha + (1 - alpha) / vocab
    n = np.arange(k + 1)
    pmf = np.append(a ** n[:-1] * (1 - a), a ** k)          # P(n accepted), n = 0..k
    mean = float((pmf * (n + 1)).sum())
    assert abs(mean - (1 - a ** (k + 1)) / (1 - a)) < 1e-12
    sd = float(np.sqrt((pmf * (n + 1 - mean) ** 2).sum()))
    got = float(g["committed"].mean())
    assert abs(got - mean) < 4 * sd / np.sqrt(lanes), (got, mean, sd)
    counts = sv.new_accept_counts(1, DEV)
    sv.spec_accept_counts_update(torch.tensor(g["committed"], device=DEV), r.draft_lens,
                                 torch.tensor(g["lane_status"], device=DEV), counts)
    rates = sv.spec_accept_rates_from_counts(counts[0])
    # each guess j > 0 is reached by ~lanes * a^j rounds; the pooled estimate of a
    # from slot survival has a standard error below sqrt(a (1 - a) / lanes)
    assert abs(rates["given_previous"][0] - a) < 4 * np.sqrt(a * (1 - a) / lanes), rates
