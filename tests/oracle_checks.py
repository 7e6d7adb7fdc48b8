"""Pin checks of the CPU oracle against facts fixed outside it.

Each ``check_*`` function raises AssertionError when the oracle disagrees with
what the pages or the mathematics fix.  ``test_oracle_pins.py`` runs them on
the oracle as written; ``test_oracle_mutations.py`` runs them on copies of the
oracle with a plausible mistake planted, to show each mistake is caught.
"""

import numpy as np

import oracle
from conftest import read_golden

# ---------------------------------------------------------------------------
# Row budget: the worked example of ignis "The row budget"
# ---------------------------------------------------------------------------


def check_row_budget_worked_example():
    for draft_tokens, budget, lanes, expected in read_golden("row_budget_worked_example.txt"):
        got = oracle.row_budget(draft_tokens, budget, lanes)
        assert got == expected, (draft_tokens, budget, lanes, got, expected)


# ---------------------------------------------------------------------------
# Greedy: the guess/check table and equivalence with plain argmax decoding
# ---------------------------------------------------------------------------


def _one_lane(rows, drafts, temperature=0.0, draft_rows=None, **kw):
    rows = np.asarray(rows, np.float64)
    k = len(drafts)
    tokens = np.full(k + 1, -1, np.int64)
    tokens[:k] = drafts
    return oracle.verify_round(rows, draft_rows, tokens, [k], [0, k + 1],
                               np.array([temperature], np.float32), **kw)


def check_guess_check_table():
    """strata2signal "Guess, then check" table, on rows with distinct argmaxes."""
    rng = np.random.default_rng(11)
    for guesses, matches, expected in read_golden("guess_check_table.txt"):
        vocab = 50
        rows = rng.normal(size=(guesses + 1, vocab))
        best = [int(np.argmax(r)) for r in rows]
        drafts = []
        for j in range(guesses):
            drafts.append(best[j] if j < matches else (best[j] + 1) % vocab)
        res = _one_lane(rows, drafts)
        assert res.lane_status[0] == oracle.STATUS_OK
        assert res.committed[0] == expected, (guesses, matches, res.committed[0])
        kept = res.out_tokens[:expected].tolist()
        assert kept == best[:expected], (kept, best)
        assert (res.out_tokens[expected:] == -1).all()


class ToyLM:
    """A deterministic 'model': logits of a prefix are a hash of the prefix.

    Logits are quantised to halves so that ties happen and the tie-break rule
    is exercised.
    """

    def __init__(self, vocab, seed):
        self.vocab = vocab
        self.seed = seed

    def logits(self, prefix):
        h = hash((self.seed,) + tuple(int(t) for t in prefix)) & 0xFFFFFFFF
        r = np.random.default_rng(h).normal(size=self.vocab) * 1.5
        return np.round(r * 2.0) / 2.0

    def next_token(self, prefix):
        """Plain decoding: the first index of the largest logit."""
        x = self.logits(prefix)
        return int(np.flatnonzero(x == x.max())[0])


def toy_state(prev, token):
    """A toy recurrent state update: 8 bytes mixed with the consumed token."""
    h = hash((bytes(prev), int(token))) & 0xFFFFFFFFFFFFFFFF
    return np.frombuffer(h.to_bytes(8, "little"), dtype=np.uint8).copy()


def check_greedy_equals_plain_decode(n_tokens=60, k=4, vocab=12):
    """Greedy speculative decoding emits exactly the plain argmax stream.

    ignis "One round, step by step" (the model decides every token; greedy output
    is the same as without speculation) and mashbox "What it does for you" (a
    greedy request keeps the model's top token at every position).  The state
    rolled by the commit must equal the state of consuming the emitted stream
    token by token (ignis step 5: "a rejected draft leaves no trace").
    """
    lm = ToyLM(vocab, seed=5)
    context = [3]
    anchor = lm.next_token(context)
    plain = [anchor]
    while len(plain) < n_tokens + k + 2:
        plain.append(lm.next_token(context + plain))

    rng = np.random.default_rng(0)
    drafters = {
        "perfect": lambda ctx, a, pos: plain[pos + 1:pos + 1 + k],
        "wrong": lambda ctx, a, pos: [(t + 1) % vocab for t in plain[pos + 1:pos + 1 + k]],
        "random": lambda ctx, a, pos: list(rng.integers(0, vocab, size=k)),
        "half": lambda ctx, a, pos: plain[pos + 1:pos + 3] + [(plain[pos + 3] + 5) % vocab] + [0],
    }
    for name, drafter in drafters.items():
        consumed = list(context)
        anchor = plain[0]
        emitted = [anchor]
        state = np.zeros(8, np.uint8)
        for t in context:
            state = toy_state(state, t)
        live = state.copy()
        while len(emitted) < n_tokens:
            drafts = [int(x) for x in drafter(consumed, anchor, len(emitted) - 1)]
            cols = [anchor] + drafts
            rows = [lm.logits(consumed + cols[:j + 1]) for j in range(k + 1)]
            res = _one_lane(rows, drafts)
            c = int(res.committed[0])
            assert 1 <= c <= k + 1
            committed_tokens = res.out_tokens[:c].tolist()
            # staged column j = state after consuming columns 0..j
            staged = []
            s = live.copy()
            for t in cols:
                s = toy_state(s, t)
                staged.append(s)
            staged = np.stack(staged)[None]
            live = oracle.commit_state(staged, live[None], [c])[0]
            consumed += cols[:c]
            anchor = committed_tokens[-1]
            emitted += committed_tokens
            plain_state = np.zeros(8, np.uint8)
            for t in consumed:
                plain_state = toy_state(plain_state, t)
            assert np.array_equal(live, plain_state), name
        assert emitted[:n_tokens] == plain[:n_tokens], name


# ---------------------------------------------------------------------------
# Sampled: exact enumeration of the acceptance rule on a tiny vocabulary
# ---------------------------------------------------------------------------

# Target rows p_j and drafter rows q_j, in sixteenths.  They are chosen so that
# every acceptance threshold min(1, p/q) and every cumulative boundary of the
# residual and bonus distributions is a multiple of 1/8; the uniforms are then
# enumerated at the midpoints of an 8-point grid, which integrates the rule
# exactly.  p_0 has a zero entry (logit -inf).
ENUM_P = [np.array([0, 6, 6, 4]) / 16, np.array([1, 3, 5, 7]) / 16, np.array([8, 4, 2, 2]) / 16]
ENUM_Q = [np.array([8, 4, 2, 2]) / 16, np.array([2, 2, 4, 8]) / 16]
ENUM_T = 0.7
GRID = (np.arange(8) + 0.5) / 8


def _enumerate_dyadic():
    """Exact probabilities of the emitted tokens, by enumeration.

    Returns (first, second, third):
      first[y]          P(t_1 = y)
      second[a, y]      P(t_2 = y and d_1 = a accepted)
      third[a, b, y]    P(t_3 = y and d_1 = a, d_2 = b accepted)
    """
    vocab, k = 4, 2
    with np.errstate(divide="ignore"):
        t_rows = [ENUM_T * np.log(p) for p in ENUM_P]
        d_rows = [ENUM_T * np.log(q) for q in ENUM_Q] + [np.zeros(vocab)]
    lanes = []
    for d1 in range(vocab):
        for d2 in range(vocab):
            w_d = ENUM_Q[0][d1] * ENUM_Q[1][d2]
            for ua0 in GRID:
                for ua1 in GRID:
                    for us in GRID:
                        lanes.append((d1, d2, ua0, ua1, us, w_d / GRID.size ** 3))
    n = len(lanes)
    target = np.concatenate([np.stack(t_rows)] * n)
    draft = np.concatenate([np.stack(d_rows)] * n)
    tokens = np.full(n * (k + 1), -1)
    tokens[0::3] = [l[0] for l in lanes]
    tokens[1::3] = [l[1] for l in lanes]
    u_acc = np.array([[l[2], l[3], 0.5] for l in lanes])
    u_smp = np.array([[l[4]] * 3 for l in lanes])
    res = oracle.verify_round(target, draft, tokens, np.full(n, k), np.arange(n + 1) * 3,
                              np.full(n, ENUM_T, np.float32), u_acc=u_acc, u_smp=u_smp)
    first = np.zeros(vocab)
    second = np.zeros((vocab, vocab))
    third = np.zeros((vocab, vocab, vocab))
    for i, (d1, d2, _, _, _, w) in enumerate(lanes):
        assert res.lane_status[i] == oracle.STATUS_OK
        c = int(res.committed[i])
        t = res.out_tokens[3 * i:3 * i + c]
        assert 1 <= c <= 3 and (res.out_tokens[3 * i + c:3 * i + 3] == -1).all()
        first[t[0]] += w
        if c >= 2:
            assert t[0] == d1
            second[d1, t[1]] += w
        if c >= 3:
            assert t[1] == d2
            third[d1, d2, t[2]] += w
    return first, second, third


def check_sampled_exact_enumeration():
    """Emitted tokens have the target's distribution, exactly.

    ignis "One round, step by step" ("sampling keeps its distribution") and
    strata2signal "Guess, then check" (with the right acceptance rule the
    output is sampled without changing the distribution; Leviathan et al.
    2022, Theorem 3.8): t_1 ~ p_0, and given that d_1 .. d_j were accepted the
    next emitted token ~ p_j.  The acceptance probability of position j is
    sum_x min(p_j(x), q_j(x)) (the same paper's acceptance rate).
    """
    first, second, third = _enumerate_dyadic()
    np.testing.assert_allclose(first, ENUM_P[0], rtol=0, atol=1e-12)
    beta0 = np.minimum(ENUM_P[0], ENUM_Q[0]).sum()
    beta1 = np.minimum(ENUM_P[1], ENUM_Q[1]).sum()
    assert abs(second.sum() - beta0) < 1e-12
    assert abs(third.sum() - beta0 * beta1) < 1e-12
    for a in range(4):
        tot = second[a].sum()
        if tot > 0:
            np.testing.assert_allclose(second[a] / tot, ENUM_P[1], rtol=0, atol=1e-12)
        for b in range(4):
            tot = third[a, b].sum()
            if tot > 0:
                np.testing.assert_allclose(third[a, b] / tot, ENUM_P[2], rtol=0, atol=1e-12)


def check_sampled_monte_carlo(n_lanes=12000, seed=2024):
    """Same property on non-dyadic rows, through the Philox uniforms.

    Chi-square tests of t_1 against p_0 and of t_2 (given d_1 accepted)
    against p_1, with drafts drawn from q by the test.
    """
    from scipy import stats

    rng = np.random.default_rng(seed)
    vocab, k, temp = 5, 2, 0.8
    t_rows = rng.normal(size=(k + 1, vocab)) * 1.3
    d_rows = t_rows + rng.normal(size=(k + 1, vocab))
    p = [np.exp(r / temp) / np.exp(r / temp).sum() for r in t_rows]
    q = [np.exp(r / temp) / np.exp(r / temp).sum() for r in d_rows]
    d1 = rng.choice(vocab, size=n_lanes, p=q[0])
    d2 = rng.choice(vocab, size=n_lanes, p=q[1])
    tokens = np.full(n_lanes * 3, -1)
    tokens[0::3], tokens[1::3] = d1, d2
    res = oracle.verify_round(np.tile(t_rows, (n_lanes, 1)), np.tile(d_rows, (n_lanes, 1)),
                              tokens, np.full(n_lanes, k), np.arange(n_lanes + 1) * 3,
                              np.full(n_lanes, temp, np.float32), seed=seed)
    out = res.out_tokens.reshape(n_lanes, 3)
    t1 = np.bincount(out[:, 0], minlength=vocab)
    assert stats.chisquare(t1, p[0] * n_lanes).pvalue > 1e-4
    acc = res.committed >= 2
    t2 = np.bincount(out[acc, 1], minlength=vocab)
    assert stats.chisquare(t2, p[1] * acc.sum()).pvalue > 1e-4
    beta0 = np.minimum(p[0], q[0]).sum()
    se = np.sqrt(beta0 * (1 - beta0) / n_lanes)
    assert abs(acc.mean() - beta0) < 5 * se


def check_sampled_special_cases():
    """Cases the rule reduces to by hand.

    * q == p: every ratio is 1 and u < 1, so every draft is accepted.
    * q one-hot on the draft d: accepted with probability p(d); on rejection
      the residual is p with d removed, renormalised.
    """
    rng = np.random.default_rng(7)
    vocab, k, temp = 6, 3, 1.1
    rows = rng.normal(size=(k + 1, vocab))
    drafts = [int(x) for x in rng.integers(0, vocab, size=k)]
    for lane in range(20):
        res = _one_lane(rows, drafts, temperature=temp, draft_rows=rows, seed=lane)
        assert res.committed[0] == k + 1
        assert res.out_tokens[:k].tolist() == drafts
    # one-hot q at d: drafter logits -inf except at d
    d = 2
    q_row = np.full(vocab, -np.inf)
    q_row[d] = 0.0
    p = np.exp(rows[0] / temp) / np.exp(rows[0] / temp).sum()
    acc_hits, resid = 0, np.zeros(vocab)
    grid = (np.arange(256) + 0.5) / 256
    for ua in grid:
        for us in grid[::8]:
            res = _one_lane(rows[:2], [d], temperature=temp,
                            draft_rows=np.stack([q_row, q_row]),
                            u_acc=[[ua, 0.5]], u_smp=[[us, us]])
            if res.committed[0] == 2:
                acc_hits += 1
            else:
                resid[res.out_tokens[0]] += 1
    assert abs(acc_hits / (grid.size * grid[::8].size) - p[d]) < 1.5 / grid.size
    expect = p.copy()
    expect[d] = 0
    expect /= expect.sum()
    assert resid[d] == 0
    np.testing.assert_allclose(resid / resid.sum(), expect, atol=2.5 / grid[::8].size)


def check_inverse_cdf_never_draws_zero_weight():
    """A token of weight 0 is never drawn, whatever u in [0, 1)."""
    w = np.array([0.0, 0.25, 0.0, 0.5, 0.25, 0.0])
    for u in [0.0, 1e-300, 0.25 - 1e-12, 0.25, 0.5, 0.75, 1.0 - 2 ** -24]:
        tok, _ = oracle.inverse_cdf(w, u)
        assert w[tok] > 0, (u, tok)
    assert oracle.inverse_cdf(w, 0.0)[0] == 1
    assert oracle.inverse_cdf(w, 0.25)[0] == 3
    assert oracle.inverse_cdf(w, 0.75)[0] == 4
    # the same through a round: a bonus draw (k = 0) from p with zero entries
    with np.errstate(divide="ignore"):
        row = np.log(w)[None, :]
    for u in [0.0, 0.25, 0.75, 1.0 - 2 ** -24]:
        res = _one_lane(row, [], temperature=1.0, draft_rows=np.zeros_like(row),
                        u_acc=[[0.5]], u_smp=[[u]])
        assert w[res.out_tokens[0]] > 0, (u, res.out_tokens[0])


# ---------------------------------------------------------------------------
# Closed form: expected tokens a round for i.i.d. acceptance
# ---------------------------------------------------------------------------


def check_expected_tokens_closed_form(n_lanes=20000, gamma=4, alpha=0.73, seed=3):
    """E[tokens a round] = (1 - alpha^(gamma+1)) / (1 - alpha).

    strata2signal "Acceptance: three numbers with one name": the textbook
    formula for gamma guesses that each survive independently with
    probability alpha.  Each draft equals its row's argmax with probability
    alpha and is otherwise a different token.
    """
    rng = np.random.default_rng(seed)
    vocab = 16
    rows = rng.normal(size=(n_lanes * (gamma + 1), vocab))
    best = np.argmax(rows, axis=1)
    hit = rng.random(n_lanes * (gamma + 1)) < alpha
    other = (best + rng.integers(1, vocab, size=best.size)) % vocab
    tokens = np.where(hit, best, other)
    tokens[gamma::gamma + 1] = -1
    res = oracle.verify_round(rows, None, tokens, np.full(n_lanes, gamma),
                              np.arange(n_lanes + 1) * (gamma + 1),
                              np.zeros(n_lanes, np.float32))
    expect = (1 - alpha ** (gamma + 1)) / (1 - alpha)
    c = res.committed.astype(np.float64)
    assert abs(c.mean() - expect) < 5 * c.std() / np.sqrt(n_lanes), (c.mean(), expect)


# ---------------------------------------------------------------------------
# Library routines: Philox (numpy), softmax / logsumexp (scipy), bf16 (torch)
# ---------------------------------------------------------------------------


def check_philox_against_numpy():
    """Blocks equal numpy's Philox4x64-10 (numpy steps the counter before a block)."""
    cases = [((0, 0, 0, 0), (0, 0)), ((5, 3, 0, 0), (123456789, 0)),
             ((2 ** 64 - 1, 7, 1, 0), (2 ** 64 - 1, 2 ** 63)),
             ((1, 0, 0, 0), (0xDEADBEEF, 0))]
    for ctr, key in cases:
        prev = (sum(c << (64 * i) for i, c in enumerate(ctr)) - 1) % (1 << 256)
        ctr_prev = np.array([(prev >> (64 * i)) & (2 ** 64 - 1) for i in range(4)], np.uint64)
        bg = np.random.Philox(counter=ctr_prev, key=np.array(key, np.uint64))
        assert [int(x) for x in bg.random_raw(4)] == list(oracle.philox4x64_10(ctr, key))


def check_softmax_against_scipy():
    from scipy import special

    rng = np.random.default_rng(1)
    for temp in [0.3, 0.7, 1.0, 1.9]:
        row = rng.normal(size=1000) * 4
        row[[3, 17, 999]] = -np.inf
        p, lse = oracle.softmax_at_temperature(row, temp)
        np.testing.assert_allclose(p, special.softmax(row / temp), rtol=1e-12, atol=0)
        assert abs(lse - special.logsumexp(row / temp)) < 1e-12 * abs(lse) + 1e-12
        assert p[3] == 0 and p[999] == 0


def check_decode_bf16_against_torch():
    import torch

    rng = np.random.default_rng(4)
    bits = rng.integers(0, 2 ** 16, size=20000).astype(np.uint16)
    bits = bits[~(((bits & 0x7F80) == 0x7F80) & ((bits & 0x007F) != 0))]  # drop NaNs
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    assert np.array_equal(oracle.decode_bf16(bits), ref)


# ---------------------------------------------------------------------------
# Commit
# ---------------------------------------------------------------------------


def check_commit_copies_column_committed_minus_one():
    rng = np.random.default_rng(9)
    lanes, cols, nbytes = 5, 4, 24
    staged = rng.integers(0, 256, size=(lanes, cols, nbytes), dtype=np.uint8)
    live = rng.integers(0, 256, size=(lanes, nbytes), dtype=np.uint8)
    committed = np.array([1, 4, 2, 0, 3])
    status = np.array([0, 0, 0, 0, oracle.STATUS_NONFINITE])
    out = oracle.commit_state(staged, live, committed, status)
    assert np.array_equal(out[0], staged[0, 0])
    assert np.array_equal(out[1], staged[1, 3])
    assert np.array_equal(out[2], staged[2, 1])
    assert np.array_equal(out[3], live[3])          # count 0: invalid, untouched
    assert np.array_equal(out[4], live[4])          # failed lane: untouched
    st = oracle.commit_status(committed, cols, status)
    assert st.tolist() == [0, 0, 0, oracle.STATUS_LAYOUT, oracle.STATUS_NONFINITE]


# ---------------------------------------------------------------------------
# Acceptance metrics: strata2signal "Acceptance: three numbers with one name"
# ---------------------------------------------------------------------------
import os

from oracle import backoff as ob
from oracle import metrics as om

_GOLDEN_DIR = os.path.join(os.path.dirname(__file__), "golden")


def _golden_rates():
    out = {}
    with open(os.path.join(_GOLDEN_DIR, "acceptance_rates_worked_example.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                name, value, decimals = line.split()
                out[name] = (float(value), int(decimals))
    return out


def _printed(value, printed):
    """value, rounded as the page rounds it, equals the printed figure."""
    want, decimals = printed
    assert abs(value - want) <= 0.5 * 10.0 ** (-decimals) + 1e-12, (value, want)


def check_acceptance_metrics_worked_example():
    """The page's 43 rounds give every figure its table prints."""
    counts = om.AcceptCounts()
    for k, n, times in read_golden("acceptance_rounds_worked_example.txt"):
        for _ in range(times):
            om.count_round(counts, k, n)
    assert (counts.rounds, counts.proposed, counts.accepted) == (43, 171, 84)
    assert counts.slot_kept[:4] == [37, 24, 16, 7]
    g = _golden_rates()
    r = om.accept_rates(counts)
    _printed(r.accepted_per_proposed, g["accepted_per_proposed"])
    _printed(r.tokens_per_round, g["tokens_per_round"])
    for j in range(4):
        _printed(r.by_slot[j], g[f"by_slot_{j + 1}"])
        _printed(r.given_previous[j], g[f"given_previous_{j + 1}"])
    assert r.depth == 4
    _printed(r.implied_alpha, g["implied_alpha"])
    # "one plus their sum is 2.95 again"
    _printed(1.0 + sum(r.by_slot), g["tokens_per_round"])
    llama = om.AcceptCounts(rounds=1, proposed=297, accepted=171)
    _printed(om.accept_rates(llama).accepted_per_proposed, g["llama_accepted_per_proposed"])


def check_acceptance_metrics_identities(seed=5):
    """On random rounds: one plus the by-slot shares is the tokens a round;
    the given-previous shares multiply up to the by-slot shares; the implied
    alpha reproduces the tokens a round; rounds that proposed nothing still
    count as rounds."""
    rng = np.random.default_rng(seed)
    for trial in range(20):
        counts = om.AcceptCounts()
        for _ in range(int(rng.integers(1, 200))):
            k = int(rng.integers(0, 16))
            om.count_round(counts, k, int(rng.integers(0, k + 1)))
        r = om.accept_rates(counts)
        assert abs(1.0 + sum(r.by_slot) - r.tokens_per_round) < 1e-12
        prod = 1.0
        for j in range(om.MAX_SLOTS):
            if counts.slot_kept[j] == 0:
                break
            prod *= r.given_previous[j]
            assert abs(prod - r.by_slot[j]) < 1e-12
        assert sum(counts.slot_kept) == counts.accepted
        assert sum(counts.slot_reached) == counts.proposed
        if r.depth > 0 and 1.0 < r.tokens_per_round < r.depth + 1.0:
            assert abs(om.tokens_a_round_of_alpha(r.implied_alpha, r.depth) - r.tokens_per_round) < 1e-9


def check_implied_alpha_recovers_independent_guesses(seed=11, rounds=200000):
    """Guesses that each survive with probability alpha, independently, give an
    implied alpha close to alpha (the textbook model the page's alpha assumes)."""
    rng = np.random.default_rng(seed)
    for alpha, depth in ((0.73, 4), (0.5, 7), (0.9, 3)):
        survive = rng.random((rounds, depth)) < alpha
        kept = np.argmin(np.concatenate([survive, np.zeros((rounds, 1), bool)], axis=1), axis=1)
        counts = om.AcceptCounts()
        counts.rounds, counts.proposed, counts.accepted = rounds, rounds * depth, int(kept.sum())
        r = om.accept_rates(counts)
        assert abs(r.implied_alpha - alpha) < 0.01, (alpha, r.implied_alpha)


def check_metrics_from_verify_outputs():
    """Counting a verify round's outputs: a lane proposes draft_lens[b] and keeps
    committed[b] - 1; failed lanes are left out."""
    counts = om.count_verify_outputs(om.AcceptCounts(), committed=[1, 4, 3, 0, 2], draft_lens=[3, 3, 7, 2, 1],
                                     lane_status=[0, 0, 0, oracle.STATUS_LAYOUT, 0])
    assert (counts.rounds, counts.proposed, counts.accepted) == (4, 14, 6)
    assert counts.slot_kept[:4] == [3, 2, 1, 0]
    assert counts.slot_reached[:8] == [4, 3, 3, 1, 1, 1, 1, 0]


# ---------------------------------------------------------------------------
# Miss back-off: mashbox "Speculative decoding", "What it does for you"
# ---------------------------------------------------------------------------
def _guess_pattern(n_passes, kept_when_guessing, lanes=1, others_guess=True):
    """Run lane 0 through n_passes; it keeps kept_when_guessing(i) guesses in
    pass i when it may guess (3 proposed).  Returns the string of passes:
    'g' guessed, 'w' waited."""
    states = [ob.BackoffState() for _ in range(lanes)]
    out = []
    for i in range(n_passes):
        prop = [3 if ob.may_guess(s) else 0 for s in states]
        kept = [0] * lanes
        if prop[0]:
            kept[0] = kept_when_guessing(i)
        if not others_guess:
            for b in range(1, lanes):
                prop[b] = 0
        out.append("g" if prop[0] else "w")
        ob.step(states, prop, kept)
    return "".join(out)


def check_backoff_waits_16_then_doubles_to_256():
    """Misses only: 4 passes guess, then 16 wait; each further 4 misses double
    the wait, up to 256."""
    want = ""
    for w in (16, 32, 64, 128, 256, 256):
        want += "gggg" + "w" * w
    want += "gggg"
    pat = _guess_pattern(len(want), lambda i: 0)
    assert pat == want, pat


def check_backoff_kept_guess_resets():
    """A pass that keeps a guess ends the miss run and sets the wait back to 16."""
    # 3 misses, a keep, then misses: the first wait starts after 4 more misses
    pat = _guess_pattern(3 + 1 + 4 + 16 + 1, lambda i: 1 if i == 3 else 0)
    assert pat == "ggg" + "g" + "gggg" + "w" * 16 + "g", pat
    # the wait doubles to 32, then a keep after it brings the next wait back to 16
    seq = "gggg" + "w" * 16 + "gggg" + "w" * 32
    keep_at = len(seq)  # first pass after the 32-pass wait keeps a guess
    pat = _guess_pattern(len(seq) + 1 + 4 + 16 + 1, lambda i: 1 if i == keep_at else 0)
    assert pat == seq + "g" + "gggg" + "w" * 16 + "g", pat


def check_backoff_passes_without_speculation():
    """A pass in which no lane of the batch has a guess counts toward no miss
    run (and does not break one), only toward a wait already running; a lane
    that may guess but has no guess in a pass that speculates counts a miss."""
    s = [ob.BackoffState(), ob.BackoffState()]
    for _ in range(3):  # lane 0 misses 3 times, lane 1 guesses and keeps
        ob.step(s, [2, 2], [0, 1])
    ob.step(s, [0, 0], [0, 0])  # nobody guesses: not counted
    assert s[0].misses == 3 and s[0].wait == 0
    ob.step(s, [0, 2], [0, 1])  # lane 0 has no guess in a pass that speculates: a miss
    assert s[0].wait == 16 and s[0].misses == 0 and s[0].backoff == 32
    for _ in range(5):  # waiting counts down in passes that do not speculate too
        ob.step(s, [0, 0], [0, 0])
    assert s[0].wait == 11
    assert ob.next_draft_lens(s, 5) == [0, 5]


# ---------------------------------------------------------------------------
# n-gram drafter: mashbox "Speculative decoding", "Options" (--speculation ngram)
# ---------------------------------------------------------------------------
from oracle import ngram as ong


def check_ngram_hand_examples():
    """Worked by hand from the definition: find the last tokens earlier in the
    history, propose what followed them there."""
    # "1 2" recurs at positions 1-2; what followed was 3 9 1
    assert ong.ngram_draft([5, 1, 2, 3, 9, 1, 2], 3)[:2] == ([3, 9, 1], 2)
    # the last token never occurred before: nothing to propose
    assert ong.ngram_draft([1, 2, 3], 3)[0] == []
    # the most recent of two occurrences; only two tokens follow it
    assert ong.ngram_draft([7, 1, 4, 1, 5, 1], 3)[:3] == ([5, 1], 1, 4)
    # a longer match wins over a more recent shorter one
    hist = [1, 2, 3, 8, 2, 3, 9, 1, 2, 3]
    assert ong.ngram_draft(hist, 3)[:2] == ([8, 2, 3], 3)
    # ... unless the longest allowed match is shorter
    assert ong.ngram_draft(hist, 3, match_max=2)[:3] == ([9, 1, 2], 2, 6)
    # the match may overlap the suffix itself
    assert ong.ngram_draft([4, 4, 4, 4], 3)[:3] == ([4], 3, 3)
    # k limits the proposal; a minimum match length can rule a lane out
    assert ong.ngram_draft([5, 1, 2, 3, 9, 1, 2], 1)[0] == [3]
    assert ong.ngram_draft([7, 1, 4, 1, 5, 1], 3, match_min=2)[0] == []
    assert ong.ngram_draft([9], 3)[0] == [] and ong.ngram_draft([1, 1], 0)[0] == []


def check_ngram_brute_force(seed=8):
    """Tiny random histories: the best (length, position) over every earlier
    occurrence of every allowed suffix, enumerated as a set."""
    rng = np.random.default_rng(seed)
    for trial in range(3000):
        L = int(rng.integers(1, 13))
        h = [int(x) for x in rng.integers(0, 3, L)]
        k = int(rng.integers(1, 6))
        mmin, mmax = sorted(int(x) for x in rng.integers(1, 6, 2))
        cands = [(m, i) for m in range(mmin, min(mmax, L - 1) + 1) for i in range(m, L)
                 if h[i - m:i] == h[L - m:]]
        want = h[max(cands)[1]:max(cands)[1] + k] if cands else []
        got = ong.ngram_draft(h, k, mmin, mmax)[0]
        assert got == want, (h, k, mmin, mmax, got, want)


# ---------------------------------------------------------------------------
# Presence / frequency penalties (FreeToken #828, PR #836), read as the usual rule
# ---------------------------------------------------------------------------
from oracle import penalties as opn


def check_bf16_rounding_against_torch(seed=12):
    """Round-to-nearest-even to bf16 equals torch's float32 -> bfloat16."""
    import torch
    rng = np.random.default_rng(seed)
    x = np.concatenate([rng.normal(0, 3, 20000), rng.normal(0, 1e-3, 2000), rng.normal(0, 1e4, 2000)]).astype(np.float32)
    # values exactly halfway between two bf16 numbers
    half = (rng.integers(0, 1 << 15, 2000).astype(np.uint32) << 16 | 0x8000).view(np.float32)
    x = np.concatenate([x, half[np.isfinite(half)]])
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(opn.round_to_bf16(x), want)


def check_penalty_rule_by_hand():
    """Counts and arithmetic of the rule, worked by hand."""
    # count 2, presence 0.5, frequency 0.25: 3 - (0.5 + 2 * 0.25) = 2
    assert opn.penalise_value(3.0, 2, 0.5, 0.25, "bf16") == 2.0
    # count 3, frequency only: 1 - 1.5 = -0.5
    assert opn.penalise_value(1.0, 3, 0.0, 0.5, "f32") == -0.5
    # no penalty leaves a bf16 logit as it is
    assert opn.penalise_value(1.3984375, 4, 0.0, 0.0, "bf16") == 1.3984375
    # fp32 arithmetic, then bf16 rounding: 1 - 1e-3 is 0.999 in fp32, 1.0 in bf16
    assert opn.penalise_value(1.0, 1, 1e-3, 0.0, "f32") == float(np.float32(1.0) - np.float32(1e-3))
    assert opn.penalise_value(1.0, 1, 1e-3, 0.0, "bf16") == 1.0
    # row j counts the history and d_1..d_j
    hist = {5: 1}
    assert opn.row_counts(hist, [5, 7], 0) == {5: 1}
    assert opn.row_counts(hist, [5, 7], 1) == {5: 2}
    assert opn.row_counts(hist, [5, 7], 2) == {5: 2, 7: 1}


def check_penalties_on_a_round():
    """A lane of 3 rows: only listed tokens and earlier drafts move; a penalised
    argmax hands the argmax to the runner-up, and the drafter's rows are left alone."""
    V = 8
    target = np.zeros((3, V))
    target[:, 2] = 5.0   # the argmax of every row
    target[:, 6] = 4.5   # the runner-up
    drafts = np.array([2, 6, -1], np.int32)
    out = opn.apply_penalties(target, "f32", drafts, np.array([2]), np.array([0, 3]),
                              pen_tokens=np.array([2]), pen_counts=np.array([1]), pen_offsets=np.array([0, 1]),
                              presence=np.array([1.0], np.float32), frequency=np.array([0.0], np.float32))
    assert out[0, 2] == 4.0 and out[1, 2] == 4.0 and out[2, 2] == 4.0   # count 1, 2, 2: presence only
    assert out[0, 6] == 4.5 and out[1, 6] == 4.5 and out[2, 6] == 3.5   # d_2 = 6 counts from row 2 on
    assert np.array_equal(out[:, [0, 1, 3, 4, 5, 7]], target[:, [0, 1, 3, 4, 5, 7]])
    res = oracle.verify_round(out, None, drafts, [2], [0, 3], np.array([0.0], np.float32))
    assert res.out_tokens[0] == 6  # the penalised argmax gave way; d_1 = 2 is rejected
    assert res.committed[0] == 1
    # with frequency the counts scale
    out = opn.apply_penalties(target, "f32", drafts, np.array([2]), np.array([0, 3]),
                              pen_tokens=np.array([2]), pen_counts=np.array([3]), pen_offsets=np.array([0, 1]),
                              presence=np.array([0.0], np.float32), frequency=np.array([0.5], np.float32))
    assert out[0, 2] == 3.5 and out[1, 2] == 3.0 and out[2, 2] == 3.0


ALL_CHECKS = [
    check_row_budget_worked_example,
    check_guess_check_table,
    check_greedy_equals_plain_decode,
    check_sampled_exact_enumeration,
    check_sampled_monte_carlo,
    check_sampled_special_cases,
    check_inverse_cdf_never_draws_zero_weight,
    check_expected_tokens_closed_form,
    check_philox_against_numpy,
    check_softmax_against_scipy,
    check_decode_bf16_against_torch,
    check_commit_copies_column_committed_minus_one,
    check_acceptance_metrics_worked_example,
    check_acceptance_metrics_identities,
    check_implied_alpha_recovers_independent_guesses,
    check_metrics_from_verify_outputs,
    check_backoff_waits_16_then_doubles_to_256,
    check_backoff_kept_guess_resets,
    check_backoff_passes_without_speculation,
    check_ngram_hand_examples,
    check_ngram_brute_force,
    check_bf16_rounding_against_torch,
    check_penalty_rule_by_hand,
    check_penalties_on_a_round,
]
