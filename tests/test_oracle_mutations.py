"""Plant plausible mistakes in the oracle (on the CPU) and show a pin catches each.

Every mutation below is a mistake that could slip into a restatement of the
method: a transposed operand, a wrong row index, a tie-break flipped, an
off-by-one in the commit, a dropped temperature, a non-strict comparison.  The
pins of ``oracle_checks`` must fail on every one of them.
"""

import numpy as np
import pytest

import oracle
import oracle.verify as ov
import oracle_checks as oc


def _argmax_last(row):
    return int(len(row) - 1 - np.argmax(row[::-1]))


def _residual_transposed(p, q):
    return np.maximum(0.0, q - p)


def _accept_transposed(u, p_d, q_d):
    return u < min(1.0, q_d / p_d if p_d > 0 else np.inf)


def _accept_without_clamp(u, p_d, q_d):
    return u < 0.5 * min(1.0, ov.acceptance_ratio(p_d, q_d)) + 0.25


def _greedy_next_row(t_rows, drafts):
    k = len(drafts)
    a = [ov.argmax_lowest(r) for r in t_rows]
    n = 0
    while n < k and int(drafts[n]) == a[min(n + 1, k)]:
        n += 1
    return a[:n + 1]


def _softmax_no_temperature(row, temperature):
    z = row
    zmax = np.max(z)
    e = np.exp(z - zmax)
    return e / e.sum(), float(zmax + np.log(e.sum()))


def _inverse_cdf_non_strict(weights, u):
    cdf = np.cumsum(weights)
    target = u * cdf[-1]
    token = int(np.nonzero(cdf >= target)[0][0])
    return token, 1.0


def _row_budget_ceil(draft_tokens, rows, lanes):
    rows = rows or 8
    return max(0, min(draft_tokens, -(-rows // lanes) - 1))


def _commit_wrong_column(staged, live, committed, lane_status=None):
    out = np.array(live, copy=True)
    for b in range(staged.shape[0]):
        c = int(committed[b])
        if 1 <= c <= staged.shape[1]:
            out[b] = staged[b, min(c, staged.shape[1] - 1)]
    return out


import oracle.backoff as ob
import oracle.metrics as om


def _rates_by_slot_over_proposed(counts):
    r = _orig_accept_rates(counts)
    r.by_slot = [counts.slot_kept[j] / counts.slot_reached[j] if counts.slot_reached[j] else float("nan")
                 for j in range(om.MAX_SLOTS)]
    return r


def _rates_given_over_rounds(counts):
    r = _orig_accept_rates(counts)
    r.given_previous = [counts.slot_kept[j] / counts.rounds for j in range(om.MAX_SLOTS)]
    return r


def _rates_tokens_without_own(counts):
    r = _orig_accept_rates(counts)
    r.tokens_per_round = counts.accepted / counts.rounds
    return r


def _alpha_depth_off_by_one(tokens_a_round, depth, iters=200):
    return _orig_implied_alpha(tokens_a_round, depth + 1, iters)


_orig_accept_rates = om.accept_rates
_orig_implied_alpha = om.implied_alpha


MUTATIONS = [
    ("argmax ties to the highest index", ov, "argmax_lowest", _argmax_last,
     oc.check_greedy_equals_plain_decode),
    ("residual max(0, q - p)", ov, "residual_weights", _residual_transposed,
     oc.check_sampled_exact_enumeration),
    ("acceptance ratio q/p", ov, "accept_draft", _accept_transposed,
     oc.check_sampled_exact_enumeration),
    ("acceptance threshold distorted", ov, "accept_draft", _accept_without_clamp,
     oc.check_sampled_monte_carlo),
    ("greedy compares d_{j+1} with row j+1", ov, "_greedy_lane", _greedy_next_row,
     oc.check_guess_check_table),
    ("temperature dropped", ov, "softmax_at_temperature", _softmax_no_temperature,
     oc.check_sampled_exact_enumeration),
    ("inverse CDF with >=", ov, "inverse_cdf", _inverse_cdf_non_strict,
     oc.check_inverse_cdf_never_draws_zero_weight),
    ("row budget rounds up", oracle, "row_budget", _row_budget_ceil,
     oc.check_row_budget_worked_example),
    ("commit copies column c", oracle, "commit_state", _commit_wrong_column,
     oc.check_commit_copies_column_committed_minus_one),
    ("by-slot share over rounds that proposed the slot", om, "accept_rates", _rates_by_slot_over_proposed,
     oc.check_acceptance_metrics_worked_example),
    ("given-previous share over all rounds", om, "accept_rates", _rates_given_over_rounds,
     oc.check_acceptance_metrics_worked_example),
    ("tokens a round without the model's own token", om, "accept_rates", _rates_tokens_without_own,
     oc.check_acceptance_metrics_worked_example),
    ("implied alpha at depth + 1", om, "implied_alpha", _alpha_depth_off_by_one,
     oc.check_acceptance_metrics_worked_example),
    ("back-off after 3 misses", ob, "MISSES_TO_WAIT", 3, oc.check_backoff_waits_16_then_doubles_to_256),
    ("back-off capped at 128", ob, "LONGEST_WAIT", 128, oc.check_backoff_waits_16_then_doubles_to_256),
    ("first wait 8 passes", ob, "FIRST_WAIT", 8, oc.check_backoff_kept_guess_resets),
]


@pytest.mark.parametrize("what,module,name,bad,check", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(monkeypatch, what, module, name, bad, check):
    monkeypatch.setattr(module, name, bad)
    with pytest.raises(AssertionError):
        check()


def test_commit_mistake_breaks_no_trace(monkeypatch):
    monkeypatch.setattr(oracle, "commit_state", _commit_wrong_column)
    with pytest.raises(AssertionError):
        oc.check_greedy_equals_plain_decode()


def _step_counts_every_pass(states, proposed, kept):
    for b, st in enumerate(states):
        if st.wait > 0:
            st.wait -= 1
            continue
        if kept[b] > 0:
            st.misses, st.backoff = 0, ob.FIRST_WAIT
            continue
        st.misses += 1
        if st.misses == ob.MISSES_TO_WAIT:
            st.wait, st.backoff, st.misses = st.backoff, min(2 * st.backoff, ob.LONGEST_WAIT), 0
    return [ob.may_guess(st) for st in states]


def _step_keep_during_run_not_reset(states, proposed, kept):
    speculates = any(p > 0 for p in proposed)
    for b, st in enumerate(states):
        if st.wait > 0:
            st.wait -= 1
            continue
        if not speculates:
            continue
        if kept[b] > 0:
            st.misses = 0  # forgets to set the wait back to 16
            continue
        st.misses += 1
        if st.misses == ob.MISSES_TO_WAIT:
            st.wait, st.backoff, st.misses = st.backoff, min(2 * st.backoff, ob.LONGEST_WAIT), 0
    return [ob.may_guess(st) for st in states]


@pytest.mark.parametrize("bad,check", [(_step_counts_every_pass, oc.check_backoff_passes_without_speculation),
                                       (_step_keep_during_run_not_reset, oc.check_backoff_kept_guess_resets)])
def test_backoff_step_mistakes_are_caught(monkeypatch, bad, check):
    monkeypatch.setattr(ob, "step", bad)
    with pytest.raises(AssertionError):
        check()


import oracle.ngram as ong


def _ngram_oldest(history, k, match_min=1, match_max=4):
    h = list(history)
    L = len(h)
    if k <= 0 or L < 2:
        return [], 0, -1
    for m in range(min(match_max, L - 1), match_min - 1, -1):
        for i in range(m, L):  # oldest first
            if h[i - m:i] == h[L - m:]:
                return h[i:min(i + k, L)], m, i
    return [], 0, -1


def _ngram_shortest(history, k, match_min=1, match_max=4):
    h = list(history)
    L = len(h)
    if k <= 0 or L < 2:
        return [], 0, -1
    for m in range(match_min, min(match_max, L - 1) + 1):
        for i in range(L - 1, m - 1, -1):
            if h[i - m:i] == h[L - m:]:
                return h[i:min(i + k, L)], m, i
    return [], 0, -1


def _ngram_includes_match(history, k, match_min=1, match_max=4):
    d, m, i = _orig_ngram(history, k, match_min, match_max)
    return (list(history)[i - 1:i - 1 + k], m, i) if i > 0 else (d, m, i)


_orig_ngram = ong.ngram_draft


@pytest.mark.parametrize("bad", [_ngram_oldest, _ngram_shortest, _ngram_includes_match])
def test_ngram_mistakes_are_caught(monkeypatch, bad):
    monkeypatch.setattr(ong, "ngram_draft", bad)
    with pytest.raises(AssertionError):
        oc.check_ngram_hand_examples()
    with pytest.raises(AssertionError):
        oc.check_ngram_brute_force()


import oracle.penalties as opn


def _round_toward_zero(x32):
    bits = np.asarray(x32, np.float32).view(np.uint32) & np.uint32(0xFFFF0000)
    return bits.view(np.float32)


def _row_counts_one_more(history_counts, drafts, j):
    return _orig_row_counts(history_counts, drafts, j + 1)


def _penalise_frequency_only(x, c, presence, frequency, dtype):
    return _orig_penalise(x, c, 0.0, frequency, dtype)


_orig_row_counts = opn.row_counts
_orig_penalise = opn.penalise_value


@pytest.mark.parametrize("name,bad,check", [
    ("round_to_bf16", _round_toward_zero, oc.check_bf16_rounding_against_torch),
    ("row_counts", _row_counts_one_more, oc.check_penalty_rule_by_hand),
    ("row_counts", _row_counts_one_more, oc.check_penalties_on_a_round),
    ("penalise_value", _penalise_frequency_only, oc.check_penalty_rule_by_hand),
])
def test_penalty_mistakes_are_caught(monkeypatch, name, bad, check):
    monkeypatch.setattr(opn, name, bad)
    with pytest.raises(AssertionError):
        check()


def test_philox_round_count_matters(monkeypatch):
    import oracle.philox as ph
    monkeypatch.setattr(ph, "ROUNDS", 9)
    with pytest.raises(AssertionError):
        oc.check_philox_against_numpy()
