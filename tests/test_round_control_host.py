"""Host side of the acceptance-metric ABI against the oracle (no GPU needed)."""

import math

import numpy as np

import oracle_checks as oc
from conftest import read_golden
from oracle import metrics as om

import speculative_decoding_verify_bf16_gb300 as sv


def _row(c):
    return [c.rounds, c.proposed, c.accepted] + list(c.slot_reached) + list(c.slot_kept)


def _same(a, b):
    return (math.isnan(a) and math.isnan(b)) or a == b


def test_rates_of_the_worked_example_through_the_abi():
    counts = om.AcceptCounts()
    for k, n, times in read_golden("acceptance_rounds_worked_example.txt"):
        for _ in range(times):
            om.count_round(counts, k, n)
    r = sv.spec_accept_rates_from_counts(_row(counts))
    g = oc._golden_rates()
    oc._printed(r["accepted_per_proposed"], g["accepted_per_proposed"])
    oc._printed(r["tokens_per_round"], g["tokens_per_round"])
    for j in range(4):
        oc._printed(r["by_slot"][j], g[f"by_slot_{j + 1}"])
        oc._printed(r["given_previous"][j], g[f"given_previous_{j + 1}"])
    oc._printed(r["implied_alpha"], g["implied_alpha"])
    assert r["depth"] == 4


def test_rates_equal_the_oracle_on_random_counts():
    rng = np.random.default_rng(17)
    for trial in range(50):
        counts = om.AcceptCounts()
        for _ in range(int(rng.integers(0, 300))):
            k = int(rng.integers(0, 16))
            om.count_round(counts, k, int(rng.integers(0, k + 1)))
        r = sv.spec_accept_rates_from_counts(_row(counts))
        o = om.accept_rates(counts)
        assert _same(r["accepted_per_proposed"], o.accepted_per_proposed)
        assert _same(r["tokens_per_round"], o.tokens_per_round)
        assert r["depth"] == o.depth
        assert _same(r["implied_alpha"], o.implied_alpha)
        for j in range(om.MAX_SLOTS):
            assert _same(r["by_slot"][j], o.by_slot[j]) and _same(r["given_previous"][j], o.given_previous[j])


def test_rates_of_no_rounds_are_nan_and_null_is_an_error():
    r = sv.spec_accept_rates_from_counts([0] * sv.ACCEPT_COUNT_WORDS)
    assert math.isnan(r["tokens_per_round"]) and math.isnan(r["accepted_per_proposed"])
    assert math.isnan(r["implied_alpha"]) and r["depth"] == 0
    assert sv.load_library().spec_accept_rates_from_counts(None, None) == sv.SPEC_ERR_INVALID_ARG
