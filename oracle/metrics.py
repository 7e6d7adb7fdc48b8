"""Acceptance metrics of speculative decoding, counted over verify rounds.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Follows strata->signal, "Draft heads and speculative decoding, in plain words",
section "Acceptance: three numbers with one name" (its table and the paragraph
after it).  One round of one lane proposes k guesses and keeps the first n of
them (n = committed - 1).  Over many rounds:

* guesses accepted / guesses proposed: sum n / sum k;
* tokens a round: one (the model's own token) plus the accepted guesses, per
  round: 1 + sum n / rounds;
* by slot: the share of rounds in which guess j survived, #(n >= j) / rounds;
  one plus their sum is the tokens a round again;
* each slot given the one before: #(n >= j) / #(n >= j - 1), with
  #(n >= 0) = rounds;
* the implied per-guess rate alpha: the single rate for which the textbook
  expectation (1 - alpha^(g + 1)) / (1 - alpha) of independent guesses at
  depth g equals the tokens a round.

Plain Python over a list of rounds; float64.
"""

from dataclasses import dataclass, field
from typing import List

MAX_SLOTS = 15


@dataclass
class AcceptCounts:
    rounds: int = 0
    proposed: int = 0
    accepted: int = 0
    slot_reached: List[int] = field(default_factory=lambda: [0] * MAX_SLOTS)  # rounds with k >= j
    slot_kept: List[int] = field(default_factory=lambda: [0] * MAX_SLOTS)     # rounds with n >= j


def count_round(counts, k, n):
    """Add one round that proposed k guesses and kept n of them."""
    if not (0 <= n <= k <= MAX_SLOTS):
        raise ValueError("need 0 <= kept <= proposed <= 15")
    counts.rounds += 1
    counts.proposed += k
    counts.accepted += n
    for j in range(1, MAX_SLOTS + 1):
        if k >= j:
            counts.slot_reached[j - 1] += 1
        if n >= j:
            counts.slot_kept[j - 1] += 1
    return counts


def count_verify_outputs(counts, committed, draft_lens, lane_status=None):
    """Add one verify round's outputs: lane b proposed draft_lens[b] and
    committed committed[b] = kept + 1 tokens.  Lanes whose status is not 0, or
    whose counts are not a verify result (draft length outside 0..15, committed
    outside 1..draft length + 1), are left out."""
    for b in range(len(committed)):
        if lane_status is not None and lane_status[b] != 0:
            continue
        k, c = int(draft_lens[b]), int(committed[b])
        if not (0 <= k <= MAX_SLOTS and 1 <= c <= k + 1):
            continue
        count_round(counts, k, c - 1)
    return counts


def tokens_a_round_of_alpha(alpha, depth):
    """(1 - alpha^(depth + 1)) / (1 - alpha): expected tokens a round for
    independent guesses that each survive with probability alpha."""
    if alpha >= 1.0:
        return depth + 1.0
    return (1.0 - alpha ** (depth + 1)) / (1.0 - alpha)


def implied_alpha(tokens_a_round, depth, iters=200):
    """The alpha in [0, 1] with tokens_a_round_of_alpha(alpha, depth) equal to
    tokens_a_round (bisection; the function increases with alpha)."""
    lo, hi = 0.0, 1.0
    if tokens_a_round <= 1.0:
        return 0.0
    if tokens_a_round >= depth + 1.0:
        return 1.0
    for _ in range(iters):
        mid = 0.5 * (lo + hi)
        if tokens_a_round_of_alpha(mid, depth) < tokens_a_round:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


@dataclass
class AcceptRates:
    accepted_per_proposed: float
    tokens_per_round: float
    by_slot: List[float]
    given_previous: List[float]
    depth: int
    implied_alpha: float


def accept_rates(counts):
    """The page's quantities from the counts.  The depth of the implied alpha
    is the mean number of guesses proposed a round, rounded to an integer."""
    r = counts.rounds
    nan = float("nan")
    app = counts.accepted / counts.proposed if counts.proposed else nan
    tpr = 1.0 + counts.accepted / r if r else nan
    by_slot = [counts.slot_kept[j] / r if r else nan for j in range(MAX_SLOTS)]
    given = []
    prev = r
    for j in range(MAX_SLOTS):
        given.append(counts.slot_kept[j] / prev if prev else nan)
        prev = counts.slot_kept[j]
    depth = int(counts.proposed / r + 0.5) if r else 0
    alpha = implied_alpha(tpr, depth) if r and depth > 0 else nan
    return AcceptRates(app, tpr, by_slot, given, depth, alpha)
