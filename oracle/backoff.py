"""Miss back-off of a drafter whose guesses keep missing.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Follows mashbox docs, "Speculative decoding", section "What it does for you"
(the paragraph on a request whose guesses keep missing).  Read with one pass
per device call, which is what one verify round is:

* a lane that is not waiting may guess; a pass of a call that speculates
  (at least one lane of the batch has a guess) counts for every lane that may
  guess, whether or not it has a guess in that pass;
* after 4 counted passes in a row in which the model kept none of the lane's
  guesses, the lane waits: it makes no guesses for the next `backoff` passes
  (16 at first); each further 4 such passes in a row double the wait, up to 256;
* a counted pass that keeps a guess resets the miss run and sets the wait back
  to 16 (a waiting lane keeps no guesses, so the reset never happens during a
  wait);
* a pass of a call that does not speculate (no lane of the batch has a guess)
  counts toward no lane's misses, only toward the wait of a lane already
  waiting; every pass of a waiting lane counts toward its wait.

State per lane: (misses, backoff, wait).  Plain Python.
"""

from dataclasses import dataclass

MISSES_TO_WAIT = 4
FIRST_WAIT = 16
LONGEST_WAIT = 256


@dataclass
class BackoffState:
    misses: int = 0          # counted passes in a row with no guess kept
    backoff: int = FIRST_WAIT  # length of the next wait
    wait: int = 0            # passes left in the current wait (0: may guess)


def may_guess(state):
    return state.wait == 0


def step(states, proposed, kept):
    """One pass of a batch.  proposed[b] is the number of guesses lane b made
    in the pass (0 while waiting), kept[b] how many of them the model kept.
    Updates the states in place and returns, per lane, whether it may guess
    in the next pass."""
    speculates = any(p > 0 for p in proposed)
    for b, s in enumerate(states):
        if s.wait > 0:
            if proposed[b] != 0 or kept[b] != 0:
                raise ValueError("a waiting lane makes no guesses")
            s.wait -= 1
            continue
        if not speculates:
            continue  # the pass counts toward no miss run
        if kept[b] > 0:
            s.misses = 0
            s.backoff = FIRST_WAIT
            continue
        s.misses += 1
        if s.misses == MISSES_TO_WAIT:
            s.wait = s.backoff
            s.backoff = min(2 * s.backoff, LONGEST_WAIT)
            s.misses = 0
    return [may_guess(s) for s in states]


def next_draft_lens(states, draft_tokens):
    """Guesses each lane may make in the next pass."""
    return [draft_tokens if may_guess(s) else 0 for s in states]
