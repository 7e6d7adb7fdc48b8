"""CPU oracle of the speculative-decoding verify round (float64, plain numpy).

TEST INFRASTRUCTURE ONLY.  This module defines what the verify round computes
so that the CUDA library can be checked against it.  Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference leg may
import it.  It shares no code, header, constant table or helper with the CUDA
library and never calls it.

Sources (page title, then section):

* ignis docs, "Speculative decoding" -- "One round, step by step": each lane
  holds an anchor and up to k drafts; the model scores the k + 1 columns in one
  pass; the longest run of drafts the model would itself have chosen is
  accepted, plus the model's own token after it, so the committed run holds 1
  to k + 1 tokens; the state advances by exactly the committed run.
* ignis docs, "Speculative decoding" -- "The row budget": drafts per lane are
  min(draft tokens, rows / lanes - 1), and a budget of 0 means 8.
* strata2signal, "Draft heads and speculative decoding, in plain words" --
  "Guess, then check" and its table: row j scores the position after the j-th
  guess; guesses are kept while they match, the model's own token is kept at the
  first mismatch; the distribution is kept "with the right acceptance rule"
  (Leviathan, Kalman and Matias 2022; Chen et al. 2023).
* The acceptance rule itself is the textbook one of those papers: accept draft
  d with probability min(1, p(d) / q(d)); at the first rejection draw from the
  normalised residual max(0, p - q); if every draft is accepted draw a bonus
  token from the last target row.
* FreeToken issue #828 -- "Design", per-request state: the verify forward only
  stages per-column scratch and ``commit`` rolls the state to the accepted
  count.

Readings where the pages are silent (each is listed in the design notes):

* ties in argmax go to the lowest token id; -0.0 equals +0.0;
* -inf logits are allowed (probability 0); NaN or +inf anywhere in a row that
  is read, or a row that is -inf everywhere, fails the lane (status NONFINITE);
* row j of a lane is checked against draft d_{j+1}; draft logits use the same
  row numbering as target logits and their last row per lane is not read;
* a lane with temperature <= 0 is greedy; a sampled lane's q uses the same
  temperature as its p;
* p(d) = 0 rejects; q(d) = 0 with p(d) > 0 accepts;
* the inverse-CDF draw walks tokens in ascending id and takes the first
  cumulative weight strictly above u' * W; if rounding leaves no such token it
  takes the largest id of positive weight; a residual of total mass 0 falls
  back to p;
* staged state column c holds the state after consuming column c (column 0
  is the anchor), so the commit copies column (committed - 1).
"""

import dataclasses

import numpy as np

from . import philox

# Per-lane status codes.  Their numbers are part of the library's public
# contract and are restated here, not imported.
STATUS_OK = 0
STATUS_INVALID_ARG = 1
STATUS_UNSUPPORTED = 2
STATUS_CUDA = 3
STATUS_NONFINITE = 4
STATUS_TOKEN_RANGE = 5
STATUS_LAYOUT = 6
STATUS_TIMEOUT = 7

DEFAULT_ROW_BUDGET = 8  # ignis, "The row budget": 0, the default, means 8


# ---------------------------------------------------------------------------
# Row budget
# ---------------------------------------------------------------------------

def row_budget(draft_tokens, rows, lanes):
    """Drafts each lane may carry: min(draft_tokens, rows // lanes - 1), >= 0.

    ignis docs, "Speculative decoding" -- "The row budget".  ``rows == 0``
    means the default budget of 8.  Division is floor division (a budget of 8
    over 3 lanes gives 8 // 3 - 1 = 1 draft, as the page's worked example
    says) and the result is clamped at 0 ("none from five lanes on").
    """
    if lanes <= 0 or draft_tokens < 0 or rows < 0:
        raise ValueError("row_budget: lanes must be > 0 and the others >= 0")
    if rows == 0:
        rows = DEFAULT_ROW_BUDGET
    return max(0, min(draft_tokens, rows // lanes - 1))


# ---------------------------------------------------------------------------
# Input decoding
# ---------------------------------------------------------------------------

def decode_bf16(bits):
    """bfloat16 bit patterns (uint16) -> float64, exactly.

    A bfloat16 is the top half of an IEEE float32, so shifting its 16 bits
    into the high half of a 32-bit word gives that float32, which widens to
    float64 without rounding.
    """
    bits = np.asarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def decode_logits(array, dtype):
    """Logits as stored ('bf16' bit patterns or 'f32' values) -> float64."""
    if dtype == "bf16":
        return decode_bf16(array)
    if dtype == "f32":
        return np.asarray(array, dtype=np.float32).astype(np.float64)
    raise ValueError(f"unknown logits dtype {dtype!r}")


# ---------------------------------------------------------------------------
# Per-row reductions
# ---------------------------------------------------------------------------

def row_is_valid(row):
    """A row can be reduced: no NaN, no +inf, and not -inf everywhere."""
    if np.isnan(row).any() or np.isposinf(row).any():
        return False
    return bool(np.isfinite(row).any())


def argmax_lowest(row):
    """Index of the largest logit; ties go to the lowest index.

    strata2signal "Guess, then check": at temperature zero the model "always
    takes its single most likely token".  numpy's argmax returns the first
    maximal element and compares -0.0 equal to +0.0.
    """
    return int(np.argmax(row))


def softmax_at_temperature(row, temperature):
    """p = softmax(row / T) in float64, with its log-sum-exp.

    Returns (p, lse) where lse = log(sum(exp(row / T))).  -inf logits get
    probability exactly 0.
    """
    z = row / float(temperature)
    zmax = np.max(z)
    e = np.exp(z - zmax)
    total = np.sum(e)
    return e / total, float(zmax + np.log(total))


# ---------------------------------------------------------------------------
# Acceptance and resampling (the textbook rule)
# ---------------------------------------------------------------------------

def acceptance_ratio(p_d, q_d):
    """p(d) / q(d) with the edge cases fixed: p(d) = 0 -> 0, q(d) = 0 -> inf."""
    if p_d == 0.0:
        return 0.0
    if q_d == 0.0:
        return np.inf
    return p_d / q_d


def accept_draft(u, p_d, q_d):
    """Accept draft d iff u < min(1, p(d) / q(d))."""
    return u < min(1.0, acceptance_ratio(p_d, q_d))


def residual_weights(p, q):
    """Unnormalised residual max(0, p - q) of the first rejected position."""
    return np.maximum(0.0, p - q)


def inverse_cdf(weights, u):
    """Draw a token from unnormalised ``weights`` with uniform ``u``.

    Walks ids in ascending order and returns the first x whose cumulative
    weight is strictly above u * W (W = total weight).  If rounding leaves no
    such x, returns the largest x of positive weight.  Also returns the
    distance from u * W to the nearest cumulative boundary, divided by W, which
    says how close the draw came to picking a neighbour.
    """
    cdf = np.cumsum(weights)
    total = cdf[-1]
    target = u * total
    above = np.nonzero(cdf > target)[0]
    if above.size:
        token = int(above[0])
    else:
        token = int(np.nonzero(weights > 0)[0][-1])
    margin = min(abs(target), float(np.min(np.abs(cdf - target)))) / total
    return token, margin


# ---------------------------------------------------------------------------
# The round
# ---------------------------------------------------------------------------

@dataclasses.dataclass
class RoundResult:
    """Oracle outputs of one verify round.

    committed  [lanes] committed-run length c_b in 1..k_b+1 (0 if the lane failed)
    out_tokens [rows]  committed tokens at off[b] + i for i < c_b, else -1
    lane_status[lanes] STATUS_* per lane
    argmax     [rows]  argmax of each target row that was read (-1 otherwise)
    max_logit  [rows]  largest raw logit of each target row that was read
    lse        [rows]  log-sum-exp of row / T (sampled lanes; NaN otherwise)
    logp_d     [rows]  log p_j(d_{j+1}) (sampled lanes, j < k_b; NaN otherwise)
    logq_d     [rows]  log q_j(d_{j+1}) (sampled lanes, j < k_b; NaN otherwise)
    resid_mass [rows]  sum max(0, p_n - q_n) at the rejected row n (NaN otherwise)
    margins    [lanes] list of (kind, position, margin): how far each random
               decision of the lane was from flipping (fp64).  Kind 'accept':
               |u - p/q|; kind 'draw': distance of u' to the nearest CDF
               boundary, in units of the drawn distribution's total mass.
    """

    committed: np.ndarray
    out_tokens: np.ndarray
    lane_status: np.ndarray
    argmax: np.ndarray
    max_logit: np.ndarray
    lse: np.ndarray
    logp_d: np.ndarray
    logq_d: np.ndarray
    resid_mass: np.ndarray
    margins: list


def _lane_layout_ok(b, k, off, rows):
    start, end = int(off[b]), int(off[b + 1])
    return k >= 0 and start >= 0 and end <= rows and end - start == k + 1


def verify_round(target, draft, draft_tokens, draft_lens, row_offsets,
                 temperatures, seed=0, u_acc=None, u_smp=None, lane_base=0):
    """One verify round over all lanes.

    target        float64 [rows, V] target logits (already decoded)
    draft         float64 [rows, V] drafter logits, same row numbering; may be
                  None when no lane samples
    draft_tokens  int [rows]; draft_tokens[off[b] + j] = d_{j+1} for j < k_b
    draft_lens    int [lanes]; k_b >= 0
    row_offsets   int [lanes + 1]; off[b+1] - off[b] must be k_b + 1
    temperatures  float32 [lanes]; <= 0 means greedy
    seed          Philox key for the uniforms (see ``philox.round_uniforms``)
    u_acc, u_smp  optional [lanes, >= k_b + 1] arrays of uniforms that replace
                  the Philox ones (used by tests that enumerate the uniforms)
    lane_base     global index of lane 0 in the Philox counter (a batch split
                  into parts draws the uniforms of the unsplit batch)
    """
    target = np.asarray(target, dtype=np.float64)
    rows, vocab = target.shape
    draft_tokens = np.asarray(draft_tokens).astype(np.int64)
    draft_lens = np.asarray(draft_lens).astype(np.int64)
    off = np.asarray(row_offsets).astype(np.int64)
    temps = np.asarray(temperatures, dtype=np.float32).astype(np.float64)
    lanes = draft_lens.shape[0]

    res = RoundResult(
        committed=np.zeros(lanes, np.int32),
        out_tokens=np.full(rows, -1, np.int32),
        lane_status=np.zeros(lanes, np.int32),
        argmax=np.full(rows, -1, np.int64),
        max_logit=np.full(rows, np.nan),
        lse=np.full(rows, np.nan),
        logp_d=np.full(rows, np.nan),
        logq_d=np.full(rows, np.nan),
        resid_mass=np.full(rows, np.nan),
        margins=[[] for _ in range(lanes)],
    )

    for b in range(lanes):
        k = int(draft_lens[b])
        if not _lane_layout_ok(b, k, off, rows):
            res.lane_status[b] = STATUS_LAYOUT
            continue
        base = int(off[b])
        drafts = draft_tokens[base:base + k]
        if ((drafts < 0) | (drafts >= vocab)).any():
            res.lane_status[b] = STATUS_TOKEN_RANGE
            continue
        sampled = temps[b] > 0.0
        if sampled and draft is None:
            res.lane_status[b] = STATUS_INVALID_ARG
            continue
        t_rows = [target[base + j] for j in range(k + 1)]
        q_rows = [np.asarray(draft[base + j], np.float64) for j in range(k)] if sampled else []
        if not all(row_is_valid(r) for r in t_rows + q_rows):
            res.lane_status[b] = STATUS_NONFINITE
            continue

        for j, r in enumerate(t_rows):
            res.argmax[base + j] = argmax_lowest(r)
            res.max_logit[base + j] = float(np.max(r))

        if not sampled:
            tokens = _greedy_lane(t_rows, drafts)
        else:
            ua = [None] * (k + 1)
            us = [None] * (k + 1)
            for j in range(k + 1):
                if u_acc is None or u_smp is None:
                    ua[j], us[j] = philox.round_uniforms(seed, lane_base + b, j)
                if u_acc is not None:
                    ua[j] = float(u_acc[b][j])
                if u_smp is not None:
                    us[j] = float(u_smp[b][j])
            tokens = _sampled_lane(t_rows, q_rows, drafts, temps[b], ua, us,
                                   res, base, res.margins[b])

        c = len(tokens)
        res.committed[b] = c
        res.out_tokens[base:base + c] = tokens
    return res


def _greedy_lane(t_rows, drafts):
    """Greedy lane: keep drafts while d_{j+1} == argmax(row j), then the model's token.

    ignis "One round, step by step", step 4, and the strata2signal
    "Guess, then check" table.  Returns the committed tokens a_0 .. a_n.
    """
    k = len(drafts)
    a = [argmax_lowest(r) for r in t_rows]
    n = 0
    while n < k and int(drafts[n]) == a[n]:
        n += 1
    return a[:n + 1]


def _sampled_lane(t_rows, q_rows, drafts, temperature, ua, us, res, base, margins):
    """Sampled lane: the textbook accept / residual / bonus rule.

    For j = 0 .. k-1 accept d_{j+1} iff u_j < min(1, p_j(d) / q_j(d)) and stop
    at the first rejection n.  If n < k the model's token is drawn from
    max(0, p_n - q_n) (normalised); if every draft was accepted it is a bonus
    draw from p_k.  Returns d_1 .. d_n and the drawn token.
    """
    k = len(drafts)
    p = []
    for j, r in enumerate(t_rows):
        pj, lse = softmax_at_temperature(r, temperature)
        p.append(pj)
        res.lse[base + j] = lse
    q = [softmax_at_temperature(r, temperature)[0] for r in q_rows]

    n = k
    for j in range(k):
        d = int(drafts[j])
        p_d, q_d = float(p[j][d]), float(q[j][d])
        res.logp_d[base + j] = np.log(p_d) if p_d > 0 else -np.inf
        res.logq_d[base + j] = np.log(q_d) if q_d > 0 else -np.inf
        if n == k:
            margins.append(("accept", j, abs(ua[j] - acceptance_ratio(p_d, q_d))))
            if not accept_draft(ua[j], p_d, q_d):
                n = j

    if n < k:
        w = residual_weights(p[n], q[n])
        res.resid_mass[base + n] = float(np.sum(w))
        if not (w > 0).any():
            w = p[n]
    else:
        w = p[k]
    token, margin = inverse_cdf(w, us[n])
    margins.append(("draw", n, margin))
    return [int(d) for d in drafts[:n]] + [token]


# ---------------------------------------------------------------------------
# State commit
# ---------------------------------------------------------------------------

def commit_state(staged, live, committed, lane_status=None):
    """Roll each lane's live state to its committed count.

    staged [lanes, cols, nbytes] uint8 -- column c is the state after
    consuming column c of the round (column 0 is the anchor);
    live   [lanes, nbytes] uint8 -- the state before the round.
    Returns the new live state: lane b gets staged[b, committed[b] - 1]
    (ignis "One round, step by step", step 5; FreeToken #828 "Design",
    per-request state).  A lane whose count is outside 1..cols, or whose
    status is not OK, keeps its live state, so nothing of a failed or
    rejected column reaches it.
    """
    staged = np.asarray(staged)
    out = np.array(live, copy=True)
    cols = staged.shape[1]
    for b in range(staged.shape[0]):
        c = int(committed[b])
        if lane_status is not None and int(lane_status[b]) != STATUS_OK:
            continue
        if 1 <= c <= cols:
            out[b] = staged[b, c - 1]
    return out


def commit_status(committed, cols, lane_status=None):
    """Per-lane status the commit reports: LAYOUT for a count outside 1..cols.

    A lane already failed by the verify keeps its status.
    """
    committed = np.asarray(committed)
    out = np.zeros(committed.shape[0], np.int32)
    for b in range(committed.shape[0]):
        if lane_status is not None and int(lane_status[b]) != STATUS_OK:
            out[b] = int(lane_status[b])
        elif not 1 <= int(committed[b]) <= cols:
            out[b] = STATUS_LAYOUT
    return out
