"""Per-row presence and frequency penalties on the target logits of a round.

TEST INFRASTRUCTURE ONLY (see the package docstring).

FreeToken tracking issue #828, "PRs" (#836, target-side verify: rejection
sampling with per-row presence and frequency penalties) names the feature and
not its formula; the reading taken is the usual one.  For token t with count
c_j(t) in row j,

    z = x - (presence * [c_j(t) > 0] + frequency * c_j(t)),

where row j of a lane scores the position after the anchor and d_1..d_j, so
c_j(t) is the token's count in the lane's history plus its count among
d_1..d_j.  The drafter's rows are not changed (q is what the drafter drew
from).  Arithmetic, in this order, in fp32: m = fl(frequency * c),
delta = fl(m + presence) (presence only when c > 0, else delta = m),
z = fl(x - delta); a bf16 logit is then rounded back to bf16 (round to
nearest, ties to even), since the penalty is applied to the stored logit.
Tokens with c_j(t) = 0 are untouched.

Plain numpy on the decoded (float64-held) values.
"""

import numpy as np


def round_to_bf16(x32):
    """float32 -> the nearest bfloat16 value (ties to even), held as float32.
    Finite inputs only."""
    bits = np.asarray(x32, np.float32).view(np.uint32).astype(np.uint64)
    lsb = (bits >> np.uint64(16)) & np.uint64(1)
    rounded = ((bits + np.uint64(0x7FFF) + lsb) >> np.uint64(16)) << np.uint64(16)
    return rounded.astype(np.uint32).view(np.float32)


def row_counts(history_counts, drafts, j):
    """Counts of row j: the history's counts plus d_1..d_j (a dict token -> count)."""
    c = dict(history_counts)
    for t in drafts[:j]:
        c[int(t)] = c.get(int(t), 0) + 1
    return c


def penalise_value(x, c, presence, frequency, dtype):
    """The penalised logit of one token with count c > 0 (see the module docstring)."""
    m = np.float32(np.float32(frequency) * np.float32(c))
    delta = np.float32(m + np.float32(presence)) if c > 0 else m
    z = np.float32(np.float32(x) - delta)
    return float(round_to_bf16(z)) if dtype == "bf16" else float(z)


def apply_penalties(target, dtype, draft_tokens, draft_lens, row_offsets, pen_tokens, pen_counts, pen_offsets,
                    presence, frequency):
    """A penalised copy of the target rows (float64 array [rows, V] of decoded
    values).  Lane b's history counts are pen_tokens / pen_counts
    [pen_offsets[b] .. pen_offsets[b + 1]) (unique tokens)."""
    out = np.array(target, dtype=np.float64, copy=True)
    V = out.shape[1]
    for b in range(len(draft_lens)):
        k, off = int(draft_lens[b]), int(row_offsets[b])
        hist = {int(pen_tokens[i]): int(pen_counts[i]) for i in range(int(pen_offsets[b]), int(pen_offsets[b + 1]))}
        drafts = [int(draft_tokens[off + j]) for j in range(k)]
        for j in range(k + 1):
            for t, c in row_counts(hist, drafts, j).items():
                if c > 0 and 0 <= t < V:
                    out[off + j, t] = penalise_value(target[off + j, t], c, presence[b], frequency[b], dtype)
    return out
