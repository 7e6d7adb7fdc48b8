"""Splitting a verify round's lanes across ranks.

Lanes are independent in every step of the round (the row sweep, the
acceptance scan, the draw -- whose uniforms are keyed by the lane's global
index -- and the state commit), so a batch splits into contiguous lane ranges
with no exchange.  A part verified with ``lane_base`` = its first global lane
gives exactly the results of the unsplit batch for those lanes.
"""


def lane_range(lanes, world, rank):
    """Contiguous, balanced [lo, hi) lane range of ``rank`` out of ``world``."""
    if world <= 0 or not 0 <= rank < world or lanes < 0:
        raise ValueError("lane_range: need world > 0, 0 <= rank < world, lanes >= 0")
    base, extra = divmod(lanes, world)
    lo = rank * base + min(rank, extra)
    hi = lo + base + (1 if rank < extra else 0)
    return lo, hi


def shard_rows(row_offsets, lo, hi):
    """Rows [row_lo, row_hi) of lanes [lo, hi) and their offsets rebased to 0.

    ``row_offsets`` is the host copy (any int sequence) of the round's
    [lanes + 1] offsets.
    """
    offs = [int(x) for x in row_offsets]
    row_lo, row_hi = offs[lo], offs[hi]
    return row_lo, row_hi, [o - row_lo for o in offs[lo:hi + 1]]
