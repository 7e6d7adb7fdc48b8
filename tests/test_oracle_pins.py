"""The CPU oracle against what the pages and the mathematics fix (no GPU)."""

import numpy as np
import pytest

import oracle
import oracle_checks as oc


@pytest.mark.parametrize("check", oc.ALL_CHECKS, ids=lambda f: f.__name__)
def test_pin(check):
    check()


def test_row_budget_rejects_bad_arguments():
    for args in [(3, 8, 0), (3, 8, -1), (-1, 8, 1), (3, -8, 1)]:
        with pytest.raises(ValueError):
            oracle.row_budget(*args)
    assert oracle.row_budget(7, 1024, 128) == 7
    assert oracle.row_budget(7, 1024, 129) == 6
    assert oracle.row_budget(0, 8, 1) == 0


def _lane(rows, drafts, temp=0.0, draft_rows=None):
    k = len(drafts)
    tok = np.full(k + 1, -1)
    tok[:k] = drafts
    return oracle.verify_round(np.asarray(rows, float), draft_rows, tok, [k], [0, k + 1],
                               np.array([temp], np.float32), seed=1)


def test_zero_drafts_commits_one_token():
    rows = np.array([[0.0, 2.0, 1.0]])
    res = _lane(rows, [])
    assert res.committed[0] == 1 and res.out_tokens[0] == 1
    res = _lane(rows, [], temp=1.0, draft_rows=np.zeros((1, 3)))
    assert res.committed[0] == 1 and 0 <= res.out_tokens[0] < 3


def test_ties_go_to_lowest_index_and_signed_zero():
    rows = np.array([[1.0, 3.0, 3.0, 2.0], [-0.0, 0.0, -1.0, -2.0]])
    res = _lane(rows, [1])
    assert res.out_tokens.tolist() == [1, 0]
    res = _lane(rows, [2])
    assert res.committed[0] == 1 and res.out_tokens[0] == 1


def test_negative_infinity_is_allowed_nan_and_pos_inf_are_not():
    rows = np.array([[-np.inf, 1.0, -np.inf], [0.0, -np.inf, 5.0]])
    assert _lane(rows, [1]).out_tokens.tolist() == [1, 2]
    for bad in [np.nan, np.inf]:
        r = rows.copy()
        r[1, 0] = bad
        res = _lane(r, [1])
        assert res.lane_status[0] == oracle.STATUS_NONFINITE and res.committed[0] == 0
        assert (res.out_tokens == -1).all()
    r = rows.copy()
    r[0, :] = -np.inf
    assert _lane(r, [1]).lane_status[0] == oracle.STATUS_NONFINITE


def test_draft_row_checked_only_where_read():
    # the last draft row of a lane is never read, so NaN there is harmless
    rows = np.array([[0.0, 1.0], [1.0, 0.0]])
    draft_rows = np.array([[0.0, 0.0], [np.nan, np.nan]])
    assert _lane(rows, [1], temp=0.5, draft_rows=draft_rows).lane_status[0] == 0
    draft_rows = np.array([[np.nan, 0.0], [0.0, 0.0]])
    assert _lane(rows, [1], temp=0.5, draft_rows=draft_rows).lane_status[0] == \
        oracle.STATUS_NONFINITE


def test_token_range_and_layout_errors():
    rows = np.zeros((6, 4))
    tok = np.array([0, 4, -1, 1, 2, -1])
    res = oracle.verify_round(rows, None, tok, [2, 2], [0, 3, 6], np.zeros(2, np.float32))
    assert res.lane_status.tolist() == [oracle.STATUS_TOKEN_RANGE, 0]
    tok = np.array([0, -5, -1, 1, 2, -1])
    res = oracle.verify_round(rows, None, tok, [2, 2], [0, 3, 6], np.zeros(2, np.float32))
    assert res.lane_status[0] == oracle.STATUS_TOKEN_RANGE
    res = oracle.verify_round(rows, None, tok, [2, 1], [0, 3, 6], np.zeros(2, np.float32))
    assert res.lane_status.tolist() == [oracle.STATUS_TOKEN_RANGE, oracle.STATUS_LAYOUT]
    res = oracle.verify_round(rows, None, tok, [2, 3], [0, 3, 7], np.zeros(2, np.float32))
    assert res.lane_status[1] == oracle.STATUS_LAYOUT
    res = oracle.verify_round(rows, None, tok, [2, 2], [0, 3, 6], np.array([0, 1], np.float32))
    assert res.lane_status[1] == oracle.STATUS_INVALID_ARG


def test_committed_run_bounds_random():
    rng = np.random.default_rng(0)
    for trial in range(30):
        lanes, vocab = 6, 9
        lens = rng.integers(0, 6, size=lanes)
        off = np.concatenate([[0], np.cumsum(lens + 1)])
        rows = rng.normal(size=(off[-1], vocab))
        drows = rows + rng.normal(size=rows.shape)
        tok = rng.integers(0, vocab, size=off[-1])
        temps = np.where(np.arange(lanes) % 2 == 1, 0.9, 0.0).astype(np.float32)
        res = oracle.verify_round(rows, drows, tok, lens, off, temps, seed=trial)
        assert (res.lane_status == 0).all()
        assert ((res.committed >= 1) & (res.committed <= lens + 1)).all()
        for b in range(lanes):
            c = res.committed[b]
            out = res.out_tokens[off[b]:off[b + 1]]
            assert (out[c:] == -1).all() and (out[:c] >= 0).all()
            # the accepted prefix is the drafts themselves
            assert (out[:c - 1] == tok[off[b]:off[b] + c - 1]).all()
