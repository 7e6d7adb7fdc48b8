"""The plain C++ statement of the oracle (oracle/verify_ref.cpp) against the same
facts that pin the numpy one, against the numpy one itself, and against
planted mistakes (no GPU).

The C++ oracle is built with g++ here; the pins of ``oracle_checks`` that
exercise the round, the row budget, the commit and the generator run with the
module-level functions of ``oracle`` replaced by the C++ ones.
"""

import numpy as np
import pytest
import torch

import oracle
import oracle_checks as oc
import workloads
from oracle import native

# The pins that go through the functions the C++ file provides.
NATIVE_CHECKS = [
    oc.check_row_budget_worked_example,
    oc.check_guess_check_table,
    oc.check_greedy_equals_plain_decode,
    oc.check_sampled_exact_enumeration,
    oc.check_sampled_monte_carlo,
    oc.check_sampled_special_cases,
    oc.check_inverse_cdf_never_draws_zero_weight,
    oc.check_expected_tokens_closed_form,
    oc.check_philox_against_numpy,
    oc.check_commit_copies_column_committed_minus_one,
    oc.check_penalties_on_a_round,
]

# Each planted mistake (OREF_MUTATE in verify_ref.cpp) and what it is.
MUTATIONS = {
    1: "acceptance ratio transposed (q/p)",
    2: "greedy draft checked against row j + 1",
    3: "argmax ties to the highest index",
    4: "temperature dropped",
    5: "non-strict inverse-CDF comparison",
    6: "residual transposed (q - p)",
    7: "row budget with ceiling division",
    8: "Philox with 9 rounds",
    9: "commit copies column c instead of c - 1",
}


def _use(monkeypatch, lib):
    monkeypatch.setattr(oracle, "verify_round",
                        lambda *a, **kw: native.verify_round(*a, threads=2, lib=lib, **kw))
    monkeypatch.setattr(oracle, "row_budget", lambda *a: native.row_budget(*a, lib=lib))
    monkeypatch.setattr(oracle, "commit_state", lambda *a, **kw: native.commit_state(*a, lib=lib, **kw))
    monkeypatch.setattr(oracle, "philox4x64_10", lambda c, k: native.philox4x64_10(c, k, lib=lib))
    monkeypatch.setattr(oracle, "round_uniforms", lambda *a: native.round_uniforms(*a, lib=lib))


@pytest.fixture(scope="module")
def lib():
    return native.load()


@pytest.mark.parametrize("check", NATIVE_CHECKS, ids=lambda f: f.__name__)
def test_native_pin(monkeypatch, lib, check):
    _use(monkeypatch, lib)
    check()


@pytest.mark.parametrize("mutation", sorted(MUTATIONS), ids=lambda m: MUTATIONS[m])
def test_a_planted_mistake_fails_a_pin(monkeypatch, mutation):
    bad = native.load(mutate=mutation)
    _use(monkeypatch, bad)
    failed = []
    for check in NATIVE_CHECKS:
        try:
            check()
        except AssertionError:
            failed.append(check.__name__)
    assert failed, f"no pin caught: {MUTATIONS[mutation]}"


def _bits(t):
    return t.view(torch.int16).numpy().view(np.uint16)


def _same_result(a, b, greedy_mask, lanes):
    for f in ("lane_status", "argmax"):
        np.testing.assert_array_equal(getattr(a, f), getattr(b, f), err_msg=f)
    for f in ("max_logit", "lse", "logp_d", "logq_d", "resid_mass"):
        x, y = getattr(a, f), getattr(b, f)
        np.testing.assert_array_equal(np.isnan(x), np.isnan(y), err_msg=f)
        np.testing.assert_allclose(x[~np.isnan(x)], y[~np.isnan(y)], rtol=1e-12, atol=1e-12, err_msg=f)
    for lane in range(lanes):
        near = any(m < 1e-9 for _, _, m in a.margins[lane])
        if greedy_mask[lane] or not near:
            assert a.committed[lane] == b.committed[lane], lane
        ma = {(k, p): m for k, p, m in a.margins[lane]}
        mb = {(k, p): m for k, p, m in b.margins[lane]}
        if not near:
            assert ma.keys() == mb.keys(), lane
            for key in ma:
                assert abs(ma[key] - mb[key]) <= 1e-9 or ma[key] == mb[key], (lane, key)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_native_equals_numpy_on_random_rounds(dtype, seed):
    """The two statements agree: greedy lanes and statuses exactly, float64
    statistics to 1e-12, sampled decisions wherever they are not within 1e-9
    of flipping (the two sum in different orders)."""
    r = workloads.make_custom_round(300 + seed, "cpu", lanes=23, vocab=3001 + seed, kmax=9, dtype=dtype,
                                    sampled="mixed")
    tok, lens, off, temps = (r.draft_tokens.numpy(), r.draft_lens.numpy(), r.row_offsets.numpy(),
                             r.temperatures.numpy())
    if dtype == "bf16":
        t_in, d_in = _bits(r.target), _bits(r.draft)
        t64, d64 = oracle.decode_bf16(t_in), oracle.decode_bf16(d_in)
    else:
        t_in, d_in = r.target.numpy(), r.draft.numpy()
        t64, d64 = t_in.astype(np.float64), d_in.astype(np.float64)
    a = oracle.verify_round(t64, d64, tok, lens, off, temps, seed=r.seed)
    b = native.verify_round(t_in, d_in, tok, lens, off, temps, seed=r.seed, threads=3)
    _same_result(a, b, temps <= 0, r.lanes)
    sure = [b_ for b_ in range(r.lanes) if not any(m < 1e-9 for _, _, m in a.margins[b_])]
    for lane in sure:
        lo, hi = off[lane], off[lane + 1]
        np.testing.assert_array_equal(a.out_tokens[lo:hi], b.out_tokens[lo:hi])


def test_native_statuses_and_edge_rows():
    """Non-finite rows, bad tokens, bad offsets and a missing drafter array give
    the numpy oracle's statuses and outputs."""
    r = workloads.make_custom_round(5, "cpu", lanes=8, vocab=200, kmax=4, dtype="f32", sampled="all", fixed_k=True)
    off = r.row_offsets.numpy()
    t, d = r.target.numpy().copy(), r.draft.numpy().copy()
    t[off[1] + 2, 7] = np.nan
    t[off[2], 5] = np.inf
    t[off[3] + 1, :] = -np.inf
    d[off[4], 3] = np.nan
    d[off[0] + 4, 9] = np.nan  # the lane's last drafter row: never read
    t[off[5]:off[6], ::3] = -np.inf
    tok = r.draft_tokens.numpy().copy()
    tok[off[6] + 1] = 200
    lens = r.draft_lens.numpy().copy()
    lens[7] = 3
    temps = r.temperatures.numpy()
    args = (tok, lens, off, temps)
    a = oracle.verify_round(t.astype(np.float64), d.astype(np.float64), *args, seed=9)
    b = native.verify_round(t, d, *args, seed=9, threads=4)
    assert b.lane_status.tolist() == [0, 4, 4, 4, 4, 0, 5, 6]
    _same_result(a, b, temps <= 0, 8)
    np.testing.assert_array_equal(a.out_tokens, b.out_tokens)
    b = native.verify_round(t, None, *args, seed=9)
    assert (b.lane_status[[0, 5]] == oracle.STATUS_INVALID_ARG).all()


def test_native_threads_do_not_change_results():
    r = workloads.make_custom_round(17, "cpu", lanes=30, vocab=5000, kmax=7, dtype="bf16", sampled="mixed")
    args = (_bits(r.target), _bits(r.draft), r.draft_tokens.numpy(), r.draft_lens.numpy(), r.row_offsets.numpy(),
            r.temperatures.numpy())
    one, used1 = native.verify_round(*args, seed=r.seed, threads=1, return_threads=True)
    many, used = native.verify_round(*args, seed=r.seed, threads=7, return_threads=True)
    assert used1 == 1 and used == 7
    for f in ("committed", "out_tokens", "lane_status", "argmax", "max_logit"):
        np.testing.assert_array_equal(getattr(one, f), getattr(many, f), err_msg=f)
    for f in ("lse", "logp_d", "logq_d", "resid_mass"):
        np.testing.assert_array_equal(getattr(one, f), getattr(many, f), err_msg=f)


def test_native_uniforms_equal_the_numpy_generator():
    for seed, lane, pos in [(0, 0, 0), (2 ** 64 - 1, 2 ** 32 + 3, 15), (0x0123456789ABCDEF, 77, 4)]:
        assert native.round_uniforms(seed, lane, pos) == oracle.round_uniforms(seed, lane, pos)
