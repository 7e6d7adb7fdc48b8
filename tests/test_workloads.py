"""The synthetic workloads have the shapes and value structure their recipe
states (generated on the CPU; no GPU needed)."""

import numpy as np
import pytest
import torch

import workloads
from conftest import cpu_round


def _f(t):
    return t.float().numpy().astype(np.float64)


def _draft_matches_argmax(r):
    """Fraction of drafts d_{j+1} equal to the argmax of row j (greedy lanes)."""
    best = torch.argmax(r.target.float(), dim=1).numpy()
    off, k = r.row_offsets.numpy(), r.draft_lens.numpy()
    hits = total = 0
    for b in range(r.lanes):
        for j in range(int(k[b])):
            hits += int(r.draft_tokens[off[b] + j]) == int(best[off[b] + j])
            total += 1
    return hits, total


@pytest.mark.parametrize("name,lanes,k,vocab,dtype,sampled", [
    (workloads.GREEDY_TINY, 1, 3, 1024, torch.float32, False),
    (workloads.GREEDY_B8, 8, 7, 151936, torch.bfloat16, False),
    (workloads.SAMPLED_B8, 8, 7, 151936, torch.bfloat16, True),
    (workloads.GREEDY_COMMIT_B64, 64, 3, 151936, torch.bfloat16, False),
])
def test_fixed_length_workloads(name, lanes, k, vocab, dtype, sampled):
    r = cpu_round(name, seed=3)
    assert (r.lanes, r.vocab, r.rows) == (lanes, vocab, lanes * (k + 1))
    assert r.target.dtype == dtype and tuple(r.target.shape) == (r.rows, vocab)
    assert (r.draft_lens.numpy() == k).all()
    assert (r.row_offsets.numpy() == np.arange(lanes + 1) * (k + 1)).all()
    assert (r.draft is not None) == sampled
    temps = r.temperatures.numpy()
    assert (temps == 0.7).all() if sampled else (temps <= 0).all()
    x = _f(r.target[:32])
    sigma = 3.0 if name == workloads.GREEDY_TINY else 2.0
    # the bulk of each row is N(0, sigma): its middle quantiles
    q25, q75 = np.percentile(x, [25, 75])
    assert abs((q75 - q25) / 1.349 - sigma) < 0.05 * sigma
    if name != workloads.GREEDY_TINY:
        # +8 at one token per row lifts the row maxima above those of plain
        # N(0, sigma) rows of the same width (mean 8.8 there, 9.5 here)
        plain = np.random.default_rng(1).standard_normal((64, vocab)) * sigma
        row_max = r.target.float().amax(dim=1).numpy()
        assert row_max.mean() - plain.max(axis=1).mean() > 0.3
    if sampled:
        noise = _f(r.draft[:32]) - x
        assert abs(noise.std() - 1.0) < 0.05
    else:
        hits, total = _draft_matches_argmax(r)
        if name == workloads.GREEDY_B8 or name == workloads.GREEDY_COMMIT_B64:
            alpha = 0.8
            assert abs(hits / total - alpha) < 4 * np.sqrt(alpha * (1 - alpha) / total), (hits, total)


def test_the_tiny_workload_matches_drafts_seventy_percent_of_the_time():
    hits = total = 0
    for seed in range(60):
        h, t = _draft_matches_argmax(workloads.make_round(workloads.GREEDY_TINY, seed=seed, device="cpu"))
        hits, total = hits + h, total + t
    assert abs(hits / total - 0.7) < 4 * np.sqrt(0.21 / total), (hits, total)


def test_the_ragged_workload():
    r = cpu_round(workloads.RAGGED_MIXED_B128, seed=0)
    k = r.draft_lens.numpy()
    off = r.row_offsets.numpy()
    assert r.lanes == 128 and r.vocab == 262144 and r.target.dtype == torch.bfloat16
    assert k.min() >= 0 and k.max() <= workloads.RAGGED_DRAFT_TOKENS and len(np.unique(k)) >= 6
    assert off[0] == 0 and (np.diff(off) == k + 1).all() and off[-1] == r.rows
    assert r.rows <= workloads.RAGGED_ROW_BUDGET
    temps = r.temperatures.numpy()
    assert (temps[0::2] <= 0).all()
    assert ((temps[1::2] >= 0.3) & (temps[1::2] <= 1.2)).all() and temps[1::2].std() > 0.15
    assert r.draft is not None and r.draft.shape == r.target.shape


def test_state_snapshots_are_finite_distinct_and_reproducible():
    n = 1 << 16
    a = workloads.state_block(3, 1, n, seed=9)
    assert a.dtype == torch.float32 and torch.equal(a, workloads.state_block(3, 1, n, seed=9))
    mag = a.abs()
    assert torch.isfinite(a).all() and (mag >= 1).all() and (mag < 2).all()
    assert 0.45 < (a < 0).float().mean() < 0.55
    # another lane, column or seed differs in (nearly) every element
    for other in (workloads.state_block(4, 1, n, seed=9), workloads.state_block(3, 2, n, seed=9),
                  workloads.state_block(3, 1, n, seed=10)):
        assert (a == other).float().mean() < 1e-3
    # element i depends on i: a shifted copy does not match
    assert (a[1:] == a[:-1]).float().mean() < 1e-3
    staged, live = workloads.make_state(2, 3, (4, 8), seed=9, device="cpu")
    assert tuple(staged.shape) == (2, 3, 32) and tuple(live.shape) == (2, 32)
    assert torch.equal(staged[1, 2], workloads.state_block(1, 2, 32, seed=9))
    assert torch.equal(live[0], workloads.state_block(0, 3, 32, seed=9))
