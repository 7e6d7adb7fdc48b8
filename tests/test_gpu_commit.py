"""GPU parity: the state-commit kernel against the oracle's commit, through the C ABI."""

import numpy as np
import pytest
import torch

import oracle
import workloads
import speculative_decoding_verify_bf16_gb300 as sv

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    sv.build_library()
    sv.load_library()


def _bytes(t):
    return t.contiguous().view(torch.uint8).cpu().numpy()


def _check(staged, live0, live1, committed, status_in, status_out):
    lanes, cols = staged.shape[0], staged.shape[1]
    st = _bytes(staged).reshape(lanes, cols, -1)
    l0 = _bytes(live0).reshape(lanes, -1)
    want = oracle.commit_state(st, l0, committed, status_in)
    np.testing.assert_array_equal(_bytes(live1).reshape(lanes, -1), want)
    np.testing.assert_array_equal(status_out, oracle.commit_status(committed, cols, status_in))


@pytest.mark.parametrize("elems,dtype", [(4096, torch.float32), (1025, torch.float32),
                                         (77, torch.uint8), (3 * 2 ** 16 + 4, torch.float32),
                                         (40000, torch.bfloat16)])
def test_commit_matches_oracle(elems, dtype):
    g = torch.Generator(device=DEV)
    g.manual_seed(elems)
    lanes, cols = 9, 5
    if dtype == torch.uint8:
        staged = torch.randint(0, 256, (lanes, cols, elems), generator=g, device=DEV, dtype=torch.uint8)
        live = torch.randint(0, 256, (lanes, elems), generator=g, device=DEV, dtype=torch.uint8)
    else:
        staged = torch.randn(lanes, cols, elems, generator=g, device=DEV).to(dtype)
        live = torch.randn(lanes, elems, generator=g, device=DEV).to(dtype)
    committed = torch.tensor([1, 5, 3, 0, 6, 2, 4, 1, 5], dtype=torch.int32, device=DEV)
    status = torch.tensor([0, 0, 0, 0, 0, 4, 0, 0, 0], dtype=torch.int32, device=DEV)
    status_in = status.cpu().numpy().copy()
    live0 = live.clone()
    sv.spec_commit_state(staged, live, committed, status)
    torch.cuda.synchronize()
    _check(staged, live0, live, committed.cpu().numpy(), status_in, status.cpu().numpy())


def test_commit_without_status_buffer():
    lanes, cols, elems = 4, 3, 1000
    staged = torch.arange(lanes * cols * elems, dtype=torch.float32, device=DEV).view(lanes, cols, elems)
    live = torch.full((lanes, elems), -1.0, device=DEV)
    committed = torch.tensor([3, 1, 2, 4], dtype=torch.int32, device=DEV)  # 4 > cols: kept
    live0 = live.clone()
    sv.spec_commit_state(staged, live, committed)
    torch.cuda.synchronize()
    _check(staged, live0, live, committed.cpu().numpy(), None, oracle.commit_status(
        committed.cpu().numpy(), cols))


def test_verify_then_commit_on_one_stream():
    """The commit reads the verify's committed counts (programmatic dependent launch)."""
    r = workloads.make_custom_round(3, DEV, lanes=16, vocab=30000, kmax=5, dtype="bf16",
                                    sampled="mixed", fixed_k=True)
    cols, elems = 6, 50000
    staged, live = workloads.make_state(16, cols, (elems,), 5, DEV)
    live0 = live.clone()
    committed = torch.zeros(16, dtype=torch.int32, device=DEV)
    out = torch.empty(r.rows, dtype=torch.int32, device=DEV)
    status = torch.empty(16, dtype=torch.int32, device=DEV)
    for _ in range(3):  # back to back, nothing in between
        live.copy_(live0)
        sv.spec_verify_accept(r.target, r.draft, r.draft_tokens, r.draft_lens, r.row_offsets,
                              r.temperatures, r.seed, committed, out, status)
        sv.spec_commit_state(staged, live, committed, status)
    torch.cuda.synchronize()
    c = committed.cpu().numpy()
    assert (c >= 1).all() and (c <= 6).all()
    _check(staged, live0, live, c, np.zeros(16, np.int32), status.cpu().numpy())


def test_commit_workload_full_size():
    """64 lanes x 24 MiB snapshots: every lane checked on the device, three against
    snapshots regenerated on the host."""
    r = workloads.make_round(workloads.GREEDY_COMMIT_B64, seed=7, device=DEV)
    committed = torch.zeros(r.lanes, dtype=torch.int32, device=DEV)
    out = torch.empty(r.rows, dtype=torch.int32, device=DEV)
    status = torch.empty(r.lanes, dtype=torch.int32, device=DEV)
    sv.spec_verify_accept(r.target, r.draft, r.draft_tokens, r.draft_lens, r.row_offsets,
                          r.temperatures, r.seed, committed, out, status)
    sv.spec_commit_state(r.staged, r.live, committed, status)
    torch.cuda.synchronize()
    c = committed.cpu().numpy()
    assert (status.cpu().numpy() == 0).all()
    for b in range(r.lanes):
        assert torch.equal(r.live[b], r.staged[b, c[b] - 1]), b
    elems = r.staged.shape[2]
    for b in (0, 31, 63):
        want = workloads.state_block(b, int(c[b]) - 1, elems, 7, "cpu")
        assert torch.equal(r.live[b].cpu(), want), b


def test_a_load_that_never_lands_fails_every_lane_it_leaves_unfinished(monkeypatch):
    """SPEC_COMMIT_TEST_WITHHOLD_COPY: the commit's first CTA announces its
    first load but never issues it.  Its wait gives up after 2 s; every lane
    that CTA still had loads in flight or work left for reports
    SPEC_ERR_TIMEOUT, and no lane reports OK without its full snapshot in
    live state.  A plain commit afterwards is exact again."""
    import time

    lanes, cols, elems = 12, 4, 3 * 2 ** 15  # 384 KB a snapshot: several chunks a lane
    g = torch.Generator(device=DEV)
    g.manual_seed(5)
    staged = torch.randn(lanes, cols, elems, generator=g, device=DEV)
    live = torch.randn(lanes, elems, generator=g, device=DEV)
    committed = torch.tensor([1, 2, 3, 4] * 3, dtype=torch.int32, device=DEV)
    status = torch.zeros(lanes, dtype=torch.int32, device=DEV)
    live0 = live.clone()
    monkeypatch.setenv("SPEC_COMMIT_TEST_WITHHOLD_COPY", "1")
    torch.cuda.synchronize()
    t0 = time.time()
    sv.spec_commit_state(staged, live, committed, status)
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    st = status.cpu().numpy()
    assert 1.5 < elapsed < 60, elapsed
    assert set(st.tolist()) <= {sv.SPEC_OK, sv.SPEC_ERR_TIMEOUT} and (st == sv.SPEC_ERR_TIMEOUT).any(), st
    c = committed.cpu().numpy()
    for b in range(lanes):
        if st[b] == sv.SPEC_OK:
            assert torch.equal(live[b], staged[b, c[b] - 1]), b
    monkeypatch.delenv("SPEC_COMMIT_TEST_WITHHOLD_COPY")
    status.zero_()
    live.copy_(live0)
    sv.spec_commit_state(staged, live, committed, status)
    torch.cuda.synchronize()
    _check(staged, live0, live, c, np.zeros(lanes, np.int32), status.cpu().numpy())
