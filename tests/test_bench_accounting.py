"""bench.py's byte accounting on the CPU: the algorithmic bytes of each
workload (the rows every round must read, at their element size, plus the
per-lane metadata and outputs) and the DRAM traffic it takes from the committed
ncu summaries."""

import numpy as np
import pytest

import bench
import workloads
from conftest import cpu_round

V = 151936


def _meta_out(rows, lanes):
    # draft tokens, lengths, offsets, temperatures; committed, out_tokens, status
    return 4 * (rows + lanes + (lanes + 1) + lanes) + 4 * (lanes + rows + lanes)


def test_greedy_round_reads_every_target_row_once():
    r = cpu_round(workloads.GREEDY_B8)
    total, rows = bench.round_bytes(r)
    assert rows == 64
    assert total - _meta_out(64, 8) == 64 * V * 2 == 19_447_808


def test_sampled_round_adds_the_drafter_rows():
    r = cpu_round(workloads.SAMPLED_B8)
    total, rows = bench.round_bytes(r)
    # 8 target rows and 7 drafter rows per lane (the bonus row has no drafter row)
    assert rows == 64 and total - _meta_out(64, 8) == (64 + 56) * V * 2 == 36_464_640


def test_ragged_round_counts_drafter_rows_of_sampled_lanes_only():
    r = cpu_round(workloads.RAGGED_MIXED_B128)
    total, rows = bench.round_bytes(r)
    k = r.draft_lens.numpy().astype(np.int64)
    sampled = r.temperatures.numpy() > 0
    assert rows == int((k + 1).sum()) == r.rows
    assert total - _meta_out(r.rows, 128) == (r.rows + int(k[sampled].sum())) * 262144 * 2


def test_commit_moves_one_snapshot_in_and_out_per_lane():
    r = workloads.make_round(workloads.GREEDY_COMMIT_B64, seed=0, device="cpu", commit_lanes=1)
    snapshot = 24 * 16 * 128 * 128 * 4  # fp32 [24][16][128][128]
    assert snapshot == 25_165_824
    assert bench.commit_bytes(r) == 2 * snapshot + 8
    total, rows = bench.round_bytes(r)
    assert rows == 4 and total - _meta_out(4, 1) == 4 * V * 2


def _profile_field(name, field):
    with open(f"{bench.ROOT}/profiles/{name}") as f:
        for line in f:
            if line.startswith(field + ":"):
                return line.split(":", 1)[1].strip()
    raise KeyError(field)


@pytest.mark.parametrize("kernel,workload,scale", [
    ("verify_accept", workloads.GREEDY_B8, 1),
    ("verify_accept", workloads.SAMPLED_B8, 1),
    ("commit_state", workloads.GREEDY_COMMIT_B64, 4),
])
def test_traffic_comes_from_the_summary_of_the_same_kernel_source(kernel, workload, scale, monkeypatch):
    name = f"{kernel}_{workload}.txt"
    if _profile_field(name, "kernel_source_sha256") != bench.kernel_source_hash():
        pytest.skip("the kernel changed since its counters were taken")
    dram = float(_profile_field(name, "dram_bytes_per_launch"))
    def mbytes(field):
        value, unit = _profile_field(name, field).split()
        return float(value) * {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}[unit]
    # the per-launch traffic is the read plus the write counter of the capture
    assert abs(mbytes("dram__bytes_read.sum") + mbytes("dram__bytes_write.sum") - dram) <= 1e3
    assert bench.profiled_traffic(kernel, workload) == int(dram * scale)
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0" * 16)
    assert bench.profiled_traffic(kernel, workload) is None


def test_no_summary_means_no_traffic():
    assert bench.profiled_traffic("verify_accept", "no_such_workload") is None


def _oracle_outputs(r):
    import oracle
    import torch
    bits = lambda t: t.view(torch.int16).numpy().view(np.uint16)
    full = oracle.verify_round(oracle.decode_bf16(bits(r.target)), oracle.decode_bf16(bits(r.draft)),
                               r.draft_tokens.numpy(), r.draft_lens.numpy(), r.row_offsets.numpy(),
                               r.temperatures.numpy(), seed=r.seed)
    return full, {"committed": torch.from_numpy(full.committed.copy()),
                  "out_tokens": torch.from_numpy(full.out_tokens.copy())}


def test_oracle_parity_counts_every_lane_of_the_inputs_it_is_given():
    r = workloads.make_custom_round(7, "cpu", lanes=6, vocab=500, kmax=5, dtype="bf16", sampled="mixed")
    full, out = _oracle_outputs(r)
    par = bench.cpu_oracle_parity(r, out)
    assert par["lanes"] == 6 and par["mismatch"] == 0 and par["sampled_exempt"] == 0
    assert par["greedy_equal"] + par["sampled_equal"] == 6
    assert par["greedy_equal"] == par["greedy_lanes"] and par["sampled_equal"] == par["sampled_lanes"] >= 1
    assert par["tokens_equal"] == par["rows"]
    # a greedy lane that differs is a mismatch, never an exemption
    greedy = int(np.nonzero(r.temperatures.numpy() <= 0)[0][0])
    out["committed"][greedy] += 1
    out["out_tokens"][int(r.row_offsets[greedy])] = -7
    par = bench.cpu_oracle_parity(r, out)
    assert par["mismatch"] == 1 and par["tokens_equal"] == par["rows"] - 1


def test_oracle_parity_exempts_only_sampled_decisions_near_a_flip():
    """A sampled lane whose acceptance uniform sits within 1e-5 of p/q may
    differ (exempt); moved away from the boundary the same difference is a
    mismatch."""
    r = workloads.make_custom_round(8, "cpu", lanes=4, vocab=300, kmax=3, dtype="bf16", sampled="all",
                                    fixed_k=True)
    full, out = _oracle_outputs(r)
    out["committed"][1] = 1 if int(full.committed[1]) != 1 else 2
    par = bench.cpu_oracle_parity(r, out, exempt_tol=1e-5)
    assert par["mismatch"] == 1 and par["sampled_exempt"] == 0
    par = bench.cpu_oracle_parity(r, out, exempt_tol=2.0)  # every decision "near a flip"
    assert par["mismatch"] == 0 and par["sampled_exempt"] == 1


def test_cpu_baseline_times_a_sample_of_whole_lanes():
    r = workloads.make_custom_round(7, "cpu", lanes=6, vocab=500, kmax=5, dtype="bf16", sampled="mixed")
    line = bench.cpu_baseline("unused", 0, budget_s=0.2, gpu_round=r)
    assert line["kind"] == "oracle" and line["cores"] >= 1 and line["value"] > 0 and line["unit"] == "rows/s"


def test_l2_note_states_whether_the_input_sets_leave_l2():
    """Tiny rounds rotate over 16 sets that all stay in L2; the note says so
    instead of claiming the sets leave L2 between reuses."""
    b = object.__new__(bench.Bench)
    b.sets, b.set_bytes = [None] * 16, 16440
    assert "L2-resident" in b.l2_note()
    b.sets, b.set_bytes = [None] * 2, 590_000_000
    note = b.l2_note()
    assert "more than the 129 MB L2" in note and "590 MB between reuses" in note
