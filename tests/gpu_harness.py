"""Run one verify round through the C ABI and through the CPU oracle, and compare.

Tolerances (derived from the arithmetic; see the design notes):

* greedy lanes, committed counts, tokens, argmax and max logit: bit-exact;
* a sampled acceptance decision may differ only where the oracle's float64
  |u - p(d)/q(d)| < 1e-5;
* a sampled draw may differ only where u' lies within 1e-5 + 4e-6 / W of a
  cumulative boundary of the drawn distribution (normalised units; W is the
  residual mass, 1 for a bonus draw): the GPU sums fp32 weights whose absolute
  errors add up to at most about 2e-6;
* log p(d), log q(d) and the log-sum-exp: within 1e-5 (absolute in log space,
  i.e. 1e-5 relative on the probabilities);
* residual mass: within 1e-5 * W + 2e-6.
"""

import numpy as np
import torch

import oracle
import speculative_decoding_verify_bf16_gb300 as sv

ACCEPT_TOL = 1e-5
LOG_TOL = 1e-5


def draw_tol(mass):
    return 1e-5 + 4e-6 / max(float(mass), 1e-30)


def logits_to_numpy(t, vocab):
    t = t[:, :vocab]
    if t.dtype == torch.bfloat16:
        bits = t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
        return oracle.decode_bf16(bits)
    return t.float().cpu().numpy().astype(np.float64)


def run_gpu(r, stats=True, stream=None):
    """Verify round r (device tensors) through the binding; numpy results."""
    dev = r.target.device
    lanes, rows = r.lanes, r.rows
    committed = torch.full((lanes,), -7, dtype=torch.int32, device=dev)
    out_tokens = torch.full((rows,), -7, dtype=torch.int32, device=dev)
    status = torch.full((lanes,), -7, dtype=torch.int32, device=dev)
    row_stats = sv.new_row_stats(rows, dev).fill_(-7) if stats else None
    target = r.target[:, :r.vocab]
    draft = r.draft[:, :r.vocab] if r.draft is not None else None
    sv.spec_verify_accept(target, draft, r.draft_tokens, r.draft_lens, r.row_offsets,
                          r.temperatures, r.seed, committed, out_tokens, status, row_stats,
                          stream=stream, rows=rows)
    torch.cuda.synchronize()
    res = {"committed": committed.cpu().numpy(), "out_tokens": out_tokens.cpu().numpy(),
           "lane_status": status.cpu().numpy()}
    if stats:
        res.update({k: v.cpu().numpy() for k, v in sv.row_stats_view(row_stats).items()})
    return res


def run_oracle(r):
    target = logits_to_numpy(r.target, r.vocab)
    draft = logits_to_numpy(r.draft, r.vocab) if r.draft is not None else None
    return oracle.verify_round(target, draft, r.draft_tokens.cpu().numpy(),
                               r.draft_lens.cpu().numpy(), r.row_offsets.cpu().numpy(),
                               r.temperatures.cpu().numpy(), seed=r.seed)


def lane_exempt(orc, b):
    """True if a random decision of lane b fell within the tolerance band."""
    for kind, pos, margin in orc.margins[b]:
        if kind == "accept" and margin < ACCEPT_TOL:
            return True
        if kind == "draw":
            mass = orc.resid_mass[pos] if np.isfinite(orc.resid_mass[pos]) else 1.0
            if mass == 0.0:
                mass = 1.0
            if margin < draw_tol(mass):
                return True
    return False


def compare(r, gpu, orc, check_stats=True, max_exempt_frac=1e-3):
    """Assert GPU == oracle on round r; returns (lanes compared, lanes exempt)."""
    off = r.row_offsets.cpu().numpy()
    lens = r.draft_lens.cpu().numpy()
    temps = r.temperatures.cpu().numpy()
    np.testing.assert_array_equal(gpu["lane_status"], orc.lane_status, err_msg="lane_status")
    exempt = 0
    for b in range(r.lanes):
        k = int(lens[b])
        lo, hi = int(off[b]), int(off[b]) + k + 1
        st = int(orc.lane_status[b])
        if st != oracle.STATUS_OK:
            assert gpu["committed"][b] == 0, (b, gpu["committed"][b])
            if st != oracle.STATUS_LAYOUT:
                assert (gpu["out_tokens"][lo:hi] == -1).all(), b
            continue
        sampled = temps[b] > 0
        if sampled and lane_exempt(orc, b):
            exempt += 1
            continue
        assert gpu["committed"][b] == orc.committed[b], (b, gpu["committed"][b], orc.committed[b])
        np.testing.assert_array_equal(gpu["out_tokens"][lo:hi], orc.out_tokens[lo:hi],
                                      err_msg=f"lane {b} tokens")
        if not check_stats or "argmax" not in gpu:
            continue
        np.testing.assert_array_equal(gpu["argmax"][lo:hi], orc.argmax[lo:hi], err_msg=f"lane {b} argmax")
        np.testing.assert_array_equal(gpu["max_logit"][lo:hi].astype(np.float64), orc.max_logit[lo:hi],
                                      err_msg=f"lane {b} max_logit")
        if sampled:
            np.testing.assert_allclose(gpu["lse"][lo:hi], orc.lse[lo:hi], rtol=0, atol=LOG_TOL,
                                       err_msg=f"lane {b} lse")
            for name in ("logp_d", "logq_d"):
                g = gpu[name][lo:hi - 1].astype(np.float64)
                o = getattr(orc, name)[lo:hi - 1]
                fin = np.isfinite(o)
                assert (np.isfinite(g) == fin).all(), (b, name, g, o)
                np.testing.assert_allclose(g[fin], o[fin], rtol=0, atol=LOG_TOL, err_msg=f"lane {b} {name}")
            n = int(orc.committed[b]) - 1
            assert gpu["drawn"][lo + n] == orc.out_tokens[lo + n]
            if np.isfinite(orc.resid_mass[lo + n]):
                w = orc.resid_mass[lo + n]
                assert abs(gpu["resid_mass"][lo + n] - w) <= 1e-5 * w + 2e-6, (b, gpu["resid_mass"][lo + n], w)
    n_sampled = int((temps > 0).sum())
    if n_sampled:
        assert exempt <= max(1, max_exempt_frac * n_sampled), (exempt, n_sampled)
    return r.lanes, exempt
