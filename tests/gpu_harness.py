"""Run one verify round through the C ABI and through the CPU oracle, and compare.

Tolerances (derived from the arithmetic; see the design notes):

* greedy lanes, committed counts, tokens, argmax and max logit: bit-exact;
* a sampled acceptance decision may differ only where the oracle's float64
  |u - p(d)/q(d)| < 1e-5;
* a drawn token may differ only if it is still an inverse-CDF draw of the
  oracle's float64 weights with u' * W moved by at most 1e-5 * W (W is the
  total weight of the drawn distribution: the residual mass, or 1 for a draw
  from p), i.e. where the oracle's draw lay within 1e-5 of a CDF boundary in
  normalised units;
* exemptions (acceptance decisions or draws allowed to differ) are counted,
  and a comparison fails if they exceed 1e-3 of its sampled lanes, rounded
  up (so one in a comparison of fewer than 1000 sampled lanes);
* log p(d), log q(d) and the log-sum-exp: within 1e-5 (absolute in log space,
  i.e. 1e-5 relative on the probabilities);
* residual mass: within 1e-5 * W + 2e-6.
"""

import numpy as np
import torch

import oracle
import speculative_decoding_verify_bf16_gb300 as sv

ACCEPT_TOL = 1e-5
DRAW_TOL = 1e-5
LOG_TOL = 1e-5
EXEMPT_FRAC = 1e-3


def exemption_cap(sampled_lanes):
    """Most exempted decisions one comparison accepts: 1e-3 of its sampled
    lanes, rounded up (none without a sampled lane)."""
    return int(np.ceil(EXEMPT_FRAC * sampled_lanes - 1e-9)) if sampled_lanes > 0 else 0


def logits_to_numpy(t, vocab):
    t = t[:, :vocab]
    if t.dtype == torch.bfloat16:
        bits = t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
        return oracle.decode_bf16(bits)
    return t.float().cpu().numpy().astype(np.float64)


def run_gpu(r, stats=True, stream=None, meta_before_wait=False):
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
                          stream=stream, rows=rows, meta_before_wait=meta_before_wait)
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


def _draw_row_weights(r, orc, b, n, target, draft):
    """Oracle-side (float64) weights of the draw made at position n of lane b."""
    off = int(r.row_offsets[b])
    k = int(r.draft_lens[b])
    temp = float(r.temperatures[b])
    p_n, _ = oracle.softmax_at_temperature(target[off + n], temp)
    if n < k:
        q_n, _ = oracle.softmax_at_temperature(draft[off + n], temp)
        w = oracle.residual_weights(p_n, q_n)
        if (w > 0).any():
            return w
    return p_n


def draw_is_valid(r, orc, b, n, token, u_draw, target, draft):
    """The GPU's drawn token is an inverse-CDF draw of the oracle's weights, up to tolerance.

    Token x is valid iff C(x) - w(x) - tau <= u' * W <= C(x) + tau, with C the
    float64 cumulative weight and tau = 1e-5 * W.
    """
    w = _draw_row_weights(r, orc, b, n, target, draft)
    cdf = np.cumsum(w)
    total = cdf[-1]
    tau = DRAW_TOL * total
    t = u_draw * total
    return (cdf[token] - w[token] - tau <= t <= cdf[token] + tau), w[token]


def compare(r, gpu, orc, check_stats=True, oracle_inputs=None):
    """Assert GPU == oracle on round r.

    Greedy lanes, statuses and row statistics must match exactly / to LOG_TOL.
    A sampled lane must match too, except where the oracle shows the decision
    on which the two differ was within tolerance of flipping; such exemptions
    may number at most 1e-3 of the sampled lanes.  Returns a dict of counts.
    """
    off = r.row_offsets.cpu().numpy()
    lens = r.draft_lens.cpu().numpy()
    temps = r.temperatures.cpu().numpy()
    np.testing.assert_array_equal(gpu["lane_status"], orc.lane_status, err_msg="lane_status")
    counts = {"lanes": r.lanes, "sampled": int((temps > 0).sum()), "accept_flips": 0, "draw_flips": 0,
              "exempted": []}
    target = draft = None
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
        if check_stats and "argmax" in gpu:
            _compare_row_stats(gpu, orc, b, lo, hi, sampled)
        c_g, c_o = int(gpu["committed"][b]), int(orc.committed[b])
        t_g, t_o = gpu["out_tokens"][lo:hi], orc.out_tokens[lo:hi]
        if sampled and (c_g != c_o or not np.array_equal(t_g, t_o)):
            n_g, n_o = c_g - 1, c_o - 1
            if n_g != n_o:
                j = min(n_g, n_o)
                margin = dict(((kind, pos), m) for kind, pos, m in orc.margins[b])[("accept", j)]
                assert margin < ACCEPT_TOL, (b, "acceptance differs", j, margin)
                counts["accept_flips"] += 1
                counts["exempted"].append(("accept", b, j, float(margin)))
            else:
                np.testing.assert_array_equal(t_g[:n_g], t_o[:n_o])
                if target is None:
                    target, draft = oracle_inputs if oracle_inputs else (
                        logits_to_numpy(r.target, r.vocab),
                        logits_to_numpy(r.draft, r.vocab) if r.draft is not None else None)
                u_draw = oracle.round_uniforms(r.seed, b, n_g)[1]
                ok, wx = draw_is_valid(r, orc, b, n_g, int(t_g[n_g]), u_draw, target, draft)
                assert ok, (b, "draw differs beyond tolerance", int(t_g[n_g]), int(t_o[n_o]), wx)
                counts["draw_flips"] += 1
                dm = dict(((kind, pos), m) for kind, pos, m in orc.margins[b]).get(("draw", n_o), float("nan"))
                counts["exempted"].append(("draw", b, n_g, int(t_g[n_g]), int(t_o[n_o]), float(dm), float(wx)))
            assert (t_g[c_g:] == -1).all()
            continue
        assert c_g == c_o, (b, c_g, c_o)
        np.testing.assert_array_equal(t_g, t_o, err_msg=f"lane {b} tokens")
        if not check_stats or "argmax" not in gpu:
            continue
        if sampled:
            n = c_o - 1
            assert gpu["drawn"][lo + n] == orc.out_tokens[lo + n]
            if np.isfinite(orc.resid_mass[lo + n]):
                w = orc.resid_mass[lo + n]
                assert abs(gpu["resid_mass"][lo + n] - w) <= 1e-5 * w + 2e-6, (b, gpu["resid_mass"][lo + n], w)
    exempt = counts["accept_flips"] + counts["draw_flips"]
    assert exempt <= exemption_cap(counts["sampled"]), ("exemptions above 1e-3 of the sampled lanes", counts)
    return counts


def _compare_row_stats(gpu, orc, b, lo, hi, sampled):
    """Decision-independent row statistics: argmax, max logit, lse, log p(d), log q(d)."""
    np.testing.assert_array_equal(gpu["argmax"][lo:hi], orc.argmax[lo:hi], err_msg=f"lane {b} argmax")
    np.testing.assert_array_equal(gpu["max_logit"][lo:hi].astype(np.float64), orc.max_logit[lo:hi],
                                  err_msg=f"lane {b} max_logit")
    if not sampled:
        return
    # lse is reported as an fp32 number: at |lse| ~ 10^3 (low temperatures) its
    # own rounding, |lse| * 2^-24, exceeds LOG_TOL, so that rounding is allowed on top.
    np.testing.assert_allclose(gpu["lse"][lo:hi], orc.lse[lo:hi], rtol=2.0 ** -23, atol=LOG_TOL,
                               err_msg=f"lane {b} lse")
    for name in ("logp_d", "logq_d"):
        g = gpu[name][lo:hi - 1].astype(np.float64)
        o = getattr(orc, name)[lo:hi - 1]
        fin = np.isfinite(o)
        assert (np.isfinite(g) == fin).all(), (b, name, g, o)
        np.testing.assert_allclose(g[fin], o[fin], rtol=0, atol=LOG_TOL, err_msg=f"lane {b} {name}")
