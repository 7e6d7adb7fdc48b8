"""Seeded synthetic inputs for the verify round.

This module only makes inputs: logits, draft tokens, per-lane draft lengths,
row offsets, temperatures, Philox seeds and recurrent-state snapshots.  It holds
none of the verify round's arithmetic, so both the CUDA library and the CPU
oracle can be fed from it.  Everything is drawn with a seeded ``torch.Generator``
on the requested device; the same (workload, seed, device type) always gives the
same tensors.

The five named workloads follow the shapes and value distributions that the
verify-round benchmark description fixes (no public dataset is involved):

  greedy_b1_k3_v1024_f32      1 lane, k=3, V=1024, fp32 logits ~ N(0, 3);
                              each draft is its row's argmax w.p. 0.7, else a
                              uniform token; greedy.
  greedy_b8_k7_v151936        8 lanes, k=7, V=151936, bf16 logits ~ N(0, 2)
                              plus +8 on one uniformly chosen "true" token per
                              row; drafts are the row's argmax w.p. 0.8 i.i.d.,
                              else uniform; greedy.
  sampled_b8_k7_v151936       as above, plus drafter logits = target + N(0, 1)
                              (fp32 sum rounded to bf16), temperature 0.7, each
                              draft drawn from q = softmax(drafter row / T) by the
                              Gumbel-max trick.
  greedy_commit_b64_k3_v151936
                              64 lanes, k=3, V=151936 greedy as the 8-lane case,
                              with fp32 recurrent-state snapshots of
                              [4 columns][24 layers][16 heads][128 x 128] per lane.
  ragged_mixed_b128_v262144   128 lanes, k_b ~ U{0..7} (the most a budget of
                              1024 rows allows 128 lanes at 7 draft tokens),
                              V=262144 bf16; even lanes greedy, odd lanes sampled
                              with T ~ U[0.3, 1.2] and drafts from q.

The second parameter of every N(., .) is the standard deviation.
"""

import dataclasses
from typing import Optional

import torch

GREEDY_TINY = "greedy_b1_k3_v1024_f32"
GREEDY_B8 = "greedy_b8_k7_v151936"
SAMPLED_B8 = "sampled_b8_k7_v151936"
GREEDY_COMMIT_B64 = "greedy_commit_b64_k3_v151936"
RAGGED_MIXED_B128 = "ragged_mixed_b128_v262144"

WORKLOADS = (GREEDY_TINY, GREEDY_B8, SAMPLED_B8, GREEDY_COMMIT_B64, RAGGED_MIXED_B128)

# The ragged workload is described as "row budget 1024" over 128 lanes with up
# to 7 draft tokens; the per-lane draft cap it implies is computed by the
# callers (library and oracle) and checked against this value.
RAGGED_DRAFT_TOKENS = 7
RAGGED_ROW_BUDGET = 1024

# Shape of one recurrent-state snapshot of the commit workload:
# [24 layers][16 heads][128][128] fp32 = 24 MiB per column.
STATE_SHAPE = (24, 16, 128, 128)


@dataclasses.dataclass
class RoundInputs:
    """All inputs of one verify round (plus optional recurrent state)."""

    name: str
    vocab: int
    lanes: int
    rows: int
    dtype: str                     # 'bf16' or 'f32' (both logits arrays)
    target: torch.Tensor           # [rows, vocab]
    draft: Optional[torch.Tensor]  # [rows, vocab] or None (no sampled lane)
    draft_tokens: torch.Tensor     # int32 [rows]; slot off[b]+j holds d_{j+1}
    draft_lens: torch.Tensor       # int32 [lanes]
    row_offsets: torch.Tensor      # int32 [lanes + 1]
    temperatures: torch.Tensor     # float32 [lanes]; <= 0 is greedy
    seed: int                      # Philox key of the round's uniforms
    staged: Optional[torch.Tensor] = None  # float32 [lanes, cols, elems]
    live: Optional[torch.Tensor] = None    # float32 [lanes, elems]

    def to(self, device):
        """Copy of the round with every tensor on ``device``."""
        kw = {}
        for f in dataclasses.fields(self):
            v = getattr(self, f.name)
            kw[f.name] = v.to(device) if isinstance(v, torch.Tensor) else v
        return RoundInputs(**kw)

    def logits_bytes(self):
        """Bytes of the target (+ draft) logits arrays."""
        n = self.target.numel() * self.target.element_size()
        if self.draft is not None:
            n += self.draft.numel() * self.draft.element_size()
        return n


def _gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _spiked_logits(g, rows, vocab, sigma, spike, device):
    """fp32 N(0, sigma) with +spike at one uniform 'true' token per row."""
    x = torch.randn(rows, vocab, generator=g, device=device) * sigma
    if spike:
        true_tok = torch.randint(0, vocab, (rows,), generator=g, device=device)
        x[torch.arange(rows, device=device), true_tok] += spike
    return x


def _argmax_or_uniform_drafts(g, target32, lens, offsets, alpha, device):
    """d_{j+1} = argmax(row j) w.p. alpha, else a uniform token (per position)."""
    rows, vocab = target32.shape
    best = torch.argmax(target32, dim=1)
    rand_tok = torch.randint(0, vocab, (rows,), generator=g, device=device)
    keep = torch.rand(rows, generator=g, device=device) < alpha
    tokens = torch.where(keep, best, rand_tok).to(torch.int32)
    return _blank_last_slot(tokens, lens, offsets)


def _drafts_from_q(g, draft32, temps_per_row, lens, offsets, device, chunk=64):
    """d_{j+1} ~ softmax(drafter row j / T) by Gumbel-max: argmax(y/T + G)."""
    rows, vocab = draft32.shape
    out = torch.empty(rows, dtype=torch.int64, device=device)
    for r0 in range(0, rows, chunk):
        r1 = min(rows, r0 + chunk)
        u = torch.rand(r1 - r0, vocab, generator=g, device=device, dtype=torch.float64)
        u = u.clamp_min(torch.finfo(torch.float64).tiny)
        gumbel = -torch.log(-torch.log(u))
        t = temps_per_row[r0:r1].to(torch.float64).clamp_min(1e-6)[:, None]
        out[r0:r1] = torch.argmax(draft32[r0:r1].to(torch.float64) / t + gumbel, dim=1)
    return _blank_last_slot(out.to(torch.int32), lens, offsets)


def _blank_last_slot(tokens, lens, offsets):
    """The slot after each lane's last draft is unused: set it to -1."""
    last = (offsets[1:] - 1).long()
    tokens = tokens.clone()
    tokens[last] = -1
    return tokens


def _offsets(lens):
    off = torch.zeros(lens.shape[0] + 1, dtype=torch.int64, device=lens.device)
    off[1:] = torch.cumsum(lens.long() + 1, 0)
    return off.to(torch.int32)


def _per_row(values, lens, offsets):
    """Expand a per-lane tensor to one entry per row."""
    counts = (offsets[1:] - offsets[:-1]).long()
    return torch.repeat_interleave(values, counts)


def make_round(name, seed=0, device="cpu", with_state=True, commit_lanes=None):
    """Inputs of one named workload (see the module docstring).

    ``with_state=False`` skips the recurrent-state snapshots of the commit
    workload (callers that share one state between several logits sets).
    ``commit_lanes`` shrinks the commit workload to fewer lanes (same shapes
    per lane), for profiler captures that must stay small.
    """
    device = torch.device(device)
    g = _gen(seed, device)
    philox_seed = (int(seed) * 0x9E3779B97F4A7C15 + 0x5EED) & ((1 << 64) - 1)
    if name == GREEDY_TINY:
        return _fixed_k_round(name, g, device, lanes=1, k=3, vocab=1024, sigma=3.0,
                              spike=0.0, alpha=0.7, dtype="f32", temperature=0.0,
                              seed=philox_seed)
    if name == GREEDY_B8:
        return _fixed_k_round(name, g, device, lanes=8, k=7, vocab=151936, sigma=2.0,
                              spike=8.0, alpha=0.8, dtype="bf16", temperature=0.0,
                              seed=philox_seed)
    if name == SAMPLED_B8:
        return _fixed_k_round(name, g, device, lanes=8, k=7, vocab=151936, sigma=2.0,
                              spike=8.0, alpha=None, dtype="bf16", temperature=0.7,
                              seed=philox_seed)
    if name == GREEDY_COMMIT_B64:
        lanes = 64 if commit_lanes is None else int(commit_lanes)
        r = _fixed_k_round(name, g, device, lanes=lanes, k=3, vocab=151936, sigma=2.0,
                           spike=8.0, alpha=0.8, dtype="bf16", temperature=0.0,
                           seed=philox_seed)
        if with_state:
            r.staged, r.live = make_state(lanes, 4, STATE_SHAPE, seed, device)
        return r
    if name == RAGGED_MIXED_B128:
        return _ragged_round(name, g, device, lanes=128, kmax=RAGGED_DRAFT_TOKENS,
                             vocab=262144, seed=philox_seed)
    raise ValueError(f"unknown workload {name!r}")


def make_custom_round(seed, device, lanes, vocab, kmax, dtype="bf16", sampled="mixed",
                      sigma=2.0, spike=8.0, alpha=0.8, fixed_k=False, ld=None,
                      temperature_range=(0.3, 1.2)):
    """Small random round for parity tests.

    sampled: 'none' | 'all' | 'mixed' (odd lanes sampled).  ``ld`` > vocab pads
    every row (the padding holds large values that must never be read).
    """
    device = torch.device(device)
    g = _gen(seed, device)
    if fixed_k:
        lens = torch.full((lanes,), kmax, dtype=torch.int32, device=device)
    else:
        lens = torch.randint(0, kmax + 1, (lanes,), generator=g, device=device).to(torch.int32)
    off = _offsets(lens)
    rows = int(off[-1])
    lane_ids = torch.arange(lanes, device=device)
    if sampled == "none":
        is_sampled = torch.zeros(lanes, dtype=torch.bool, device=device)
    elif sampled == "all":
        is_sampled = torch.ones(lanes, dtype=torch.bool, device=device)
    else:
        is_sampled = (lane_ids % 2) == 1
    lo, hi = temperature_range
    temps = lo + (hi - lo) * torch.rand(lanes, generator=g, device=device)
    temps = torch.where(is_sampled, temps, torch.zeros_like(temps)).to(torch.float32)
    t32 = _spiked_logits(g, rows, vocab, sigma, spike, device)
    d32 = None
    if bool(is_sampled.any()):
        d32 = t32 + torch.randn(rows, vocab, generator=g, device=device)
    target, draft = _store(t32, dtype), (_store(d32, dtype) if d32 is not None else None)
    greedy_tok = _argmax_or_uniform_drafts(g, target.float(), lens, off, alpha, device)
    if draft is not None:
        q_tok = _drafts_from_q(g, draft.float(), _per_row(temps, lens, off), lens, off, device)
        tokens = torch.where(_per_row(is_sampled, lens, off), q_tok, greedy_tok)
    else:
        tokens = greedy_tok
    if ld is not None and ld > vocab:
        target = _pad_rows(target, ld)
        if draft is not None:
            draft = _pad_rows(draft, ld)
    seed64 = (int(seed) * 0xD1B54A32D192ED03 + 7) & ((1 << 64) - 1)
    return RoundInputs("custom", vocab, lanes, rows, dtype, target, draft, tokens, lens,
                       off, temps, seed64)


def _pad_rows(x, ld):
    """Rows of length ld whose first vocab entries are x; padding = huge value."""
    rows, vocab = x.shape
    pad = torch.full((rows, ld), 3.0e38, dtype=x.dtype, device=x.device)
    pad[:, :vocab] = x
    return pad


def _store(x32, dtype):
    if dtype == "bf16":
        return x32.to(torch.bfloat16)
    if dtype == "f32":
        return x32.to(torch.float32)
    raise ValueError(dtype)


def _fixed_k_round(name, g, device, lanes, k, vocab, sigma, spike, alpha, dtype,
                   temperature, seed):
    lens = torch.full((lanes,), k, dtype=torch.int32, device=device)
    off = _offsets(lens)
    rows = lanes * (k + 1)
    t32 = _spiked_logits(g, rows, vocab, sigma, spike, device)
    target = _store(t32, dtype)
    temps = torch.full((lanes,), float(temperature), dtype=torch.float32, device=device)
    draft = None
    if temperature > 0:
        draft = _store(t32 + torch.randn(rows, vocab, generator=g, device=device), dtype)
        del t32
        tokens = _drafts_from_q(g, draft.float(), _per_row(temps, lens, off), lens, off, device)
    else:
        del t32
        tokens = _argmax_or_uniform_drafts(g, target.float(), lens, off, alpha, device)
    return RoundInputs(name, vocab, lanes, rows, dtype, target, draft, tokens, lens, off,
                       temps, seed)


def _ragged_round(name, g, device, lanes, kmax, vocab, seed):
    lens = torch.randint(0, kmax + 1, (lanes,), generator=g, device=device).to(torch.int32)
    off = _offsets(lens)
    rows = int(off[-1])
    lane_ids = torch.arange(lanes, device=device)
    is_sampled = (lane_ids % 2) == 1
    temps = 0.3 + 0.9 * torch.rand(lanes, generator=g, device=device)
    temps = torch.where(is_sampled, temps, torch.zeros_like(temps)).to(torch.float32)
    target = torch.empty(rows, vocab, dtype=torch.bfloat16, device=device)
    draft = torch.empty(rows, vocab, dtype=torch.bfloat16, device=device)
    chunk = 64
    for r0 in range(0, rows, chunk):
        r1 = min(rows, r0 + chunk)
        t32 = _spiked_logits(g, r1 - r0, vocab, 2.0, 8.0, device)
        target[r0:r1] = t32.to(torch.bfloat16)
        draft[r0:r1] = (t32 + torch.randn(r1 - r0, vocab, generator=g, device=device)).to(torch.bfloat16)
    greedy_tok = _argmax_or_uniform_drafts(g, target.float(), lens, off, 0.8, device)
    q_tok = _drafts_from_q(g, draft.float(), _per_row(temps, lens, off), lens, off, device)
    tokens = torch.where(_per_row(is_sampled, lens, off), q_tok, greedy_tok)
    return RoundInputs(name, vocab, lanes, rows, "bf16", target, draft, tokens, lens, off,
                       temps, seed)


# ---------------------------------------------------------------------------
# Recurrent-state snapshots
# ---------------------------------------------------------------------------

_H1 = 0x7FEB352D
_H2 = 0x2C1B3C6D
_H3 = 0x297A2D39
_M32 = 0xFFFFFFFF


def _mix32(x):
    """A 32-bit integer mixing hash on int64 tensors (values kept < 2^32)."""
    x = x & _M32
    x = x ^ (x >> 16)
    x = (x * _H1) & _M32
    x = x ^ (x >> 15)
    x = (x * _H2) & _M32
    x = x ^ (x >> 16)
    return x


def state_block(lane, col, elems, seed, device="cpu"):
    """float32 [elems]: the snapshot of (lane, col); finite values in +-[1, 2).

    The bit pattern of element i is a hash of (seed, lane, col, i), so a copy
    from the wrong lane, column or offset is visible in every element.
    """
    i = torch.arange(elems, dtype=torch.int64, device=device)
    salt = _mix32(torch.tensor([(int(seed) * _H3 + lane * 0x10001 + col * 0x3F1) & _M32],
                               dtype=torch.int64, device=device))
    h = _mix32(i ^ salt)
    bits = (h & 0x007FFFFF) | 0x3F800000 | ((h & 1) << 31)
    bits = torch.where(bits >= (1 << 31), bits - (1 << 32), bits)
    return bits.to(torch.int32).view(torch.float32)


def make_state(lanes, cols, shape, seed, device):
    """staged [lanes, cols, elems] and live [lanes, elems] fp32 snapshots.

    Live starts as a distinct block (column index ``cols``) so a lane that is
    not committed is recognisable.
    """
    elems = 1
    for s in shape:
        elems *= s
    staged = torch.empty(lanes, cols, elems, dtype=torch.float32, device=device)
    live = torch.empty(lanes, elems, dtype=torch.float32, device=device)
    for b in range(lanes):
        for c in range(cols):
            staged[b, c] = state_block(b, c, elems, seed, device)
        live[b] = state_block(b, cols, elems, seed, device)
    return staged, live
