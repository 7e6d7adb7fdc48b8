"""A greedy speculative decoding loop built from the library's pieces, on the GPU.

Per round: the n-gram drafter proposes from each lane's history, the miss
back-off caps the draft lengths, a toy model scores the k_b + 1 columns, the
verify kernel commits, and the acceptance counts and back-off state advance.
Greedy speculation must emit exactly what plain argmax decoding emits
(strata2signal "Guess, then check"; ignis "One round, step by step"), and the
device's counts and back-off state must equal the oracle's over the same rounds.
"""

import numpy as np
import pytest
import torch

import workloads
from oracle import backoff as ob
from oracle import metrics as om
from oracle import ngram as ong

import speculative_decoding_verify_bf16_gb300 as sv

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


class TrigramLM:
    """A deterministic model whose logits depend on the last two tokens only, so
    that greedy decoding falls into cycles the n-gram drafter can copy."""

    def __init__(self, vocab, seed):
        self.vocab, self.seed = vocab, seed

    def logits(self, prefix):
        h = hash((self.seed, int(prefix[-2]), int(prefix[-1]))) & 0xFFFFFFFF
        return np.round(np.random.default_rng(h).normal(size=self.vocab) * 4.0) / 4.0

    def next_token(self, prefix):
        x = self.logits(prefix)
        return int(np.flatnonzero(x == x.max())[0])


def test_ngram_backoff_verify_loop_equals_plain_decode():
    lanes, vocab, draft_k, n_out = 6, 64, 4, 120
    lms = [TrigramLM(vocab, 100 + b) for b in range(lanes)]
    rng = np.random.default_rng(4)
    prompts = [[int(x) for x in rng.integers(0, vocab, 12)] for _ in range(lanes)]
    plain = []
    for b in range(lanes):
        seq = list(prompts[b])
        for _ in range(n_out + 2 * draft_k):
            seq.append(lms[b].next_token(seq))
        plain.append(seq[len(prompts[b]):])

    hist = [list(p) for p in prompts]          # committed tokens, prompt included
    counts = sv.new_accept_counts(1, DEV)
    states = sv.new_backoff_states(lanes, DEV)
    allowed = torch.full((lanes,), draft_k, dtype=torch.int32, device=DEV)
    orc_counts, orc_states = om.AcceptCounts(), [ob.BackoffState() for _ in range(lanes)]
    orc_allowed = [draft_k] * lanes
    rounds = 0
    while min(len(h) - len(p) for h, p in zip(hist, prompts)) < n_out:
        rounds += 1
        # drafts from each lane's history, capped by the back-off
        flat = torch.tensor([t for h in hist for t in h], dtype=torch.int32, device=DEV)
        offs = torch.tensor(np.cumsum([0] + [len(h) for h in hist]), dtype=torch.int64, device=DEV)
        drafts = torch.full((lanes, draft_k), -1, dtype=torch.int32, device=DEV)
        dlens = torch.empty(lanes, dtype=torch.int32, device=DEV)
        sv.spec_ngram_draft(flat, offs, draft_k, drafts, dlens, match_min=1, match_max=4)
        d_host, l_host = drafts.cpu().numpy(), dlens.cpu().numpy()
        a_host = allowed.cpu().numpy()
        assert a_host.tolist() == orc_allowed
        ks = []
        for b in range(lanes):
            want = ong.ngram_draft(hist[b], draft_k, 1, 4)[0]
            assert l_host[b] == len(want) and d_host[b, :len(want)].tolist() == want
            ks.append(int(min(l_host[b], a_host[b])))
        # the model scores the anchor and the drafts of every lane
        rows, dt, offs_r = [], [], [0]
        for b in range(lanes):
            cols = [hist[b][-1]] + d_host[b, :ks[b]].tolist()
            for j in range(ks[b] + 1):
                rows.append(lms[b].logits(hist[b] + cols[1:j + 1]))
            dt += d_host[b, :ks[b]].tolist() + [-1]
            offs_r.append(offs_r[-1] + ks[b] + 1)
        k_t = torch.tensor(ks, dtype=torch.int32, device=DEV)
        r = workloads.RoundInputs("loop", vocab, lanes, offs_r[-1], "f32",
                                  torch.tensor(np.stack(rows), dtype=torch.float32, device=DEV), None,
                                  torch.tensor(dt, dtype=torch.int32, device=DEV), k_t,
                                  torch.tensor(offs_r, dtype=torch.int32, device=DEV),
                                  torch.zeros(lanes, dtype=torch.float32, device=DEV), rounds)
        committed = torch.empty(lanes, dtype=torch.int32, device=DEV)
        out = torch.empty(r.rows, dtype=torch.int32, device=DEV)
        status = torch.empty(lanes, dtype=torch.int32, device=DEV)
        sv.spec_verify_accept(r.target, None, r.draft_tokens, r.draft_lens, r.row_offsets, r.temperatures,
                              r.seed, committed, out, status)
        sv.spec_accept_counts_update(committed, k_t, status, counts)
        sv.spec_backoff_step(states, k_t, committed, status, draft_k, allowed)
        c_host, o_host, s_host = committed.cpu().numpy(), out.cpu().numpy(), status.cpu().numpy()
        assert (s_host == 0).all()
        for b in range(lanes):
            hist[b] += o_host[offs_r[b]:offs_r[b] + c_host[b]].tolist()
        om.count_verify_outputs(orc_counts, c_host, ks, s_host)
        ob.step(orc_states, ks, [int(c) - 1 for c in c_host])
        orc_allowed = ob.next_draft_lens(orc_states, draft_k)

    for b in range(lanes):
        out_b = hist[b][len(prompts[b]):]
        seq = prompts[b] + plain[b]
        while len(seq) < len(hist[b]):  # lanes run on until the slowest has n_out tokens
            seq.append(lms[b].next_token(seq))
        assert len(out_b) >= n_out and out_b == seq[len(prompts[b]):len(hist[b])], b
    torch.cuda.synchronize()
    c = counts[0].tolist()
    assert c == [orc_counts.rounds, orc_counts.proposed, orc_counts.accepted] + orc_counts.slot_reached + \
        orc_counts.slot_kept
    assert states[:, :3].cpu().tolist() == [[s.misses, s.backoff, s.wait] for s in orc_states]
    # the drafter's copies paid: more than one token a round on average
    assert orc_counts.accepted > 0 and (orc_counts.rounds + orc_counts.accepted) / orc_counts.rounds > 1.5
