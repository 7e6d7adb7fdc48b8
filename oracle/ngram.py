"""Copy-from-the-conversation (n-gram / prompt-lookup) drafter.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Follows mashbox docs, "Speculative decoding", section "Options"
(--speculation ngram: the drafter looks up the last few tokens earlier in the
request and proposes the tokens that followed them there; --draft-k: 1 to 8
guesses a pass, 3 by default).  Read as:

* a lane's history h[0..L) ends with the anchor h[L-1];
* for a match length m, the suffix is h[L-m..L); an earlier occurrence is an
  end position i < L with h[i-m..i) == h[L-m..L);
* the drafter uses the longest m in [match_min, match_max] (and m < L) that has
  an earlier occurrence, and of those occurrences the most recent (largest i);
* it proposes h[i..min(i + k, L)), the tokens that followed the occurrence;
  no occurrence of any allowed length proposes nothing.

Plain Python loops.
"""


def ngram_draft(history, k, match_min=1, match_max=4):
    """Drafts for one lane: (tokens, match_length, end_position); ([], 0, -1) if none."""
    h = list(history)
    L = len(h)
    if k <= 0 or L < 2:
        return [], 0, -1
    for m in range(min(match_max, L - 1), match_min - 1, -1):
        suffix = h[L - m:]
        for i in range(L - 1, m - 1, -1):  # most recent first
            if h[i - m:i] == suffix:
                return h[i:min(i + k, L)], m, i
    return [], 0, -1


def ngram_draft_batch(histories, k, match_min=1, match_max=4):
    """Drafts of every lane: (list of token lists, list of lengths)."""
    drafts = [ngram_draft(h, k, match_min, match_max)[0] for h in histories]
    return drafts, [len(d) for d in drafts]
