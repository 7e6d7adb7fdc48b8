"""CPU oracle of the speculative-decoding verify round.

TEST INFRASTRUCTURE ONLY.  A plain, slow, float64 restatement of what the
verify round computes, written from the pages that describe the method, used to
check the CUDA library.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import it.  It shares no code
with the CUDA library (no kernels, headers, helpers or constant tables) and
never calls it; the product path never calls this package.

``oracle.metrics`` counts the acceptance metrics of verify rounds,
``oracle.backoff`` is the per-lane miss back-off of a drafter,
``oracle.ngram`` the copy-from-the-conversation drafter and
``oracle.penalties`` the per-row presence / frequency penalties; all are plain
Python restatements of the pages' rules.

Every function is pinned by ``-m "not gpu"`` tests against facts fixed outside
the oracle itself: the pages' worked examples, exact enumeration of the
acceptance rule on tiny vocabularies, a closed form, library routines (numpy's
Philox4x64, scipy's softmax / logsumexp) and invariants.
"""

from . import backoff, metrics, ngram, penalties
from .philox import philox4x64_10, round_uniforms, word_to_uniform
from .verify import (
    DEFAULT_ROW_BUDGET,
    STATUS_CUDA,
    STATUS_INVALID_ARG,
    STATUS_LAYOUT,
    STATUS_NONFINITE,
    STATUS_OK,
    STATUS_TIMEOUT,
    STATUS_TOKEN_RANGE,
    STATUS_UNSUPPORTED,
    RoundResult,
    accept_draft,
    acceptance_ratio,
    argmax_lowest,
    commit_state,
    commit_status,
    decode_bf16,
    decode_logits,
    inverse_cdf,
    residual_weights,
    row_budget,
    row_is_valid,
    softmax_at_temperature,
    verify_round,
)
