"""Python binding of libspecverify, the GB300 verify-round library.

Argument marshalling only: every step of the verify round runs in the CUDA
kernels behind the C ABI of ``include/spec_verify.h``.  Tensors must already be
on the GPU; PyTorch provides device memory and the current stream.  If the
shared library has not been built every entry point raises -- there is no CPU
fallback.
"""

import ctypes
import os

import torch

from .build import LIB_PATH, build_library

__all__ = [
    "SPEC_OK", "SPEC_ERR_INVALID_ARG", "SPEC_ERR_UNSUPPORTED", "SPEC_ERR_CUDA",
    "SPEC_ERR_NONFINITE", "SPEC_ERR_TOKEN_RANGE", "SPEC_ERR_LAYOUT", "SPEC_ERR_TIMEOUT",
    "SPEC_MAX_DRAFTS", "SpecError", "ROW_STATS_FIELDS", "load_library", "build_library",
    "spec_row_budget", "spec_verify_accept", "spec_commit_state", "spec_status_string",
    "spec_verify_launch_shape", "spec_round_uniforms", "new_row_stats", "row_stats_view",
    "spec_accept_counts_update", "spec_accept_rates_from_counts", "new_accept_counts", "accept_counts_view",
    "spec_backoff_step", "new_backoff_states", "BACKOFF_FIELDS", "ACCEPT_COUNT_WORDS",
    "spec_ngram_draft", "SPEC_NGRAM_MAX_MATCH", "spec_apply_penalties", "SPEC_VERIFY_META_BEFORE_WAIT",
    "SPEC_VERIFY_TEST_WITHHOLD_COPY",
]

SPEC_OK = 0
SPEC_ERR_INVALID_ARG = 1
SPEC_ERR_UNSUPPORTED = 2
SPEC_ERR_CUDA = 3
SPEC_ERR_NONFINITE = 4
SPEC_ERR_TOKEN_RANGE = 5
SPEC_ERR_LAYOUT = 6
SPEC_ERR_TIMEOUT = 7
SPEC_MAX_DRAFTS = 15
SPEC_VERIFY_META_BEFORE_WAIT = 1
SPEC_VERIFY_TEST_WITHHOLD_COPY = 2

_DTYPES = {torch.float32: 0, torch.bfloat16: 1}

# spec_row_stats: 8 x 32-bit words per row.
ROW_STATS_FIELDS = ("argmax", "max_logit", "lse", "logp_d", "logq_d", "resid_mass", "drawn", "flags")
_ROW_STATS_INT = {"argmax", "drawn", "flags"}


class SpecError(RuntimeError):
    """A non-zero status returned by the library."""

    def __init__(self, code, what):
        self.code = code
        super().__init__(f"{what}: {spec_status_string(code)} ({code})")


class _Args(ctypes.Structure):
    _fields_ = [
        ("target_logits", ctypes.c_void_p),
        ("draft_logits", ctypes.c_void_p),
        ("dtype", ctypes.c_int),
        ("ld", ctypes.c_int64),
        ("V", ctypes.c_int32),
        ("lanes", ctypes.c_int32),
        ("rows", ctypes.c_int32),
        ("draft_tokens", ctypes.c_void_p),
        ("draft_lens", ctypes.c_void_p),
        ("row_offsets", ctypes.c_void_p),
        ("temperatures", ctypes.c_void_p),
        ("seed", ctypes.c_uint64),
        ("committed", ctypes.c_void_p),
        ("out_tokens", ctypes.c_void_p),
        ("lane_status", ctypes.c_void_p),
        ("row_stats", ctypes.c_void_p),
        ("lane_base", ctypes.c_uint32),
        ("flags", ctypes.c_uint32),
    ]


_lib = None


class _AcceptCounts(ctypes.Structure):
    _fields_ = [("rounds", ctypes.c_uint64), ("proposed", ctypes.c_uint64), ("accepted", ctypes.c_uint64),
                ("slot_reached", ctypes.c_uint64 * SPEC_MAX_DRAFTS), ("slot_kept", ctypes.c_uint64 * SPEC_MAX_DRAFTS)]


class _AcceptRates(ctypes.Structure):
    _fields_ = [("accepted_per_proposed", ctypes.c_double), ("tokens_per_round", ctypes.c_double),
                ("by_slot", ctypes.c_double * SPEC_MAX_DRAFTS), ("given_previous", ctypes.c_double * SPEC_MAX_DRAFTS),
                ("depth", ctypes.c_int32), ("reserved", ctypes.c_int32), ("implied_alpha", ctypes.c_double)]


ACCEPT_COUNT_WORDS = 3 + 2 * SPEC_MAX_DRAFTS
BACKOFF_FIELDS = ("misses", "backoff", "wait", "reserved")


def load_library():
    """Load libspecverify.so (built in-tree); raise if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is not built; call speculative_decoding_verify_bf16_gb300."
                           "build_library() (needs nvcc) -- there is no CPU fallback")
    lib = ctypes.CDLL(LIB_PATH)
    lib.spec_row_budget.restype = ctypes.c_int32
    lib.spec_row_budget.argtypes = [ctypes.c_int32] * 3
    lib.spec_verify_accept.restype = ctypes.c_int
    lib.spec_verify_accept.argtypes = [ctypes.POINTER(_Args), ctypes.c_void_p]
    lib.spec_commit_state.restype = ctypes.c_int
    lib.spec_commit_state.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                      ctypes.c_int32, ctypes.c_int32, ctypes.c_uint64,
                                      ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                      ctypes.c_void_p, ctypes.c_void_p]
    lib.spec_status_string.restype = ctypes.c_char_p
    lib.spec_status_string.argtypes = [ctypes.c_int]
    lib.spec_round_uniforms.restype = ctypes.c_int
    lib.spec_round_uniforms.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int32, ctypes.c_int32,
                                        ctypes.c_void_p, ctypes.c_void_p]
    lib.spec_verify_launch_shape.restype = ctypes.c_int
    lib.spec_verify_launch_shape.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int,
                                             ctypes.c_int32] + [ctypes.POINTER(ctypes.c_int32)] * 4
    lib.spec_accept_counts_update.restype = ctypes.c_int
    lib.spec_accept_counts_update.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                              ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p]
    lib.spec_accept_rates_from_counts.restype = ctypes.c_int
    lib.spec_accept_rates_from_counts.argtypes = [ctypes.POINTER(_AcceptCounts), ctypes.POINTER(_AcceptRates)]
    lib.spec_backoff_init.restype = ctypes.c_int
    lib.spec_backoff_init.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p]
    lib.spec_ngram_draft.restype = ctypes.c_int
    lib.spec_ngram_draft.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                     ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]
    lib.spec_apply_penalties.restype = ctypes.c_int
    lib.spec_apply_penalties.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32] + \
        [ctypes.c_void_p] * 10
    lib.spec_backoff_step.restype = ctypes.c_int
    lib.spec_backoff_step.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                      ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]
    _lib = lib
    return lib


def spec_status_string(code):
    return load_library().spec_status_string(int(code)).decode()


def spec_row_budget(draft_tokens, row_budget, lanes):
    """Drafts per lane under a row budget; raises ValueError on bad arguments."""
    r = load_library().spec_row_budget(int(draft_tokens), int(row_budget), int(lanes))
    if r < 0:
        raise ValueError(f"spec_row_budget({draft_tokens}, {row_budget}, {lanes}): "
                         f"{spec_status_string(-r)}")
    return int(r)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t, name, dtype, device, numel=None):
    if not isinstance(t, torch.Tensor) or t.device != device:
        raise ValueError(f"{name} must be a tensor on {device}")
    if t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {dtype} tensor")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{name} needs at least {numel} elements")


def new_row_stats(rows, device):
    """An int32 [rows, 8] buffer laid out as spec_row_stats."""
    return torch.empty(rows, 8, dtype=torch.int32, device=device)


def row_stats_view(buf):
    """Dict of named columns of a row-stats buffer (float fields viewed as float32)."""
    out = {}
    for i, name in enumerate(ROW_STATS_FIELDS):
        col = buf[:, i].contiguous()
        out[name] = col if name in _ROW_STATS_INT else col.view(torch.float32)
    return out


def spec_verify_accept(target, draft, draft_tokens, draft_lens, row_offsets, temperatures, seed,
                       committed, out_tokens, lane_status=None, row_stats=None, stream=None,
                       rows=None, lane_base=0, meta_before_wait=False, test_flags=0):
    """Launch the fused verify kernel (see spec_verify_accept in include/spec_verify.h).

    target, draft: [rows, >= V] bf16 or float32 CUDA tensors with unit inner
    stride (draft may be None when no lane samples); the row stride is taken as
    ld.  draft_tokens, out_tokens: int32 [rows]; draft_lens, committed,
    lane_status: int32 [lanes]; row_offsets: int32 [lanes + 1]; temperatures:
    float32 [lanes]; row_stats: int32 [rows, 8] from new_row_stats().
    ``rows`` defaults to target.shape[0] (it must equal row_offsets[-1]).
    ``lane_base`` is the global index of lane 0 in the Philox counter (a batch
    split into parts draws the uniforms of the unsplit batch).
    ``meta_before_wait`` sets SPEC_VERIFY_META_BEFORE_WAIT: the caller promises
    that the kernel preceding this launch on the stream did not write
    draft_tokens, draft_lens, row_offsets or temperatures.  ``test_flags`` adds
    test-only flags (SPEC_VERIFY_TEST_WITHHOLD_COPY).
    """
    lib = load_library()
    if target.dim() != 2 or target.stride(1) != 1 or target.dtype not in _DTYPES:
        raise ValueError("target must be a 2-D bf16/float32 tensor with unit inner stride")
    dev = target.device
    if dev.type != "cuda":
        raise ValueError("target must be on a CUDA device")
    if draft is not None and (draft.dtype != target.dtype or draft.device != dev or draft.dim() != 2
                              or draft.stride(1) != 1 or draft.stride(0) != target.stride(0)):
        raise ValueError("draft must match target's dtype, device and row stride")
    lanes = draft_lens.numel()
    nrows = target.shape[0] if rows is None else int(rows)
    if nrows > target.shape[0] or (draft is not None and nrows > draft.shape[0]):
        raise ValueError("rows exceeds the rows of the logits tensors")
    _need(draft_tokens, "draft_tokens", torch.int32, dev, nrows)
    _need(draft_lens, "draft_lens", torch.int32, dev)
    _need(row_offsets, "row_offsets", torch.int32, dev, lanes + 1)
    _need(temperatures, "temperatures", torch.float32, dev, lanes)
    _need(committed, "committed", torch.int32, dev, lanes)
    _need(out_tokens, "out_tokens", torch.int32, dev, nrows)
    if lane_status is not None:
        _need(lane_status, "lane_status", torch.int32, dev, lanes)
    if row_stats is not None:
        _need(row_stats, "row_stats", torch.int32, dev, nrows * 8)
    a = _Args(
        target_logits=target.data_ptr(),
        draft_logits=None if draft is None else draft.data_ptr(),
        dtype=_DTYPES[target.dtype],
        ld=target.stride(0),
        V=target.shape[1],
        lanes=lanes,
        rows=nrows,
        draft_tokens=draft_tokens.data_ptr(),
        draft_lens=draft_lens.data_ptr(),
        row_offsets=row_offsets.data_ptr(),
        temperatures=temperatures.data_ptr(),
        seed=int(seed) & ((1 << 64) - 1),
        committed=committed.data_ptr(),
        out_tokens=out_tokens.data_ptr(),
        lane_status=None if lane_status is None else lane_status.data_ptr(),
        row_stats=None if row_stats is None else row_stats.data_ptr(),
        lane_base=int(lane_base),
        flags=(SPEC_VERIFY_META_BEFORE_WAIT if meta_before_wait else 0) | int(test_flags),
    )
    code = lib.spec_verify_accept(ctypes.byref(a), _stream(stream))
    if code != SPEC_OK:
        raise SpecError(code, "spec_verify_accept")


def spec_verify_accept_raw(args, stream):
    """Call spec_verify_accept with a prepared _Args (no checks); returns the status."""
    return load_library().spec_verify_accept(ctypes.byref(args), stream)


def make_args(target, draft, draft_tokens, draft_lens, row_offsets, temperatures, seed,
              committed, out_tokens, lane_status=None, row_stats=None, V=None, rows=None, lane_base=0,
              meta_before_wait=False):
    """Build the C argument struct once (for tight loops that call it repeatedly)."""
    return _Args(
        target_logits=target.data_ptr(),
        draft_logits=None if draft is None else draft.data_ptr(),
        dtype=_DTYPES[target.dtype],
        ld=target.stride(0),
        V=target.shape[1] if V is None else int(V),
        lanes=draft_lens.numel(),
        rows=target.shape[0] if rows is None else int(rows),
        draft_tokens=draft_tokens.data_ptr(),
        draft_lens=draft_lens.data_ptr(),
        row_offsets=row_offsets.data_ptr(),
        temperatures=temperatures.data_ptr(),
        seed=int(seed) & ((1 << 64) - 1),
        committed=committed.data_ptr(),
        out_tokens=out_tokens.data_ptr(),
        lane_status=None if lane_status is None else lane_status.data_ptr(),
        row_stats=None if row_stats is None else row_stats.data_ptr(),
        lane_base=int(lane_base),
        flags=SPEC_VERIFY_META_BEFORE_WAIT if meta_before_wait else 0,
    )


def spec_commit_state(staged, live, committed, lane_status=None, stream=None):
    """Copy staged[b, committed[b] - 1] into live[b] for every lane (on the GPU).

    staged: [lanes, cols, ...] and live: [lanes, ...] CUDA tensors of one dtype
    whose per-column snapshot is contiguous.
    """
    lib = load_library()
    lanes, cols = staged.shape[0], staged.shape[1]
    dev = staged.device
    if live.device != dev or live.dtype != staged.dtype or live.shape[0] != lanes:
        raise ValueError("live must match staged's device, dtype and lane count")
    if not staged[0, 0].is_contiguous() or not live[0].is_contiguous():
        raise ValueError("each snapshot must be contiguous")
    esize = staged.element_size()
    bytes_per_col = live[0].numel() * esize
    if staged[0, 0].numel() * esize != bytes_per_col:
        raise ValueError("staged and live snapshots differ in size")
    _need(committed, "committed", torch.int32, dev, lanes)
    if lane_status is not None:
        _need(lane_status, "lane_status", torch.int32, dev, lanes)
    code = lib.spec_commit_state(
        _ptr(staged), _ptr(live), _ptr(committed), lanes, cols, bytes_per_col,
        staged.stride(0) * esize, staged.stride(1) * esize, live.stride(0) * esize,
        _ptr(lane_status), _stream(stream))
    if code != SPEC_OK:
        raise SpecError(code, "spec_commit_state")


def spec_round_uniforms(seed, lanes, positions, lane_base=0, device=None, stream=None):
    """float32 [lanes, positions, 2]: the (u, u') pairs the verify kernel draws."""
    lib = load_library()
    device = device or torch.device("cuda", torch.cuda.current_device())
    out = torch.empty(lanes, positions, 2, dtype=torch.float32, device=device)
    code = lib.spec_round_uniforms(int(seed) & ((1 << 64) - 1), int(lane_base), int(lanes), int(positions),
                                   _ptr(out), _stream(stream))
    if code != SPEC_OK:
        raise SpecError(code, "spec_round_uniforms")
    return out


def spec_verify_launch_shape(lanes, rows, V, dtype=torch.bfloat16, with_draft=False):
    """Launch shape spec_verify_accept would pick (see include/spec_verify.h)."""
    lib = load_library()
    vals = [ctypes.c_int32() for _ in range(4)]
    code = lib.spec_verify_launch_shape(int(lanes), int(rows), int(V), _DTYPES[dtype], int(bool(with_draft)),
                                        *[ctypes.byref(v) for v in vals])
    if code != SPEC_OK:
        raise SpecError(code, "spec_verify_launch_shape")
    return dict(zip(("cluster_ctas", "threads", "slice", "smem_bytes"), (v.value for v in vals)))


# ---------------------------------------------------------------------------
# Acceptance metrics and miss back-off (include/spec_round_control.h)
# ---------------------------------------------------------------------------
def new_accept_counts(n, device):
    """Zeroed int64 [n, 33] buffer laid out as n spec_accept_counts."""
    return torch.zeros(n, ACCEPT_COUNT_WORDS, dtype=torch.int64, device=device)


def accept_counts_view(row):
    """Dict of one spec_accept_counts row (any int64 tensor or sequence of 33 words)."""
    w = [int(x) for x in (row.tolist() if isinstance(row, torch.Tensor) else row)]
    k = SPEC_MAX_DRAFTS
    return {"rounds": w[0], "proposed": w[1], "accepted": w[2],
            "slot_reached": w[3:3 + k], "slot_kept": w[3 + k:3 + 2 * k]}


def spec_accept_counts_update(committed, draft_lens, lane_status, counts, per_lane=False, stream=None):
    """Add one verify round's outputs to device counts (new_accept_counts(1) for the
    batch, new_accept_counts(lanes) with per_lane=True)."""
    lib = load_library()
    dev = committed.device
    lanes = committed.numel()
    _need(committed, "committed", torch.int32, dev)
    _need(draft_lens, "draft_lens", torch.int32, dev, lanes)
    if lane_status is not None:
        _need(lane_status, "lane_status", torch.int32, dev, lanes)
    _need(counts, "counts", torch.int64, dev, (lanes if per_lane else 1) * ACCEPT_COUNT_WORDS)
    rc = lib.spec_accept_counts_update(_ptr(committed), _ptr(draft_lens), _ptr(lane_status), lanes,
                                       _ptr(counts), 1 if per_lane else 0, _stream(stream))
    if rc != SPEC_OK:
        raise SpecError(rc, "spec_accept_counts_update")


def spec_accept_rates_from_counts(counts_row):
    """The page's rates from one set of counts (host call)."""
    c = accept_counts_view(counts_row)
    cs = _AcceptCounts(c["rounds"], c["proposed"], c["accepted"],
                       (ctypes.c_uint64 * SPEC_MAX_DRAFTS)(*c["slot_reached"]),
                       (ctypes.c_uint64 * SPEC_MAX_DRAFTS)(*c["slot_kept"]))
    r = _AcceptRates()
    rc = load_library().spec_accept_rates_from_counts(ctypes.byref(cs), ctypes.byref(r))
    if rc != SPEC_OK:
        raise SpecError(rc, "spec_accept_rates_from_counts")
    return {"accepted_per_proposed": r.accepted_per_proposed, "tokens_per_round": r.tokens_per_round,
            "by_slot": list(r.by_slot), "given_previous": list(r.given_previous), "depth": r.depth,
            "implied_alpha": r.implied_alpha}


def new_backoff_states(lanes, device, stream=None):
    """int32 [lanes, 4] back-off states, initialised on the device."""
    st = torch.empty(lanes, 4, dtype=torch.int32, device=device)
    rc = load_library().spec_backoff_init(_ptr(st), lanes, _stream(stream))
    if rc != SPEC_OK:
        raise SpecError(rc, "spec_backoff_init")
    return st


def spec_backoff_step(states, proposed, committed, lane_status, draft_tokens, next_draft_lens, stream=None):
    """Advance the back-off of every lane by one verify round; writes the next
    round's draft lengths."""
    lib = load_library()
    dev = states.device
    lanes = proposed.numel()
    _need(states, "states", torch.int32, dev, lanes * 4)
    _need(proposed, "proposed", torch.int32, dev)
    _need(committed, "committed", torch.int32, dev, lanes)
    if lane_status is not None:
        _need(lane_status, "lane_status", torch.int32, dev, lanes)
    _need(next_draft_lens, "next_draft_lens", torch.int32, dev, lanes)
    rc = lib.spec_backoff_step(_ptr(states), _ptr(proposed), _ptr(committed), _ptr(lane_status), lanes,
                               int(draft_tokens), _ptr(next_draft_lens), _stream(stream))
    if rc != SPEC_OK:
        raise SpecError(rc, "spec_backoff_step")


SPEC_NGRAM_MAX_MATCH = 16


def spec_ngram_draft(tokens, hist_offsets, k, drafts, draft_lens, match_min=1, match_max=4, stream=None):
    """Copy-from-the-conversation drafts for every lane: tokens int32 [total],
    hist_offsets int64 [lanes + 1], drafts int32 [lanes, >= k] (row stride taken
    as the draft stride), draft_lens int32 [lanes]."""
    lib = load_library()
    dev = tokens.device
    lanes = hist_offsets.numel() - 1
    _need(tokens, "tokens", torch.int32, dev)
    _need(hist_offsets, "hist_offsets", torch.int64, dev, lanes + 1)
    _need(draft_lens, "draft_lens", torch.int32, dev, lanes)
    if drafts.dim() != 2 or drafts.dtype != torch.int32 or drafts.device != dev or drafts.stride(1) != 1 \
            or drafts.shape[0] < lanes:
        raise ValueError("drafts must be an int32 [lanes, >= k] tensor with unit inner stride")
    rc = lib.spec_ngram_draft(_ptr(tokens), _ptr(hist_offsets), lanes, int(k), int(match_min), int(match_max),
                              _ptr(drafts), drafts.stride(0), _ptr(draft_lens), _stream(stream))
    if rc != SPEC_OK:
        raise SpecError(rc, "spec_ngram_draft")


def spec_apply_penalties(target, row_offsets, draft_tokens, draft_lens, pen_tokens, pen_counts, pen_offsets,
                         presence=None, frequency=None, lane_status=None, stream=None):
    """Per-row presence / frequency penalties on the target logits (see
    spec_apply_penalties in include/spec_round_control.h).  The logits in
    ``target`` are overwritten with the penalised values.  target: the round's
    [rows, >= V] bf16/float32 logits (V = target.shape[1], ld its row stride);
    pen_tokens / pen_counts int32 [n] (per lane ascending distinct ids, counts
    >= 1), pen_offsets int64 [lanes + 1]; presence / frequency float32 [lanes]
    or None; lane_status int32 [lanes] or None receives each lane's status (a
    lane whose list breaks the contract is left untouched)."""
    lib = load_library()
    if target.dim() != 2 or target.stride(1) != 1 or target.dtype not in _DTYPES:
        raise ValueError("target must be a 2-D bf16/float32 tensor with unit inner stride")
    dev = target.device
    lanes = draft_lens.numel()
    _need(row_offsets, "row_offsets", torch.int32, dev, lanes + 1)
    _need(draft_tokens, "draft_tokens", torch.int32, dev)
    _need(draft_lens, "draft_lens", torch.int32, dev)
    _need(pen_tokens, "pen_tokens", torch.int32, dev)
    _need(pen_counts, "pen_counts", torch.int32, dev, pen_tokens.numel())
    _need(pen_offsets, "pen_offsets", torch.int64, dev, lanes + 1)
    for t, name in ((presence, "presence"), (frequency, "frequency")):
        if t is not None:
            _need(t, name, torch.float32, dev, lanes)
    if lane_status is not None:
        _need(lane_status, "lane_status", torch.int32, dev, lanes)
    rc = lib.spec_apply_penalties(_ptr(target), _DTYPES[target.dtype], target.stride(0), target.shape[1], lanes,
                                  _ptr(row_offsets), _ptr(draft_tokens), _ptr(draft_lens), _ptr(pen_tokens),
                                  _ptr(pen_counts), _ptr(pen_offsets), _ptr(presence), _ptr(frequency),
                                  _ptr(lane_status), _stream(stream))
    if rc != SPEC_OK:
        raise SpecError(rc, "spec_apply_penalties")
