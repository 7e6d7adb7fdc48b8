"""The plain C++ statement of the oracle (``oracle/verify_ref.cpp``), built with
g++ and called through ctypes.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  The C++ file is a
second, independent statement of the same definitions as ``oracle/verify.py``:
both are pinned by the same page facts in ``tests/``, and they must agree with
each other.  Being compiled and threaded over lanes, this one is also what
``bench.py`` times as the CPU baseline on the host's cores.

``build()`` compiles ``liboracle_ref.so`` next to this file (plain ``g++``, no
CUDA); ``verify_round`` returns the same ``RoundResult`` as the numpy oracle.
"""

import ctypes
import os
import shutil
import subprocess

import numpy as np

from .verify import RoundResult

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "verify_ref.cpp")
LIB_PATH = os.path.join(HERE, "liboracle_ref.so")

# No -march=native and no fused multiply-adds: the same results on every host.
CXX_FLAGS = ["-O2", "-std=c++17", "-shared", "-fPIC", "-pthread", "-ffp-contract=off"]

_libs = {}


def build(force=False, mutate=0, out_path=None):
    """Compile the C++ oracle; ``mutate`` > 0 plants one of the test-only
    mistakes (OREF_MUTATE) into a separate library.  Returns the library path."""
    path = out_path or (LIB_PATH if not mutate else os.path.join(HERE, f"liboracle_ref_m{mutate}.so"))
    if not force and os.path.exists(path) and os.path.getmtime(path) >= os.path.getmtime(SOURCE):
        return path
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        raise RuntimeError("g++ not found: the C++ oracle needs a host C++ compiler")
    tmp = f"{path}.{os.getpid()}.tmp"
    cmd = [cxx, *CXX_FLAGS, f"-DOREF_MUTATE={int(mutate)}", "-o", tmp, SOURCE]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("building the C++ oracle failed:\n" + " ".join(cmd) + "\n" + res.stdout + res.stderr)
    os.replace(tmp, path)
    return path


def load(mutate=0, path=None):
    key = path or mutate
    if key in _libs:
        return _libs[key]
    lib = ctypes.CDLL(path or build(mutate=mutate))
    P = ctypes.c_void_p
    lib.oref_row_budget.restype = ctypes.c_int32
    lib.oref_row_budget.argtypes = [ctypes.c_int32] * 3
    lib.oref_philox4x64_10.restype = None
    lib.oref_philox4x64_10.argtypes = [P, P, P]
    lib.oref_round_uniforms.restype = None
    lib.oref_round_uniforms.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64, P]
    lib.oref_verify_round.restype = ctypes.c_int32
    lib.oref_verify_round.argtypes = ([P, P, ctypes.c_int32, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                       P, P, P, P, ctypes.c_int32, ctypes.c_uint64, ctypes.c_uint64,
                                       P, P, ctypes.c_int32, ctypes.c_int32] + [P] * 12)
    lib.oref_commit_state.restype = None
    lib.oref_commit_state.argtypes = [P, P, P, P, ctypes.c_int32, ctypes.c_int32, ctypes.c_uint64]
    _libs[key] = lib
    return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def row_budget(draft_tokens, rows, lanes, lib=None):
    r = (lib or load()).oref_row_budget(int(draft_tokens), int(rows), int(lanes))
    if r < 0:
        raise ValueError("row_budget: lanes must be > 0 and the others >= 0")
    return int(r)


def philox4x64_10(counter, key, lib=None):
    mask = (1 << 64) - 1
    c = np.array([int(w) & mask for w in counter], np.uint64)
    k = np.array([int(w) & mask for w in key], np.uint64)
    out = np.zeros(4, np.uint64)
    (lib or load()).oref_philox4x64_10(_ptr(c), _ptr(k), _ptr(out))
    return tuple(int(w) for w in out)


def round_uniforms(seed, lane, position, lib=None):
    out = np.zeros(2, np.float64)
    mask = (1 << 64) - 1
    (lib or load()).oref_round_uniforms(int(seed) & mask, int(lane) & mask, int(position) & mask, _ptr(out))
    return float(out[0]), float(out[1])


def _logits(a):
    """(array, dtype code, ld) of a logits array: float64 / float32 values or bf16 bit patterns (uint16)."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        code = 1
    elif a.dtype == np.float32:
        code = 0
    else:
        a, code = a.astype(np.float64, copy=False), 2
    if a.ndim != 2:
        raise ValueError("logits must be 2-D [rows, V]")
    if a.strides[1] != a.itemsize or a.strides[0] % a.itemsize:
        a = np.ascontiguousarray(a)
    return a, code, a.strides[0] // a.itemsize


def verify_round(target, draft, draft_tokens, draft_lens, row_offsets, temperatures, seed=0, u_acc=None,
                 u_smp=None, lane_base=0, threads=1, lib=None, return_threads=False):
    """The round, as ``oracle.verify_round``: same arguments and result.  The
    logits may also be given as bfloat16 bit patterns (uint16) or float32,
    which the C++ code widens exactly.  ``threads`` workers (0: one per host
    thread) take lanes one at a time."""
    lib = lib or load()
    t, code, ld = _logits(target)
    rows, vocab = t.shape
    d = None
    if draft is not None:
        d, dcode, dld = _logits(draft)
        if dcode != code or dld != ld:
            if code == 1 or dcode == 1:
                raise ValueError("target and draft must have the same dtype and row stride")
            t, d = np.ascontiguousarray(t, np.float64), np.ascontiguousarray(d, np.float64)
            code, ld = 2, vocab
    lens = np.ascontiguousarray(draft_lens, np.int32)
    lanes = lens.shape[0]
    tok = np.ascontiguousarray(draft_tokens, np.int32)
    off = np.ascontiguousarray(row_offsets, np.int32)
    temps = np.ascontiguousarray(temperatures, np.float32)
    ua = us = None
    stride = 0
    if u_acc is not None or u_smp is not None:
        stride = max(len(u) for u in (u_acc if u_acc is not None else u_smp))

        def table(u):
            if u is None:
                return None
            out = np.zeros((lanes, stride), np.float64)
            for b, row in enumerate(u):
                out[b, :len(row)] = row
            return out
        ua, us = table(u_acc), table(u_smp)
    res = RoundResult(
        committed=np.zeros(lanes, np.int32), out_tokens=np.full(rows, -1, np.int32),
        lane_status=np.zeros(lanes, np.int32), argmax=np.full(rows, -1, np.int64),
        max_logit=np.full(rows, np.nan), lse=np.full(rows, np.nan), logp_d=np.full(rows, np.nan),
        logq_d=np.full(rows, np.nan), resid_mass=np.full(rows, np.nan), margins=[[] for _ in range(lanes)])
    accept_margin = np.full(rows, np.nan)
    draw_margin = np.full(lanes, np.nan)
    draw_pos = np.full(lanes, -1, np.int32)
    used = lib.oref_verify_round(
        _ptr(t), _ptr(d), code, ld, rows, vocab, _ptr(tok), _ptr(lens), _ptr(off), _ptr(temps), lanes,
        int(seed) & ((1 << 64) - 1), int(lane_base), _ptr(ua), _ptr(us), stride, int(threads),
        _ptr(res.committed), _ptr(res.out_tokens), _ptr(res.lane_status), _ptr(res.argmax), _ptr(res.max_logit),
        _ptr(res.lse), _ptr(res.logp_d), _ptr(res.logq_d), _ptr(res.resid_mass), _ptr(accept_margin),
        _ptr(draw_margin), _ptr(draw_pos))
    for b in range(lanes):
        if draw_pos[b] < 0:
            continue
        base = int(off[b])
        res.margins[b] = [("accept", j, float(accept_margin[base + j])) for j in range(int(lens[b]))
                          if np.isfinite(accept_margin[base + j]) or accept_margin[base + j] == np.inf]
        res.margins[b].append(("draw", int(draw_pos[b]), float(draw_margin[b])))
    return (res, int(used)) if return_threads else res


def commit_state(staged, live, committed, lane_status=None, lib=None):
    """As ``oracle.commit_state``: staged [lanes, cols, ...], live [lanes, ...]
    byte-compatible arrays; returns the new live state."""
    staged = np.ascontiguousarray(staged)
    out = np.array(live, copy=True, order="C")
    lanes, cols = staged.shape[0], staged.shape[1]
    per = out[0].nbytes if lanes else 0
    c = np.ascontiguousarray(committed, np.int32)
    st = None if lane_status is None else np.ascontiguousarray(lane_status, np.int32)
    (lib or load()).oref_commit_state(_ptr(staged), _ptr(out), _ptr(c), _ptr(st), lanes, cols, per)
    return out
