"""The C-ABI library loads and exports what include/*.h declares (no GPU needed)."""

import ctypes
import glob
import os
import re
import subprocess

import pytest

from conftest import ROOT, read_golden

import speculative_decoding_verify_bf16_gb300 as sv


def _declared_functions():
    names = set()
    for path in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(path).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w \t\*]*?\b(spec_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    sv.build_library()
    return sv.load_library()


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for want in ["spec_row_budget", "spec_verify_accept", "spec_commit_state",
                 "spec_status_string", "spec_verify_launch_shape", "spec_round_uniforms"]:
        assert want in names, names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", sv.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for name in _declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)


def test_row_budget_worked_example_through_the_abi(lib):
    for draft_tokens, budget, lanes, expected in read_golden("row_budget_worked_example.txt"):
        assert sv.spec_row_budget(draft_tokens, budget, lanes) == expected


def test_row_budget_errors_through_the_abi(lib):
    for args in [(3, 8, 0), (3, 8, -2), (-1, 8, 1), (3, -1, 1)]:
        assert lib.spec_row_budget(*args) == -sv.SPEC_ERR_INVALID_ARG
        with pytest.raises(ValueError):
            sv.spec_row_budget(*args)
    assert sv.spec_row_budget(7, 1024, 128) == 7


def test_status_strings(lib):
    names = ["SPEC_OK", "SPEC_ERR_INVALID_ARG", "SPEC_ERR_UNSUPPORTED", "SPEC_ERR_CUDA",
             "SPEC_ERR_NONFINITE", "SPEC_ERR_TOKEN_RANGE", "SPEC_ERR_LAYOUT", "SPEC_ERR_TIMEOUT"]
    for code, name in enumerate(names):
        assert sv.spec_status_string(code) == name
    assert sv.spec_status_string(99) == "SPEC_ERR_UNKNOWN"


def test_calls_with_bad_arguments_fail_on_the_host(lib):
    # NULL argument struct and NULL out pointer: rejected before touching a GPU.
    assert lib.spec_verify_accept(None, None) == sv.SPEC_ERR_INVALID_ARG
    assert lib.spec_round_uniforms(1, 0, 4, 4, None, None) == sv.SPEC_ERR_INVALID_ARG
    assert lib.spec_commit_state(None, None, None, -1, 1, 16, 16, 16, 16, None, None) == \
        sv.SPEC_ERR_INVALID_ARG
    assert lib.spec_commit_state(None, None, None, 0, 1, 16, 16, 16, 16, None, None) == sv.SPEC_OK


def _c_layout(struct, fields, tmp_path):
    """sizeof and offsetof of `struct`'s `fields` from a C program built against the headers."""
    src = tmp_path / "layout.c"
    body = "".join(f'  printf("%zu\\n", offsetof({struct}, {f}));\n' for f in fields)
    src.write_text(f'#include <stddef.h>\n#include <stdio.h>\n#include "spec_round_control.h"\n'
                   f'int main(void) {{\n  printf("%zu\\n", sizeof({struct}));\n{body}  return 0;\n}}\n')
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True)
    vals = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    return vals[0], vals[1:]


@pytest.mark.parametrize("struct,cls", [("spec_verify_args", sv._Args),
                                        ("spec_accept_counts", sv._AcceptCounts),
                                        ("spec_accept_rates", sv._AcceptRates)])
def test_binding_structs_match_the_c_layout(struct, cls, tmp_path):
    """The ctypes structures the binding passes have the C structs' size and field offsets."""
    fields = [name for name, _ in cls._fields_]
    size, offsets = _c_layout(struct, fields, tmp_path)
    assert ctypes.sizeof(cls) == size
    assert [getattr(cls, f).offset for f in fields] == offsets


def test_binding_constants_match_the_header_defines():
    text = "".join(open(p).read() for p in glob.glob(os.path.join(ROOT, "include", "*.h")))
    defines = {m.group(1): int(m.group(2)) for m in re.finditer(r"#define\s+(SPEC_\w+)\s+(\d+)u?\b", text)}
    for name in ("SPEC_MAX_DRAFTS", "SPEC_VERIFY_META_BEFORE_WAIT", "SPEC_VERIFY_TEST_WITHHOLD_COPY",
                 "SPEC_NGRAM_MAX_MATCH"):
        assert getattr(sv, name) == defines[name], name


def test_verify_argument_checks_come_before_any_device_work(lib):
    """An empty batch, V <= 0, rows < lanes, ld < V, an unknown dtype or a NULL
    required pointer is rejected on the host, before any CUDA call (so this runs
    without a GPU; the pointers are never dereferenced)."""
    fake = 4096  # a non-NULL address the library must not touch

    def args(**kw):
        a = sv._Args(target_logits=fake, draft_logits=None, dtype=1, ld=64, V=64, lanes=2, rows=4,
                     draft_tokens=fake, draft_lens=fake, row_offsets=fake, temperatures=fake, seed=1,
                     committed=fake, out_tokens=fake, lane_status=None, row_stats=None, lane_base=0, flags=0)
        for k, v in kw.items():
            setattr(a, k, v)
        return a

    for kw in [dict(lanes=0), dict(lanes=-3), dict(V=0), dict(V=-1), dict(rows=1), dict(ld=63), dict(dtype=7),
               dict(target_logits=None), dict(draft_tokens=None), dict(draft_lens=None), dict(row_offsets=None),
               dict(temperatures=None), dict(committed=None), dict(out_tokens=None)]:
        assert lib.spec_verify_accept(ctypes.byref(args(**kw)), None) == sv.SPEC_ERR_INVALID_ARG, kw
    out = [ctypes.c_int32() for _ in range(4)]
    for bad in [(0, 4, 64, 1), (2, 1, 64, 1), (2, 4, 0, 1), (2, 4, 64, 9)]:
        assert lib.spec_verify_launch_shape(*bad, 0, *[ctypes.byref(o) for o in out]) == sv.SPEC_ERR_INVALID_ARG
    # an empty commit or uniform request is a no-op, not an error
    assert lib.spec_round_uniforms(1, 0, 0, 4, None, None) == sv.SPEC_OK
    assert lib.spec_commit_state(None, None, None, 0, 4, 16, 64, 16, 16, None, None) == sv.SPEC_OK
    assert lib.spec_commit_state(None, None, None, 3, 0, 16, 64, 16, 16, None, None) == sv.SPEC_ERR_INVALID_ARG
