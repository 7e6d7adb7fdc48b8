"""Build libspecverify.so in-tree with nvcc for GB300 (sm_103a)."""

import os
import shutil
import subprocess
import tempfile
from concurrent.futures import ThreadPoolExecutor

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
REPO_DIR = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(REPO_DIR, "include")
LIB_NAME = "libspecverify.so"
LIB_PATH = os.path.join(PKG_DIR, LIB_NAME)

NVCC_FLAGS = [
    "-O3", "-std=c++17", "-lineinfo",
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-Xcompiler", "-fPIC",
]


def _sources():
    files = [os.path.join(CSRC, f) for f in sorted(os.listdir(CSRC))]
    files += [os.path.join(INCLUDE, f) for f in sorted(os.listdir(INCLUDE)) if f.endswith(".h")]
    return files


def _translation_units():
    return [os.path.join(CSRC, f) for f in sorted(os.listdir(CSRC)) if f.endswith(".cu")]


def _nvcc():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libspecverify.so")
    return nvcc


def up_to_date():
    if not os.path.exists(LIB_PATH):
        return False
    built = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(f) <= built for f in _sources())


def build_library(force=False, verbose=False):
    """Compile the csrc/*.cu translation units into one library in the package
    directory; return its path."""
    if not force and up_to_date():
        return LIB_PATH
    tmp = LIB_PATH + ".tmp"
    nvcc = _nvcc()
    with tempfile.TemporaryDirectory(prefix="specverify-build-") as objdir:
        # Translation units compile in parallel (each kernel build is one), then link.
        units = _translation_units()
        objs = [os.path.join(objdir, os.path.basename(u) + ".o") for u in units]
        cmds = [[nvcc, *NVCC_FLAGS, *(["-Xptxas=-v"] if verbose else []), "-I" + INCLUDE, "-c", "-o", o, u]
                for u, o in zip(units, objs)]
        with ThreadPoolExecutor(max_workers=max(1, min(len(cmds), os.cpu_count() or 1))) as pool:
            results = list(pool.map(lambda c: (c, subprocess.run(c, capture_output=True, text=True)), cmds))
        link = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-shared", "-o", tmp, *objs]
        results.append((link, subprocess.run(link, capture_output=True, text=True)))
        for cmd, res in results:
            if res.returncode != 0:
                raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + res.stdout + res.stderr)
            if verbose:
                print(res.stdout + res.stderr)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build_library(force=True, verbose=True))
