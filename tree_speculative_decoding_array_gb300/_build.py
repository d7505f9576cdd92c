"""Builds the CUDA shared libraries in place with nvcc for sm_103a.

``build_all()`` compiles every ``.cu`` of the tsv library (``csrc/``) and of the
synthetic-input filler (``synth/csrc/``) in parallel and links
``libtsv.so`` / ``libtsv_synth.so`` next to their sources.  Object files go
to ``_build/`` at the repository root.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-Xptxas", "-warn-spills"]

TARGETS = {
    "tsv": (os.path.join(PKG, "csrc"), os.path.join(PKG, "libtsv.so"), []),
    "synth": (os.path.join(ROOT, "synth", "csrc"), os.path.join(ROOT, "synth", "libtsv_synth.so"), ["-fmad=false"]),
}


def nvcc() -> str:
    p = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(p):
        raise RuntimeError("nvcc not found; the CUDA toolkit is required to build the tsv library")
    return p


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"command failed ({r.returncode}): {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return r.stdout + r.stderr


def build_target(name: str, jobs: int | None = None, verbose: bool = False) -> str:
    src_dir, out, extra = TARGETS[name]
    obj_dir = os.path.join(ROOT, "_build", name)
    os.makedirs(obj_dir, exist_ok=True)
    srcs = sorted(f for f in os.listdir(src_dir) if f.endswith(".cu"))
    cc = nvcc()
    cmds = []
    objs = []
    for s in srcs:
        o = os.path.join(obj_dir, s[:-3] + ".o")
        objs.append(o)
        cmds.append([cc, *ARCH, *FLAGS, *extra, "-I", os.path.join(ROOT, "include"), "-c",
                     os.path.join(src_dir, s), "-o", o])
    with cf.ThreadPoolExecutor(max_workers=jobs or min(len(cmds), os.cpu_count() or 4)) as ex:
        logs = list(ex.map(_run, cmds))
    if verbose:
        for s, log in zip(srcs, logs):
            if log.strip():
                print(f"--- {s}\n{log}")
    tmp = out + ".tmp"
    _run([cc, *ARCH, "-shared", "-o", tmp, *objs])
    os.replace(tmp, out)
    return out


def build_all(verbose: bool = False) -> list[str]:
    return [build_target(n, verbose=verbose) for n in TARGETS]


if __name__ == "__main__":
    import sys

    for p in build_all(verbose="-v" in sys.argv):
        print(p)
