"""Build the CUDA libraries in-tree with nvcc for sm_103a.

  libmsc.so        -- the C ABI of include/msc.h (scan + decode kernels)
  libmsc_peaks.so  -- roofline microbenchmarks (MUFU ex2, FFMA, FFMA2, copy)

Run ``python -m selective_state_space_144_b300.build`` (or call build()).
A library is rebuilt when any of its sources or headers is newer than it.
"""
from __future__ import annotations

import glob
import hashlib
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")

NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
         "--expt-relaxed-constexpr", f"-I{INCLUDE}", "-Xptxas", "-v"]

LIBS = {
    "libmsc.so": ["msc_api.cu", "scan_fwd.cu", "scan_tma.cu", "state_update.cu",
                  "conv1d.cu", "scan_bwd.cu"],
    "libmsc_peaks.so": ["peaks.cu"],
}


def lib_path(name: str) -> str:
    return os.path.join(PKG, name)


def _digest(deps: list[str], cmd: list[str]) -> str:
    """Content hash of the sources, headers and compile command."""
    h = hashlib.sha256()
    for d in sorted(deps):
        h.update(os.path.basename(d).encode())
        with open(d, "rb") as f:
            h.update(f.read())
    h.update(" ".join(cmd).encode())
    return h.hexdigest()


def _stale(target: str, digest: str) -> bool:
    """A library is rebuilt when missing or built from other content (file
    times are not used: copies of the tree do not preserve them)."""
    stamp = target + ".sha256"
    if not os.path.exists(target) or not os.path.exists(stamp):
        return True
    with open(stamp) as f:
        return f.read().strip() != digest


def build(force: bool = False, verbose: bool = False) -> list[str]:
    """Compile every library whose inputs changed; return the paths."""
    headers = (glob.glob(os.path.join(CSRC, "*.cuh"))
               + glob.glob(os.path.join(CSRC, "*.h"))
               + glob.glob(os.path.join(INCLUDE, "*.h")))
    out = []
    for name, srcs in LIBS.items():
        target = lib_path(name)
        paths = [os.path.join(CSRC, s) for s in srcs]
        digest = _digest(paths + headers, [*ARCH, *FLAGS])
        if force or _stale(target, digest):
            tmp = target + f".tmp{os.getpid()}"
            cmd = [NVCC, *ARCH, *FLAGS, "-o", tmp, *paths, "-lcudart"]
            res = subprocess.run(cmd, capture_output=True, text=True)
            if res.returncode != 0:
                sys.stderr.write(res.stdout + res.stderr)
                raise RuntimeError(f"nvcc failed building {name}")
            if verbose:
                sys.stderr.write(res.stderr)
            os.replace(tmp, target)
            with open(target + ".sha256", "w") as f:
                f.write(digest + "\n")
        out.append(target)
    return out


if __name__ == "__main__":
    for p in build(force="--force" in sys.argv, verbose=True):
        print(p)
