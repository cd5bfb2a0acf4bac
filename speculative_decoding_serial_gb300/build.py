"""Builds the CUDA library (libwhead.so) in-tree with nvcc for sm_103a."""
from __future__ import annotations

import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libwhead.so")
SOURCES = [os.path.join(CSRC, "whead_api.cu")]
DEPS = SOURCES + [os.path.join(CSRC, "walk_kernel.cuh"), os.path.join(ROOT, "include", "whead.h")]
# measurement-only library used by the benchmark for the roofline's on-chip figures
PROBE_LIB = os.path.join(BUILD, "libwhead_probe.so")
PROBE_SRC = os.path.join(CSRC, "onchip_probe.cu")

NVCC_FLAGS = ["-O3", "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo",
              "-Xcompiler", "-fPIC", "-shared", "-Xptxas", "-v"]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def needs_build() -> bool:
    for lib, deps in ((LIB, DEPS), (PROBE_LIB, [PROBE_SRC])):
        if not os.path.exists(lib) or any(os.path.getmtime(d) > os.path.getmtime(lib) for d in deps):
            return True
    return False


def _compile(out: str, sources, log_name: str, verbose: bool) -> None:
    tmp = out + f".tmp{os.getpid()}"
    cmd = [nvcc()] + NVCC_FLAGS + ["-I", os.path.join(ROOT, "include"), "-o", tmp] + list(sources)
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + res.stdout + res.stderr)
    with open(os.path.join(BUILD, log_name), "w") as f:
        f.write(res.stderr)
    if verbose:
        print(res.stderr)
    os.replace(tmp, out)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libwhead.so (and the probe library) if missing or older than their sources; returns LIB."""
    os.makedirs(BUILD, exist_ok=True)
    if force or not os.path.exists(LIB) or any(os.path.getmtime(d) > os.path.getmtime(LIB) for d in DEPS):
        _compile(LIB, SOURCES, "ptxas_info.txt", verbose)
    if force or not os.path.exists(PROBE_LIB) or os.path.getmtime(PROBE_SRC) > os.path.getmtime(PROBE_LIB):
        _compile(PROBE_LIB, [PROBE_SRC], "ptxas_probe.txt", verbose)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
