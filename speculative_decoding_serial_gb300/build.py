"""Builds the CUDA library (libwhead.so) in-tree with nvcc for sm_103a."""
from __future__ import annotations

import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libwhead.so")
# the host library and the walk kernel's instantiations (Markov / recurrent head x base logits read at each step /
# copied a step ahead), compiled in parallel
SOURCES = [os.path.join(CSRC, n) for n in ("whead_api.cu", "walk_resident.cu", "walk_resident_rec.cu",
                                           "walk_async.cu", "walk_async_rec.cu")]
DEPS = SOURCES + [os.path.join(CSRC, n) for n in ("walk_kernel.cuh", "walk_launch.cuh", "walk_launch.h")] + [
    os.path.join(ROOT, "include", "whead.h")]
# measurement-only library used by the benchmark for the roofline's on-chip figures
PROBE_LIB = os.path.join(BUILD, "libwhead_probe.so")
PROBE_SRC = os.path.join(CSRC, "onchip_probe.cu")

NVCC_FLAGS = ["-O3", "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo",
              "-Xcompiler", "-fPIC", "-Xptxas", "-v"]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def needs_build() -> bool:
    for lib, deps in ((LIB, DEPS), (PROBE_LIB, [PROBE_SRC])):
        if not os.path.exists(lib) or any(os.path.getmtime(d) > os.path.getmtime(lib) for d in deps):
            return True
    return False


def _compile(out: str, sources, log_name: str, verbose: bool) -> None:
    """Each source to an object file (all at once, one nvcc process per source), then one shared library."""
    tag = f".tmp{os.getpid()}"
    objs = [os.path.join(BUILD, os.path.splitext(os.path.basename(src))[0] + tag + ".o") for src in sources]
    procs = [subprocess.Popen([nvcc()] + NVCC_FLAGS + ["-I", os.path.join(ROOT, "include"), "-c", "-o", obj, src],
                              stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)
             for src, obj in zip(sources, objs)]
    logs, failed = [], []
    for src, p in zip(sources, procs):
        o, e = p.communicate()
        logs.append(e)
        if p.returncode != 0:
            failed.append(f"{os.path.basename(src)}:\n{o}{e}")
    try:
        if failed:
            raise RuntimeError("nvcc failed:\n" + "\n".join(failed))
        tmp = out + tag
        res = subprocess.run([nvcc(), "-shared", "-gencode", "arch=compute_103a,code=sm_103a", "-o", tmp] + objs,
                             capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError("nvcc link failed:\n" + res.stdout + res.stderr)
    finally:
        for obj in objs:
            if os.path.exists(obj):
                os.remove(obj)
    with open(os.path.join(BUILD, log_name), "w") as f:
        f.write("".join(logs))
    if verbose:
        print("".join(logs))
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
