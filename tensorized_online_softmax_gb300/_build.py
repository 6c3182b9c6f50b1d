"""Compile the CUDA library (C ABI of include/fat_attn.h) for sm_103a, in-tree."""
from __future__ import annotations

import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_NAME = "libfat_attn.so"
LIB_PATH = os.path.join(BUILD_DIR, LIB_NAME)
NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-std=c++17", "-lineinfo",
    "-Xcompiler", "-fPIC",
    # the per-device launch state sits in function-local statics of kernel
    # templates; without this GCC marks them unique across every loaded
    # library, so a second copy of this library in one process would find
    # another copy's state and skip its own kernel set-up
    "-Xcompiler", "-fno-gnu-unique",
]


def translation_units():
    """Every .cu in csrc: the C ABI plus one file per group of kernel instances."""
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _sources():
    # (this file too: a change of flags rebuilds)
    return (glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh"))
            + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(ROOT, "include", "*.h"))
            + [os.path.abspath(__file__)])


def nvcc_path() -> str | None:
    cand = shutil.which("nvcc")
    if cand:
        return cand
    for p in ("/usr/local/cuda/bin/nvcc",):
        if os.path.exists(p):
            return p
    return None


def is_stale(path: str = LIB_PATH) -> bool:
    if not os.path.exists(path):
        return True
    t = os.path.getmtime(path)
    return any(os.path.getmtime(s) > t for s in _sources())


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Build ``_build/libfat_attn.so`` with nvcc (sm_103a only).

    The translation units compile in parallel (one nvcc per unit), then link.
    """
    if not force and not is_stale():
        return LIB_PATH
    nvcc = nvcc_path()
    if nvcc is None:
        raise RuntimeError("nvcc not found: cannot build the CUDA library")
    os.makedirs(BUILD_DIR, exist_ok=True)
    tag = f".tmp{os.getpid()}"
    units = translation_units()
    objs = [os.path.join(BUILD_DIR, os.path.basename(u)[:-3] + tag + ".o") for u in units]
    procs = []
    for u, o in zip(units, objs):
        cmd = [nvcc, *NVCC_FLAGS, *extra_flags, "-c", "-o", o, u]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        procs.append((u, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT,
                                          text=True)))
    failed, logs = [], []
    for u, pr in procs:
        out, _ = pr.communicate()
        logs.append(out)
        if pr.returncode != 0:
            failed.append((u, out))
    if failed:
        for o in objs:
            if os.path.exists(o):
                os.remove(o)
        raise RuntimeError("nvcc failed:\n" + "\n".join(f"{u}:\n{out}" for u, out in failed))
    if verbose:
        print("".join(logs))
    tmp = LIB_PATH + tag
    res = subprocess.run([nvcc, "-shared", "-gencode", "arch=compute_103a,code=sm_103a", "-o", tmp,
                          *objs], capture_output=True, text=True)
    for o in objs:
        os.remove(o)
    if res.returncode != 0:
        raise RuntimeError("nvcc link failed:\n" + res.stdout + res.stderr)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH
