"""Build ``libkda.so`` (the C-ABI CUDA library) in-tree with nvcc for sm_103a.

Each ``csrc/*.cu`` translation unit is compiled in parallel to an object in
``_build/`` and the objects are linked into ``libkda.so`` next to this file.
The same sources compiled with ``-DKDA_FAULT_INJECTION`` give
``libkda_faultinj.so``, a test-only copy of the library whose
``kda_test_force_timeout`` makes the prefill's bounded device wait give up on
purpose (the tests use it to check the timeout path); both are built in one
parallel pass.  Usage: ``python -m serving_kda_chunked_gb300.build [--force]``.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libkda.so")
FAULTINJ_LIB = os.path.join(HERE, "libkda_faultinj.so")
VARIANTS = ((LIB, "", []), (FAULTINJ_LIB, "faultinj", ["-DKDA_FAULT_INJECTION"]))

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr",
              "-Xcompiler", "-fPIC", "-I", INCLUDE]


def nvcc() -> str:
    for cand in (os.environ.get("CUDA_HOME", ""), "/usr/local/cuda"):
        p = os.path.join(cand, "bin", "nvcc") if cand else ""
        if p and os.path.exists(p):
            return p
    p = shutil.which("nvcc")
    if not p:
        raise RuntimeError("nvcc not found: the KDA CUDA library cannot be built")
    return p


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps() -> list[str]:
    return (sources() + glob.glob(os.path.join(CSRC, "*.cuh"))
            + glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)])


def up_to_date() -> bool:
    for lib, _, _ in VARIANTS:
        if not os.path.exists(lib):
            return False
        t = os.path.getmtime(lib)
        if any(os.path.getmtime(d) > t for d in _deps()):
            return False
    return True


def build(force: bool = False, verbose: bool = False, extra_flags=None) -> str:
    if not force and up_to_date():
        return LIB
    cc = nvcc()
    procs = []
    links = []
    for lib, sub, vflags in VARIANTS:
        bdir = os.path.join(BUILD, sub) if sub else BUILD
        os.makedirs(bdir, exist_ok=True)
        flags = NVCC_FLAGS + vflags + list(extra_flags or [])
        objs = []
        for src in sources():
            obj = os.path.join(bdir, os.path.basename(src)[:-3] + ".o")
            objs.append(obj)
            cmd = [cc, *ARCH, *flags, "-c", src, "-o", obj]
            if verbose:
                print(" ".join(cmd), flush=True)
            procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                                stderr=subprocess.STDOUT)))
        links.append((lib, objs))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        text = out.decode(errors="replace")
        if p.returncode != 0:
            failed.append((src, text))
        elif verbose and text.strip():
            print(text, flush=True)
    if failed:
        msg = "\n".join("%s:\n%s" % (s, t) for s, t in failed)
        raise RuntimeError("nvcc failed:\n" + msg)
    for lib, objs in links:
        tmp = lib + ".tmp.%d" % os.getpid()
        cmd = [cc, *ARCH, "-shared", "-cudart", "shared", *objs, "-o", tmp]
        subprocess.run(cmd, check=True)
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
