"""Build libadp.so (the engine's C ABI) in-tree with nvcc for sm_103a.

Seven translation units compiled in parallel, then linked as a shared library with the
static CUDA runtime. -fmad=false keeps every multiply-add that the arithmetic contract does
not fuse explicitly as a separate multiply and add; no fast-math flags.

A second library, libadp_test.so, links the same objects with the host engine compiled once more
under -DADP_TEST_HOOKS: it also exports the test-only hooks (withholding a phase's outputs,
shortening the in-kernel waits, moving the epoch counter).  The tests load it; the release
library, which the benchmark and applications load, does not carry those hooks.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libadp.so")
TEST_LIB = os.path.join(HERE, "libadp_test.so")
SOURCES = ["decode.cu", "decode_batch.cu", "prefill.cu", "repack.cu", "engine.cu", "noalloc.cu", "probe.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-fmad=false", "-Xcompiler", "-fPIC", "-Xcompiler", "-ffp-contract=off",
         "-Xcompiler", "-fvisibility=hidden"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the engine")


def _extra_flags() -> list[str]:
    """Extra nvcc flags from ADP_NVCC_FLAGS (e.g. -DADP_CYCLE_STAMPS for the timeline's cycle
    breakdowns); a change of them forces a rebuild."""
    return os.environ.get("ADP_NVCC_FLAGS", "").split()


FLAGS_STAMP = os.path.join(HERE, "_build", "flags.txt")


def _stale() -> bool:
    if not os.path.exists(LIB) or not os.path.exists(TEST_LIB):
        return True
    try:
        if open(FLAGS_STAMP).read() != " ".join(_extra_flags()):
            return True
    except OSError:
        return True
    t = min(os.path.getmtime(LIB), os.path.getmtime(TEST_LIB))
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    deps.append(os.path.join(os.path.dirname(HERE), "include", "adp.h"))
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not _stale():
        return LIB
    cc = nvcc()
    outdir = os.path.join(HERE, "_build")
    os.makedirs(outdir, exist_ok=True)

    def compile_one(job):
        src, extra, obj_name = job
        obj = os.path.join(outdir, obj_name)
        cmd = [cc, *ARCH, *FLAGS, *_extra_flags(), *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr)
        return obj

    jobs = [(src, [], src.replace(".cu", ".o")) for src in SOURCES]
    jobs.append(("engine.cu", ["-DADP_TEST_HOOKS"], "engine_hooks.o"))
    with cf.ThreadPoolExecutor(len(jobs)) as ex:
        objs = list(ex.map(compile_one, jobs))
    release = objs[:len(SOURCES)]
    test = [o if not o.endswith(os.sep + "engine.o") else objs[-1] for o in release]
    for lib, members in ((LIB, release), (TEST_LIB, test)):
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [cc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *members]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr}")
        os.replace(tmp, lib)
    with open(FLAGS_STAMP, "w") as fh:
        fh.write(" ".join(_extra_flags()))
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
