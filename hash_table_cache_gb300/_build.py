"""Compile the CUDA library (libhkv.so) in-tree for sm_103a with nvcc."""
from __future__ import annotations

import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libhkv.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["table.cu", "find.cu", "upsert.cu", "export.cu", "no_alloc.cu"]
# measurement helper used by bench.py, kept out of the table library
PROBE_SOURCE = "access_probe.cu"
PROBE_LIB = os.path.join(PKG, "libhkv_probe.so")
# digest-ablation build of the library (find without the digest line, HKV
# §5.4 Table 7): same ABI, used only by the ablation test and bench.py
NODIGEST_LIB = os.path.join(PKG, "libhkv_nodigest.so")
NODIGEST_FLAGS = ("-DHKV_FIND_NO_DIGEST=1",)
# pipelined build (the bucket kernel stages each warp's next bucket in shared
# memory with bulk copies): same ABI, for the pipeline measurement only
PIPELINE_LIB = os.path.join(PKG, "libhkv_pipeline.so")
PIPELINE_FLAGS = ("-DHKV_UPSERT_PIPELINE=1",)
VARIANTS = {"nodigest": (NODIGEST_LIB, NODIGEST_FLAGS), "pipeline": (PIPELINE_LIB, PIPELINE_FLAGS)}


def _nvcc():
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "hkv.h"))
    return max(os.path.getmtime(f) for f in files)


def build_all(force: bool = False) -> None:
    """libhkv.so (+ libhkv_probe.so) and the measurement variants
    (libhkv_nodigest.so, libhkv_pipeline.so), compiled concurrently."""
    with ThreadPoolExecutor(max_workers=1 + len(VARIANTS)) as ex:
        jobs = [ex.submit(build, force)]
        jobs += [ex.submit(build, force, False, fl, lib) for lib, fl in VARIANTS.values()]
        for j in jobs:
            j.result()


def build(force: bool = False, verbose: bool = False, extra_flags=(), out: str = LIB) -> str:
    """Compile every source and link `out` (default: the in-tree libhkv.so).
    `extra_flags` are passed to nvcc (e.g. -D tuning macros)."""
    if not force and out in (LIB, NODIGEST_LIB, PIPELINE_LIB) and os.path.exists(out) and \
            os.path.getmtime(out) >= _deps():
        return out
    build_dir = BUILD if out == LIB else os.path.join(BUILD, os.path.basename(out) + ".objs")
    os.makedirs(build_dir, exist_ok=True)
    nvcc = _nvcc()
    flags = ["-O3", "-std=c++17", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC",
             "-I", INCLUDE, "-I", CSRC, *extra_flags]
    if verbose:
        flags += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(build_dir, src.replace(".cu", ".o"))
        cmd = [nvcc, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
        return obj, r.stderr

    with_probe = out == LIB
    with ThreadPoolExecutor(max_workers=len(SOURCES) + 1) as ex:
        results = list(ex.map(compile_one, SOURCES + ([PROBE_SOURCE] if with_probe else [])))
    if verbose:
        for _, err in results:
            print(err)
    if with_probe:
        _link([results[-1][0]], PROBE_LIB)
        results = results[:-1]
    _link([o for o, _ in results], out)
    return out


def _link(objs, out):
    tmp = out + f".tmp{os.getpid()}"
    r = subprocess.run([_nvcc(), "-shared", *ARCH, "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, out)


if __name__ == "__main__":
    import sys
    build(force=True, verbose="-v" in sys.argv)
    print(LIB)
