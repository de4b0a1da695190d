"""Build libpagedkv.so in-tree for sm_103a (nvcc, one translation unit per job).

    python -m paged_kv_cache_170_gb300.build [--force] [--verbose] [--variant faulttest]

The ``faulttest`` variant (its own folder, ``_build_faulttest/``) is for the
test of the kernels' bounded waits only: the decode's producer never issues the
first ring entry of the CTA that owns the step's first tile, and the waits
give up after about half a second instead of 1.5 s.  Nothing but that test loads it.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(OUT_DIR, "libpagedkv.so")
SOURCES = ["pa_kv.cu", "pa_decode.cu", "pa_decode_f32.cu", "pa_decode_f16.cu", "pa_decode_bf16.cu",
           "pa_decode_noalloc.cu", "pa_share.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
DEBUG = (["-DPA_DEBUG"] if os.environ.get("PA_DEBUG") == "1" else []) + \
    (["-DPA_TRACE"] if os.environ.get("PA_TRACE") == "1" else [])
if os.environ.get("PA_TRACE") == "1" and os.environ.get("PA_TRACE_CTAS"):
    # comma-separated CTA indices whose warps print their trace counters
    _ctas = [int(c) for c in os.environ["PA_TRACE_CTAS"].split(",")]
    DEBUG.append("-DPA_TRACE_CTA(c)=(" + "||".join(f"(c)=={c}" for c in _ctas) + ")")
FLAGS = DEBUG + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _deps_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(ROOT, "include", "pagedkv.h")]
    return max(os.path.getmtime(f) for f in files)


VARIANTS = {
    "": [],
    # one lost arrival and a 1e9-cycle wait limit (see the module docstring)
    "faulttest": ["-DPA_FAULT_WITHHOLD_FIRST_ENTRY", "-DPA_WAIT_LIMIT_CYCLES=1000000000LL"],
}


def lib_path(variant: str = "") -> str:
    return LIB if not variant else os.path.join(PKG, f"_build_{variant}", "libpagedkv.so")


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False, variant: str = "") -> str:
    out_dir = os.path.dirname(lib_path(variant))
    lib = lib_path(variant)
    flags = FLAGS + VARIANTS[variant]
    os.makedirs(out_dir, exist_ok=True)
    stamp = os.path.join(out_dir, "flags.txt")
    flags_now = " ".join(ARCH + flags)
    same_flags = os.path.exists(stamp) and open(stamp).read() == flags_now
    if not force and same_flags and os.path.exists(lib) and os.path.getmtime(lib) >= _deps_mtime():
        return lib
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_verbose else []

    def compile_one(src: str) -> tuple[str, str]:
        obj = os.path.join(out_dir, src.replace(".cu", ".o"))
        cmd = [cc, *ARCH, *flags, *extra, "-I", os.path.join(ROOT, "include"), "-c", os.path.join(CSRC, src),
               "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=min(len(SOURCES), os.cpu_count() or 4)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose or ptxas_verbose:
        for _, log in results:
            sys.stderr.write(log)
    objs = [o for o, _ in results]
    tmp = lib + ".tmp"
    r = subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, lib)
    with open(stamp, "w") as f:
        f.write(flags_now)
    return lib


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--ptxas", action="store_true", help="print ptxas register/smem usage")
    ap.add_argument("--variant", choices=sorted(VARIANTS), default="")
    args = ap.parse_args()
    print(build(force=args.force, verbose=args.verbose, ptxas_verbose=args.ptxas, variant=args.variant))
