"""Build the in-tree CUDA library ``libmoe_b300.so`` for sm_103a with nvcc.

Usage: ``python -m mixture_experts_layer_99_b300.build [--check]`` (or
``build()``). The library is placed next to this file so that it travels with
the source tree; it links the CUDA runtime statically and needs no other CUDA
library at load time. ``--check`` (``build(check=True)``) builds the checked
variant ``libmoe_b300_check.so`` (-DMOE_CHECK: index checks in the kernels
that index with data another kernel wrote; the same ABI).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libmoe_b300.so")
LIB_CHECK = os.path.join(HERE, "libmoe_b300_check.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["api.cu", "router.cu", "router_tc.cu", "dispatch.cu", "dispatch_tiles.cu", "dispatch_static.cu", "ffn_simt.cu", "ffn_tc.cu", "combine.cu", "backward.cu", "backward_f32.cu", "ffn_wgrad_tc.cu"]


def nvcc_path() -> str:
    p = shutil.which("nvcc")
    if p:
        return p
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found")


def stale(lib: str) -> bool:
    """True if ``lib`` is missing or older than any CUDA source or header."""
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    inc = os.path.join(HERE, "..", "include")
    for d in (CSRC, inc):
        for f in os.listdir(d):
            if os.path.getmtime(os.path.join(d, f)) > t:
                return True
    return False


def build(verbose: bool = False, extra: list[str] | None = None, check: bool = False) -> str:
    """Compile every source to an object file (in parallel, one nvcc per
    file, objects under _build/ or _build_check/ beside the sources) and link
    the shared library."""
    srcs = [os.path.join(CSRC, s) for s in SOURCES if os.path.exists(os.path.join(CSRC, s))]
    lib = LIB_CHECK if check else LIB
    extra = [*(extra or []), *(["-DMOE_CHECK"] if check else [])]
    objdir = os.path.join(HERE, "_build_check" if check else "_build")
    os.makedirs(objdir, exist_ok=True)
    common = ["-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-lineinfo", *ARCH,
              "-Xcompiler", "-fvisibility=hidden", "-DMOE_BUILD_SO",
              "-I", os.path.join(HERE, "..", "include"), *extra]
    objs, procs = [], []
    for src in srcs:
        obj = os.path.join(objdir, os.path.basename(src) + ".o")
        objs.append(obj)
        cmd = [nvcc_path(), *common, "-c", "-o", obj, src]
        if verbose:
            print(" ".join(cmd))
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                            stderr=subprocess.STDOUT, text=True)))
    failed = False
    for src, pr in procs:
        out, _ = pr.communicate()
        if pr.returncode != 0:
            sys.stderr.write(out)
            failed = True
        elif verbose and out:
            print(out)
    if failed:
        raise RuntimeError(f"nvcc failed building {os.path.basename(lib)}")
    cmd = [nvcc_path(), "-shared", *ARCH, "-cudart", "static", "-o", lib + ".tmp", *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError(f"nvcc failed linking {os.path.basename(lib)}")
    os.replace(lib + ".tmp", lib)
    return lib


if __name__ == "__main__":
    args = [a for a in sys.argv[1:] if a not in ("-v", "--check")]
    print(build(verbose="-v" in sys.argv, extra=args, check="--check" in sys.argv))
