"""Build libforge.so (and the test kit) in-tree for sm_103a with nvcc.

Each translation unit is compiled in parallel and linked into a shared
library with the CUDA runtime linked statically, so the library needs no
CUDA shared object at load time (the driver is found at first use).  Outputs
go to ``optimizer_tcgen05_dw_gb300/_build/``; a stamp holding the hash of the
sources and flags makes rebuilds incremental.
"""

import hashlib
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
INCLUDE = os.path.join(ROOT, "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-Xcompiler", "-fvisibility=hidden", "--expt-relaxed-constexpr",
                     "-I" + CSRC, "-I" + INCLUDE]

LIBS = {
    "libforge.so": ["api.cu", "tc_fused.cu", "tc_step.cu", "tc_fp8.cu", "tc_plain.cu", "elementwise.cu"],
    "libforge_testkit.so": ["testkit.cu"],
}
HEADERS = ["common.h", "launch.h", "optim.cuh", "ptx.cuh", "tc_kernel.cuh"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or put the CUDA toolkit on PATH)")


def lib_path(name: str = "libforge.so") -> str:
    return os.path.join(BUILD, name)


def _nvcc_version() -> str:
    """The toolkit's release line (e.g. "Cuda compilation tools, release 13.0,
    V13.0.88"), part of the digest so a build by another toolkit never matches."""
    try:
        out = subprocess.run([nvcc(), "--version"], capture_output=True, text=True, timeout=60).stdout
    except (OSError, RuntimeError, subprocess.SubprocessError):
        return "unknown"
    lines = [ln.strip() for ln in out.splitlines() if "release" in ln]
    return lines[0] if lines else "unknown"


def _digest(sources) -> str:
    h = hashlib.sha256()
    h.update(_nvcc_version().encode() + b"\0")
    for f in sorted(set(sources) | set(HEADERS)):
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(f.encode() + b"\0" + fh.read())
    with open(os.path.join(INCLUDE, "forge.h"), "rb") as fh:
        h.update(fh.read())
    # the flags without this checkout's absolute include paths, so that the
    # same sources hash alike wherever the repository sits
    flags = [f.replace(CSRC, "<csrc>").replace(INCLUDE, "<include>") for f in NVCC_FLAGS]
    h.update(" ".join(flags).encode())
    return h.hexdigest()


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("command failed: " + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    return r.stdout + r.stderr


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> dict:
    """Compile every library; returns {name: path}.  Skips up-to-date ones."""
    os.makedirs(BUILD, exist_ok=True)
    exe = nvcc()
    out = {}
    jobs = []
    for name, srcs in LIBS.items():
        target = lib_path(name)
        stamp = target + ".stamp"
        dig = _digest(srcs)
        out[name] = target
        if not force and os.path.exists(target) and os.path.exists(stamp):
            with open(stamp) as fh:
                if fh.read().strip() == dig:
                    continue
        jobs.append((name, srcs, target, stamp, dig))
    if not jobs:
        return out
    compile_cmds = []
    for name, srcs, target, stamp, dig in jobs:
        for src in srcs:
            obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
            cmd = [exe] + NVCC_FLAGS + (["-Xptxas", "-v"] if ptxas_info else []) + \
                ["-c", os.path.join(CSRC, src), "-o", obj]
            compile_cmds.append(cmd)
    with ThreadPoolExecutor(max_workers=min(8, len(compile_cmds))) as ex:
        logs = list(ex.map(_run, compile_cmds))
    if verbose or ptxas_info:
        for log in logs:
            if log.strip():
                print(log, file=sys.stderr)
    for name, srcs, target, stamp, dig in jobs:
        objs = [os.path.join(BUILD, os.path.splitext(s)[0] + ".o") for s in srcs]
        tmp = target + ".tmp"
        _run([exe] + ARCH + ["-shared", "-o", tmp] + objs + ["-lrt", "-ldl", "-lpthread"])
        os.replace(tmp, target)
        with open(stamp, "w") as fh:
            fh.write(dig)
    return out


if __name__ == "__main__":
    force = "--force" in sys.argv
    print(build(force=force, verbose=True, ptxas_info="--ptxas-info" in sys.argv))
