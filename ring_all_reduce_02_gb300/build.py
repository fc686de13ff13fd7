"""Build libra.so in-tree for sm_103a with nvcc (no cmake, no torch extension).

Each translation unit under csrc/ compiles in parallel (the kernel slice
source once per dtype and op); the objects link into
``ring_all_reduce_02_gb300/libra.so`` with the CUDA runtime linked statically,
so the library loads without any search-path setup.

    python -m ring_all_reduce_02_gb300.build [--verbose]
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libra.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# -fmad=false: no multiply-add contraction anywhere (every hop rounds on its own);
# no fast-math: IEEE division, subnormals kept.
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-fmad=false", "-Xcompiler", "-fPIC",
              f"-I{INCLUDE}", f"-I{CSRC}"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libra.so")
    return cand


SLICE_SOURCE = "ra_launch_op.cu"  # compiled once per (dtype id, op id)
SLICES = [(dt, op) for dt in range(4) for op in range(5)]


def sources() -> list[tuple[str, str, list[str]]]:
    """(source, object name, extra defines) for every compilation."""
    out = []
    for f in sorted(os.listdir(CSRC)):
        if not f.endswith(".cu"):
            continue
        src = os.path.join(CSRC, f)
        if f == SLICE_SOURCE:
            for dt, op in SLICES:
                out.append((src, f"ra_launch_op_{dt}_{op}.o", [f"-DRA_SLICE_DT={dt}", f"-DRA_SLICE_OP={op}"]))
        else:
            out.append((src, f[:-3] + ".o", []))
    return out


def _deps_newer(target: str) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, defines=(), lib_path: str = LIB) -> str:
    """Compile and link; ``defines`` ("NAME=VALUE") override the kernels' build-time tunables."""
    if not force and not _deps_newer(lib_path):
        return lib_path
    nvcc = _nvcc()
    out_dir = OUT_DIR if lib_path == LIB else lib_path + ".objs"
    os.makedirs(out_dir, exist_ok=True)
    extra = (["-Xptxas", "-v"] if verbose else []) + [f"-D{d}" for d in defines]

    def compile_one(job) -> str:
        src, obj_name, slice_defs = job
        obj = os.path.join(out_dir, obj_name)
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *extra, *slice_defs, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            sys.stderr.write(r.stderr)
        return obj

    jobs = sources()
    with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, jobs))
    tmp = lib_path + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


PROBE_SRC = os.path.join(HERE, "probe", "stream_probe.cu")
PROBE_LIB = os.path.join(HERE, "libra_probe.so")


def build_probe(force: bool = False) -> str:
    """Compile the stream probes (measurement kernels, not the collective path) into libra_probe.so."""
    if not force and os.path.exists(PROBE_LIB) and os.path.getmtime(PROBE_LIB) >= os.path.getmtime(PROBE_SRC):
        return PROBE_LIB
    tmp = PROBE_LIB + ".tmp"
    cmd = [_nvcc(), *ARCH, "-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-shared", "-cudart", "static",
           PROBE_SRC, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on stream_probe.cu:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, PROBE_LIB)
    return PROBE_LIB


if __name__ == "__main__":
    print(build(force=True, verbose="--verbose" in sys.argv))
    print(build_probe(force=True))
