"""Build the CUDA library in-tree: ``_build/libtg_gemm_<machine>.so``.

Translation units (compiled in parallel, one ``-gencode`` for sm_103a):
* ``csrc/tg_host.cu``    - C ABI, validation, planner, workspaces, TMA
                           descriptors, pack and zero-fill kernels;
* ``csrc/tg_kernels.cu`` - the persistent GEMM kernel, once per tile width
                           (-DTG_BN=64/128/192/256);
* ``csrc/tg_noalloc.cu`` - the split-K entry point whose scratch is a static
                           device array (no run-time allocation);
* ``csrc/tg_direct.cu``  - the direct-load kernel for small problems.
The CUDA runtime is linked statically, so the library loads on a machine
without a GPU (every CUDA call then returns an error) and exports only the
``tg_*`` entry points of ``include/tg_gemm.h``.

``build(checks=True)`` builds the same sources with ``-DTG_DEBUG_CHECKS``
into ``_build/libtg_gemm_checks_<machine>.so``: the kernels then verify
their work units, ring slots, tensor-memory columns, shared-memory layout
and split-K scratch indices on the device and report a failure through
``tg_device_error`` (TG_ERR_DEVICE_CHECK) instead of touching memory out of
range.  Tests run it beside the product library.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import platform
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
WIDTHS = (64, 128, 192, 256)
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def library_path(checks: bool = False) -> str:
    name = "libtg_gemm_checks" if checks else "libtg_gemm"
    return os.path.join(BUILD, f"{name}_{platform.machine()}.so")


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")


def _sources() -> list[str]:
    out = []
    for d in (CSRC, INCLUDE):
        for name in sorted(os.listdir(d)):
            if name.endswith((".cu", ".cuh", ".h")):
                out.append(os.path.join(d, name))
    return out


def _common_flags() -> list[str]:
    return [ARCH, "-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr",
            "-Xcompiler", "-fPIC,-fvisibility=hidden", f"-I{INCLUDE}", f"-I{CSRC}"]


def _compile(args):
    src, obj, defs = args
    cmd = [_nvcc(), *_common_flags(), *defs, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(obj)}:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def build(force: bool = False, verbose: bool = False, extra_flags: list[str] | None = None,
          checks: bool = False) -> str:
    """Compile and link the library if any source is newer than it (checks:
    the TG_DEBUG_CHECKS build, objects and library under their own names)."""
    out = library_path(checks)
    if not force and os.path.exists(out):
        newest = max(os.path.getmtime(s) for s in _sources())
        if os.path.getmtime(out) >= newest:
            return out
    os.makedirs(BUILD, exist_ok=True)
    machine = platform.machine() + ("_checks" if checks else "")
    jobs = [(os.path.join(CSRC, "tg_host.cu"), os.path.join(BUILD, f"tg_host_{machine}.o"), []),
            (os.path.join(CSRC, "tg_noalloc.cu"), os.path.join(BUILD, f"tg_noalloc_{machine}.o"), []),
            (os.path.join(CSRC, "tg_direct.cu"), os.path.join(BUILD, f"tg_direct_{machine}.o"), [])]
    for bn in WIDTHS:
        jobs.append((os.path.join(CSRC, "tg_kernels.cu"),
                     os.path.join(BUILD, f"tg_kernels_bn{bn}_{machine}.o"), [f"-DTG_BN={bn}"]))
    flags = (["-DTG_DEBUG_CHECKS"] if checks else []) + list(extra_flags or [])
    if flags:
        jobs = [(s, o, d + flags) for (s, o, d) in jobs]
    with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        results = list(ex.map(_compile, jobs))
    if verbose:
        for obj, err in results:
            if err.strip():
                print(f"== {os.path.basename(obj)}\n{err}")
    tmp = out + f".tmp{os.getpid()}"
    cmd = [_nvcc(), ARCH, "-shared", "-cudart", "static", "-o", tmp,
           *[o for o, _ in results], "-Xlinker", "--exclude-libs,ALL"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    import sys

    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                extra_flags=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else None,
                checks="--checks" in sys.argv))
