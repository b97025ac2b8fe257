"""Build libdllm.so (the CUDA library behind include/dllm.h) for sm_103a, in-tree, and its
bounds-checked twin libdllm_checked.so (the same sources compiled with DLLM_BOUNDS_CHECK: every
global-memory access of every kernel is checked against its buffer first; see include/dllm.h).

Each translation unit under csrc/ is compiled by its own nvcc process (in parallel, both
variants at once), then linked with the CUDA runtime linked statically.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libdllm.so")
LIB_CHECKED = os.path.join(HERE, "libdllm_checked.so")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"
# variant -> (library, object folder, extra nvcc flags)
VARIANTS = {
    "regular": (LIB, BUILD, []),
    "checked": (LIB_CHECKED, os.path.join(BUILD, "checked"), ["-DDLLM_BOUNDS_CHECK"]),
}


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found (set NVCC or install the CUDA toolkit)")


def _flags():
    return ["-std=c++17", "-O3", ARCH, "-lineinfo", "-Xcompiler", "-fPIC,-fvisibility=hidden",
            "-I", os.path.join(ROOT, "include"), "-I", CSRC, "-Xptxas", "-v,-warn-spills",
            "--expt-relaxed-constexpr"]


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    return [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(ROOT, "include", "dllm.h")]


def _compile(job: tuple[str, str, list[str]]) -> tuple[str, str]:
    src, objdir, extra = job
    obj = os.path.join(objdir, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc(), *_flags(), *extra, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def _link(lib: str, objs: list[str]) -> None:
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc(), ARCH, "-shared", "-cudart=static", "-o", tmp, *objs, "-ldl", "-lpthread", "-lrt"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link libdllm.so and libdllm_checked.so where a source is newer than the
    library. Returns the path of libdllm.so."""
    newest = max(os.path.getmtime(p) for p in _deps())
    todo = [v for v, (lib, _, _) in VARIANTS.items()
            if force or not os.path.exists(lib) or os.path.getmtime(lib) < newest]
    if not todo:
        return LIB
    srcs = _sources()
    jobs = []
    for v in todo:
        objdir, extra = VARIANTS[v][1], VARIANTS[v][2]
        os.makedirs(objdir, exist_ok=True)
        jobs += [(s, objdir, extra) for s in srcs]
    with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
        results = list(ex.map(_compile, jobs))
    for i, v in enumerate(todo):
        part = results[i * len(srcs):(i + 1) * len(srcs)]
        logs = [log for _, log in part]
        if verbose:
            for log in logs:
                sys.stderr.write(log)
        with open(os.path.join(VARIANTS[v][1], "ptxas.log"), "w") as f:
            f.write("\n".join(logs))
        _link(VARIANTS[v][0], [obj for obj, _ in part])
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
