"""Build libe3gb.so in-tree with nvcc for sm_103a.

Each irreps configuration of csrc/configs.def is its own translation unit (instances.cu
compiled with -DE3GB_CFG=<id>); units compile in parallel and are linked into
message_passing_gb300/lib/libe3gb.so. Rebuilds only what changed.
"""
from __future__ import annotations

import os
import re
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
LIBDIR = os.path.join(HERE, "lib")
OBJDIR = os.path.join(LIBDIR, "obj")
LIB = os.path.join(LIBDIR, "libe3gb.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-std=c++20", "--expt-relaxed-constexpr", "-O3", "-lineinfo", "-Xcompiler", "-fPIC",
         "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def config_ids() -> list[int]:
    ids = []
    with open(os.path.join(CSRC, "configs.def")) as f:
        for line in f:
            m = re.match(r"\s*E3GB_CONFIG\((\d+),", line)
            if m:
                ids.append(int(m.group(1)))
    return ids


def _headers() -> list[str]:
    hs = [os.path.join(CSRC, h) for h in os.listdir(CSRC) if h.endswith((".hpp", ".cuh", ".def"))]
    return hs + [os.path.join(ROOT, "include", "e3gb.h")]


def _stale(obj: str, deps: list[str]) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(d) > t for d in deps)


def units() -> list[tuple[str, str, list[str]]]:
    """(source, object, extra flags)"""
    u = [(os.path.join(CSRC, s), os.path.join(OBJDIR, s.replace(".cu", ".o")), [])
         for s in ("api.cu", "sh.cu", "graph.cu", "coo.cu", "radial.cu")]
    for i in config_ids():
        # forward, backward, double backward (plain, pipelined), narrow forward, radial conv
        for part in (0, 1, 2, 3, 4, 5):
            u.append((os.path.join(CSRC, "instances.cu"), os.path.join(OBJDIR, f"cfg{i}_{part}.o"),
                      [f"-DE3GB_CFG={i}", f"-DE3GB_PART={part}"]))
    return u


def build(verbose: bool = False, ptxas_info: bool = False, jobs: int | None = None) -> str:
    os.makedirs(OBJDIR, exist_ok=True)
    cc = nvcc()
    hdr = _headers()
    todo = [(s, o, x) for s, o, x in units() if _stale(o, [s] + hdr) or ptxas_info]

    def compile_one(job):
        src, obj, extra = job
        tmp = obj + f".{os.getpid()}.tmp.o"
        cmd = [cc, *ARCH, *FLAGS, *extra, "-c", src, "-o", tmp]
        if ptxas_info:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {os.path.basename(obj)}:\n{r.stderr[-6000:]}")
        os.replace(tmp, obj)
        return obj, r.stderr

    n = jobs or max(1, min(len(todo), os.cpu_count() or 1))
    logs = []
    if todo:
        with ThreadPoolExecutor(n) as ex:
            for obj, err in ex.map(compile_one, todo):
                logs.append((obj, err))
                if verbose:
                    print("built", os.path.basename(obj), file=sys.stderr)
    objs = [o for _, o, _ in units()]
    if todo or not os.path.exists(LIB) or _stale(LIB, objs):
        tmp = LIB + f".{os.getpid()}.tmp"
        r = subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr[-4000:]}")
        os.replace(tmp, LIB)
    if ptxas_info:
        for obj, err in logs:
            print(f"== {os.path.basename(obj)}\n{err}")
    return LIB


if __name__ == "__main__":
    build(verbose=True, ptxas_info="-v" in sys.argv)
