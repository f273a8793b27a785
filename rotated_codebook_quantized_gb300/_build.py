"""Build of libtq.so: every CUDA source compiled for sm_103a with nvcc, in parallel.

Run ``python -m rotated_codebook_quantized_gb300._build`` or call ``build()``.
Objects go to ``_build/`` inside the package; the shared library is written
next to this file, where the binding loads it from.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJDIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libtq.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
              "--expt-relaxed-constexpr"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


# qmv_inst.cu is compiled once per (levels, group) pair so the templates build in parallel.
QMV_VARIANTS = [(lv, g) for lv in (3, 4, 8, 16) for g in (16, 32, 64, 128)]
# qmv_rows.cu: its entry points, then the kernel instances of each bit-packed book.
ROWS_VARIANTS = (0, 4, 8, 16)


def sources() -> list[tuple[str, str, list[str]]]:
    """(source, object name, extra defines) for every translation unit."""
    out = []
    for f in sorted(os.listdir(CSRC)):
        if not f.endswith(".cu"):
            continue
        src = os.path.join(CSRC, f)
        if f == "qmv_inst.cu":
            for lv, g in QMV_VARIANTS:
                out.append((src, f"qmv_l{lv}_g{g}.o", [f"-DTQ_LEVELS={lv}", f"-DTQ_GROUP={g}"]))
        elif f == "qmv_rows.cu":  # the entry points (0), then one unit per bit-packed book
            for lv in ROWS_VARIANTS:
                out.append((src, f"qmv_rows_l{lv}.o", [f"-DTQ_ROWS_LEVELS={lv}"]))
        else:
            out.append((src, f[:-3] + ".o", []))
    return out


def _compile(unit: tuple[str, str, list[str]], extra: list[str]) -> str:
    src, objname, defs = unit
    obj = os.path.join(OBJDIR, objname)
    deps = [src] + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    deps.append(os.path.join(INCLUDE, "tq.h"))
    if os.path.exists(obj) and os.path.getmtime(obj) >= max(os.path.getmtime(d) for d in deps):
        return obj
    cmd = [nvcc()] + ARCH + NVCC_FLAGS + defs + extra + ["-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if r.stderr.strip() and "-Xptxas" in " ".join(extra):
        sys.stderr.write(r.stderr)
    return obj


def build(verbose: bool = False, extra: list[str] | None = None) -> str:
    """Compile every .cu under csrc/ and link libtq.so; returns its path."""
    os.makedirs(OBJDIR, exist_ok=True)
    extra = list(extra or [])
    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra), srcs))
    if os.path.exists(LIB) and os.path.getmtime(LIB) >= max(os.path.getmtime(o) for o in objs):
        return LIB
    tmp = LIB + ".tmp"
    cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs + ["-lcudart"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    if verbose:
        print(f"built {LIB}")
    return LIB


if __name__ == "__main__":
    build(verbose=True, extra=sys.argv[1:])
