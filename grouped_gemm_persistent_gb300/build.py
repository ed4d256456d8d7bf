"""Build libtg.so (the CUDA kernels and the C ABI) in-tree with nvcc for sm_103a.

    python -m grouped_gemm_persistent_gb300.build [--force] [--verbose-ptxas]

Translation units compile in parallel: the host API and the auxiliary kernels once, the kernel
instantiations once per (output dtype, dense / grouped / MoE) pair.  The result is
grouped_gemm_persistent_gb300/libtg.so; objects go to
grouped_gemm_persistent_gb300/_build/.  A rebuild happens only when a source
or a flag changed (content hash).
"""
from __future__ import annotations

import argparse
import hashlib
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libtg.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
                "--expt-relaxed-constexpr"]

UNITS = [("tg_api", "tg_api.cu", []), ("tg_aux", "tg_aux.cu", [])] + [
    (f"tg_inst_f{f}_m{m}", "tg_inst.cu", [f"-DTG_INST_F32={f}", f"-DTG_INST_MODE={m}"])
    for f in (0, 1) for m in (0, 1, 2)
]


def nvcc() -> str:
    exe = shutil.which("nvcc")
    if exe:
        return exe
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libtg")


def _digest(extra_flags) -> str:
    h = hashlib.sha256()
    for d in (CSRC, INCLUDE):
        for name in sorted(os.listdir(d)):
            p = os.path.join(d, name)
            if os.path.isfile(p):
                h.update(name.encode())
                with open(p, "rb") as f:
                    h.update(f.read())
    # flags with the checkout's location taken out, so a copy elsewhere hashes the same
    h.update(" ".join(FLAGS + list(extra_flags)).replace(ROOT, "<root>").encode())
    return h.hexdigest()


def _strip_comments(src: str) -> str:
    """C/C++/CUDA source without its comments, trailing blanks and empty lines (string
    and character literals are kept as they are)."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    lines = [l.rstrip() for l in "".join(out).splitlines()]
    return "\n".join(l for l in lines if l)


def code_digest() -> str:
    """Hash of the kernel and API sources with comments and blank lines taken out: it
    changes only when the compiled code can change (the key of profiles/traffic.txt)."""
    h = hashlib.sha256()
    for d in (CSRC, INCLUDE):
        for name in sorted(os.listdir(d)):
            p = os.path.join(d, name)
            if os.path.isfile(p):
                h.update(name.encode())
                with open(p, encoding="utf-8") as f:
                    h.update(_strip_comments(f.read()).encode())
    h.update(" ".join(FLAGS).replace(ROOT, "<root>").encode())
    return h.hexdigest()


def build(force: bool = False, verbose_ptxas: bool = False, jobs: int | None = None) -> str:
    os.makedirs(BUILD, exist_ok=True)
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    stamp = os.path.join(BUILD, "stamp")
    digest = _digest(extra)
    if not force and os.path.exists(LIB) and os.path.exists(stamp) and open(stamp).read() == digest:
        return LIB
    exe = nvcc()

    def compile_unit(unit):
        name, src, defs = unit
        obj = os.path.join(BUILD, name + ".o")
        cmd = [exe] + FLAGS + extra + defs + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return name, obj, r

    with ThreadPoolExecutor(max_workers=jobs or min(len(UNITS), os.cpu_count() or 1)) as ex:
        results = list(ex.map(compile_unit, UNITS))
    failed = False
    for name, _, r in results:
        if verbose_ptxas or r.returncode != 0:
            sys.stderr.write(f"--- {name}\n{r.stdout}{r.stderr}")
        failed |= r.returncode != 0
    if failed:
        raise RuntimeError("nvcc failed (see output above)")
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [exe] + ARCH + ["-shared", "-Xlinker", "--no-undefined", "-o", tmp] + [obj for _, obj, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError("link of libtg.so failed")
    os.replace(tmp, LIB)
    with open(stamp, "w") as f:
        f.write(digest)
    return LIB


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose-ptxas", action="store_true", help="print registers / spills / smem per kernel")
    a = ap.parse_args()
    print(build(force=a.force, verbose_ptxas=a.verbose_ptxas))


if __name__ == "__main__":
    main()
