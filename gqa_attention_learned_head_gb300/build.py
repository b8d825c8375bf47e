"""Builds libsinkattn.so in-tree for sm_103a with nvcc (no cmake, no torch extension).

    python -m gqa_attention_learned_head_gb300.build [--force]

Each .cu file compiles in its own nvcc process (in parallel); the objects are
linked into ``gqa_attention_learned_head_gb300/_build/libsinkattn.so``.  A
rebuild happens only when a source or header is newer than the library.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
INCLUDE = ROOT / "include"
BUILD = PKG / "_build"
LIB = BUILD / "libsinkattn.so"

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-I", str(INCLUDE), "-I", str(CSRC)]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and Path(cand).exists():
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libsinkattn")


def sources():
    return sorted(CSRC.glob("*.cu"))


def _stale() -> bool:
    if not LIB.exists():
        return True
    t = LIB.stat().st_mtime
    deps = list(CSRC.glob("*")) + list(INCLUDE.glob("*.h")) + [Path(__file__)]
    return any(p.stat().st_mtime > t for p in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> Path:
    if not force and not _stale():
        return LIB
    nvcc = nvcc_path()
    BUILD.mkdir(exist_ok=True)
    srcs = sources()

    def compile_one(src: Path) -> Path:
        obj = BUILD / (src.stem + ".o")
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *extra_flags, "-c", str(src), "-o", str(obj)]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src.name}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, file=sys.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = LIB.with_suffix(f".{os.getpid()}.tmp")
    cmd = [nvcc, *ARCH, "-shared", "-Xcompiler", "-fPIC", *map(str, objs), "-o", str(tmp)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


# Host code with the most validation logic: the C ABI layer and the no-allocation entry point.
SANITIZED_SOURCES = ("api.cu", "decode_noalloc.cu")
SAN_BUILD = PKG / "_build_san"
SAN_LIB = SAN_BUILD / "libsinkattn.so"
SAN_FLAGS = ["-Xcompiler", "-fsanitize=address", "-Xcompiler", "-fsanitize=undefined", "-Xcompiler", "-fno-omit-frame-pointer",
             "-Xcompiler", "-fno-sanitize-recover=undefined"]


def build_sanitized() -> Path:
    """A copy of the library whose host code in SANITIZED_SOURCES is compiled with AddressSanitizer
    and UndefinedBehaviorSanitizer (the other objects are the regular ones), for tests of the host
    validation paths.  A process loading it must load the ASan runtime first (LD_PRELOAD)."""
    build()
    nvcc = nvcc_path()
    SAN_BUILD.mkdir(exist_ok=True)
    objs = [str(BUILD / (src.stem + ".o")) for src in sources() if src.name not in SANITIZED_SOURCES]
    for name in SANITIZED_SOURCES:
        obj = SAN_BUILD / (Path(name).stem + ".o")
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *SAN_FLAGS, "-c", str(CSRC / name), "-o", str(obj)]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {name}:\n{r.stdout}\n{r.stderr}")
        objs.append(str(obj))
    cmd = [nvcc, *ARCH, "-shared", "-Xcompiler", "-fPIC", *SAN_FLAGS, *objs, "-o", str(SAN_LIB)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    return SAN_LIB


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--ptxas-info", action="store_true", help="print register / shared memory use")
    ap.add_argument("--sanitize", action="store_true",
                    help="also build _build_san/libsinkattn.so, its host validation code under ASan + UBSan")
    args = ap.parse_args()
    if args.sanitize:
        print(build_sanitized())
    extra = ["-Xptxas", "-v"] if args.ptxas_info else []
    print(build(force=args.force or args.ptxas_info, verbose=args.verbose or args.ptxas_info, extra_flags=extra))
