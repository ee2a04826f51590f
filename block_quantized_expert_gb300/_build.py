"""Build libmoe.so in-tree with nvcc for sm_103a (used by build() and the binding)."""
from __future__ import annotations

import os
import subprocess
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

PKG = Path(__file__).resolve().parent
CSRC = PKG / "csrc"
OUT_DIR = PKG / "_build"
LIB = OUT_DIR / "libmoe.so"
PEAKS_SRC = PKG / "peaks" / "peaks.cu"
PEAKS_LIB = OUT_DIR / "libmoe_peaks.so"
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "--expt-relaxed-constexpr"]


def sources():
    return sorted(CSRC.glob("*.cu"))


def _stale() -> bool:
    if not LIB.exists():
        return True
    t = LIB.stat().st_mtime
    deps = list(CSRC.glob("*")) + [PKG.parent / "include" / "moe.h", Path(__file__)]
    return any(p.stat().st_mtime > t for p in deps)


def build(force: bool = False, verbose: bool = False) -> Path:
    """Compile every .cu under csrc/ (in parallel) and link libmoe.so."""
    if not force and not _stale():
        return LIB
    OUT_DIR.mkdir(parents=True, exist_ok=True)
    srcs = sources()
    objs = [OUT_DIR / (s.stem + ".o") for s in srcs]

    def compile_one(pair):
        src, obj = pair
        cmd = [NVCC, *ARCH, *FLAGS, "-c", str(src), "-o", str(obj)]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src.name}:\n{r.stderr}")
        return r.stderr

    with ThreadPoolExecutor(max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        logs = list(ex.map(compile_one, zip(srcs, objs)))
    tmp = LIB.with_suffix(f".{os.getpid()}.tmp")
    r = subprocess.run([NVCC, *ARCH, "-shared", "-o", str(tmp), *map(str, objs)],
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, LIB)
    if verbose:
        print("".join(logs))
    return LIB


def build_peaks(force: bool = False) -> Path:
    """Compile the roofline-denominator microbenchmarks into libmoe_peaks.so."""
    deps = [PEAKS_SRC, CSRC / "tc_ptx.cuh", Path(__file__)]
    if not force and PEAKS_LIB.exists() and all(p.stat().st_mtime <= PEAKS_LIB.stat().st_mtime for p in deps):
        return PEAKS_LIB
    OUT_DIR.mkdir(parents=True, exist_ok=True)
    tmp = PEAKS_LIB.with_suffix(f".{os.getpid()}.tmp")
    r = subprocess.run([NVCC, *ARCH, *FLAGS, "-shared", "-o", str(tmp), str(PEAKS_SRC)],
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {PEAKS_SRC.name}:\n{r.stderr}")
    os.replace(tmp, PEAKS_LIB)
    return PEAKS_LIB


if __name__ == "__main__":
    import sys
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    build_peaks(force="--force" in sys.argv)
    print(LIB)
