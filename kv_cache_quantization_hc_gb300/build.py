"""Build libhc.so (the C-ABI library) in-tree with nvcc for sm_103a.

The translation units compile in parallel; the link uses nvcc's default
static CUDA runtime, so the library depends on no libcudart at load time.
A stamp of the sources' hash and the flags skips rebuilding an up-to-date
library built for this machine's architecture.
"""
import fcntl
import hashlib
import os
import platform
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libhc.so")

SOURCES = ["api.cu", "encode.cu", "encode_rows.cu", "fetch_fp8.cu", "fetch_fp8_rows.cu",
           "fetch_int4.cu", "fetch_raw.cu", "table.cu", "crc32.cu", "select.cu",
           "hash.cpp"]


def _headers():
    """Every header the translation units may include: all of csrc/'s, and hc.h."""
    hs = sorted(f for f in os.listdir(CSRC) if f.endswith((".h", ".cuh")))
    return [os.path.join(CSRC, h) for h in hs] + [os.path.join(INCLUDE, "hc.h")]


ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE]

_ELF_MACHINE = {"x86_64": 62, "aarch64": 183, "arm64": 183}


def _nvcc():
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libhc.so")


def _stamp(extra_flags):
    h = hashlib.sha256()
    for p in [os.path.join(CSRC, s) for s in SOURCES] + _headers():
        with open(p, "rb") as f:
            h.update(p.encode() + b"\0" + f.read())
    h.update(" ".join(FLAGS + list(extra_flags)).encode())
    h.update(platform.machine().encode())
    return h.hexdigest()


def _lib_matches_host(path):
    """True if the ELF at path was built for this machine's architecture."""
    try:
        with open(path, "rb") as f:
            hdr = f.read(20)
    except OSError:
        return False
    if len(hdr) < 20 or hdr[:4] != b"\x7fELF":
        return False
    machine = int.from_bytes(hdr[18:20], "little")
    return machine == _ELF_MACHINE.get(platform.machine(), -1)


def build(force=False, verbose=False, extra_flags=(), out_dir=None):
    """Compile and link libhc.so; returns its path.  ``out_dir`` places the
    objects and the library elsewhere (a variant built with extra flags).
    Concurrent callers (the ranks of a torchrun job) take turns on a lock
    file in the build directory: the first builds, the others then find the
    stamp up to date."""
    build_dir = BUILD if out_dir is None else out_dir
    os.makedirs(build_dir, exist_ok=True)
    with open(os.path.join(build_dir, "lock"), "w") as lock:
        fcntl.flock(lock, fcntl.LOCK_EX)
        try:
            return _build_locked(build_dir, force, verbose, extra_flags, out_dir)
        finally:
            fcntl.flock(lock, fcntl.LOCK_UN)


def _build_locked(build_dir, force, verbose, extra_flags, out_dir):
    lib = LIB if out_dir is None else os.path.join(out_dir, "libhc.so")
    stamp = _stamp(extra_flags)
    stamp_path = os.path.join(build_dir, "stamp")
    if not force and _lib_matches_host(lib) and os.path.exists(stamp_path):
        with open(stamp_path) as f:
            if f.read().strip() == stamp:
                return lib
    nvcc = _nvcc()

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc, *FLAGS, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    with open(stamp_path, "w") as f:
        f.write(stamp)
    return lib


if __name__ == "__main__":
    print(build(force=True, verbose=True))
