"""Build libwq.so from csrc/*.cu for sm_103a with nvcc (in-tree, no cmake).

Each translation unit compiles in parallel; the link step makes the shared
library next to this file.  Float contraction is disabled (-fmad=false) and
no fast-math flag is used: the kernels' float arithmetic is IEEE round to
nearest, operation by operation.

Reuse of earlier objects is keyed on content, not on file times: every
object and the library carry a stamp, the SHA-256 of the sources and headers
they depend on, the compiler flags, the nvcc version and the host machine.
A tree copied to another machine (whose files keep or lose their times) is
therefore always rebuilt from its own sources, and a stale object can never
be linked."""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import platform
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libwq.so")
LIB_STAMP = os.path.join(BUILD, "libwq.so.stamp")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVFLAGS = ["-O3", "-std=c++17", "-lineinfo", "-fmad=false", "-Xcompiler", "-fPIC",
           "-Xcompiler", "-fvisibility=hidden", "--expt-relaxed-constexpr", "-I", INCLUDE]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libwq.so")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def headers():
    hdrs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hdrs += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return sorted(hdrs)


def _nvcc_version(exe: str) -> str:
    r = subprocess.run([exe, "--version"], capture_output=True, text=True)
    return r.stdout.strip()


def _digest(paths, extra: str) -> str:
    h = hashlib.sha256(extra.encode())
    for p in paths:
        h.update(os.path.basename(p).encode())
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def _stamp_ok(stamp_path: str, target: str, digest: str) -> bool:
    if not (os.path.exists(target) and os.path.exists(stamp_path)):
        return False
    with open(stamp_path) as f:
        return f.read().strip() == digest


def _write_stamp(stamp_path: str, digest: str) -> None:
    with open(stamp_path, "w") as f:
        f.write(digest + "\n")


def _compile(src: str, key: str, extra) -> tuple:
    """Compile one translation unit unless its stamped object matches `key`
    (sources, headers, flags, toolchain).  Returns (object, compiled?)."""
    obj = os.path.join(BUILD, os.path.basename(src) + ".o")
    stamp = obj + ".stamp"
    digest = _digest([src], key + "|" + " ".join(extra))
    if _stamp_ok(stamp, obj, digest):
        return obj, False
    cmd = [nvcc(), *ARCH, *NVFLAGS, *extra, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    _write_stamp(stamp, digest)
    return obj, True


def build(verbose: bool = False, extra=()) -> str:
    """Compile every translation unit whose content stamp is stale, link
    libwq.so when any object changed, and return the library's path."""
    os.makedirs(BUILD, exist_ok=True)
    exe = nvcc()
    srcs = sources()
    # the common key: every header, the flags, the compiler and the machine
    key = _digest(headers(), "|".join([*ARCH, *NVFLAGS, _nvcc_version(exe), platform.machine()]))
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        res = list(ex.map(lambda s: _compile(s, key, list(extra)), srcs))
    objs = [o for o, _ in res]
    compiled = sum(1 for _, c in res if c)
    lib_digest = _digest(objs, "link|" + " ".join(ARCH))
    if not _stamp_ok(LIB_STAMP, LIB, lib_digest):
        cmd = [exe, *ARCH, "-shared", "-o", LIB, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        _write_stamp(LIB_STAMP, lib_digest)
        linked = True
    else:
        linked = False
    if verbose:
        print(f"built {LIB} ({compiled} of {len(srcs)} units compiled, "
              f"{'linked' if linked else 'link up to date'}, {platform.machine()})", file=sys.stderr)
    return LIB


if __name__ == "__main__":
    build(verbose=True)
