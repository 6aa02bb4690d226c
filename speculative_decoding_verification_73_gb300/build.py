"""Build libspecverify.so (the CUDA kernels and their C ABI) in place.

    python -m speculative_decoding_verification_73_gb300.build

Compiles every csrc/*.cu for sm_103a in parallel with nvcc, then links one
shared library next to this file.  The CUDA runtime is linked statically,
so the library only needs the CUDA driver at run time.
"""

import concurrent.futures
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libspecverify.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "--expt-relaxed-constexpr"]


def nvcc():
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libspecverify")
    return path


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _compile(src, verbose, build_dir=BUILD, defines=()):
    obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc(), *ARCH, *FLAGS, *[f"-D{d}" for d in defines], "-c", src, "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    proc = subprocess.run(cmd, capture_output=True, text=True)
    if proc.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{proc.stdout}\n{proc.stderr}")
    return obj, proc.stderr


def build(force=False, verbose=False, defines=(), out=LIB):
    """Compile and link; skip when the library is newer than every source.
    `defines` (NAME=VALUE strings) override the kernels' tuning constants;
    `out` names the library file (its objects go to a folder beside it)."""
    srcs = sources()
    heads = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cuh")]
    heads.append(os.path.join(os.path.dirname(PKG), "include", "spec_verify.h"))
    newest = max(os.path.getmtime(f) for f in srcs + heads)
    if not force and not defines and os.path.exists(out) and os.path.getmtime(out) >= newest:
        return out
    build_dir = BUILD if out == LIB else out + ".objs"
    os.makedirs(build_dir, exist_ok=True)
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        results = list(ex.map(lambda s: _compile(s, verbose, build_dir, defines), srcs))
    if verbose:
        for _, log in results:
            sys.stderr.write(log)
    tmp = out + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp] + [o for o, _ in results]
    proc = subprocess.run(cmd, capture_output=True, text=True)
    if proc.returncode != 0:
        raise RuntimeError(f"link failed:\n{proc.stdout}\n{proc.stderr}")
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIB)
