"""Build libhsa.so (the C-ABI library) from csrc/*.cu for sm_103a, in-tree.

nvcc compiles each translation unit in parallel with
``-gencode arch=compute_103a,code=sm_103a`` and links them into
``full_attention_kv_gb300/_build/libhsa.so``.  No cmake, no torch extension
machinery: the library has a plain C ABI and no torch types.
"""
import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libhsa.so")
ROOT = os.path.dirname(HERE)

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr", "-I" + os.path.join(ROOT, "include")]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libhsa")
    return exe


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _headers():
    return sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) +
                  glob.glob(os.path.join(ROOT, "include", "*.h")))


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src, extra, out_dir=OUT_DIR):
    obj = os.path.join(out_dir, os.path.basename(src) + ".o")
    if not _stale(obj, [src] + _headers()):
        return obj, ""
    cmd = [nvcc()] + ARCH + NVCC_FLAGS + extra + ["-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, " ".join(cmd), r.stderr))
    return obj, r.stderr


def build(force: bool = False, verbose_ptxas: bool = False, out_dir: str = None,
          defines=()) -> str:
    """Compile and link the library; returns its path.

    out_dir / defines build a variant elsewhere (a test-only build with other
    compile-time settings, e.g. a short HSA_WAIT_NS); the product library is
    ``_build/libhsa.so`` with no extra defines."""
    out = OUT_DIR if out_dir is None else out_dir
    lib = os.path.join(out, "libhsa.so")
    os.makedirs(out, exist_ok=True)
    srcs = _sources()
    if force:
        for o in glob.glob(os.path.join(out, "*.o")):
            os.remove(o)
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    extra += ["-D" + d for d in defines]
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        results = list(ex.map(lambda s: _compile(s, extra, out), srcs))
    objs = [o for o, _ in results]
    if verbose_ptxas:
        for o, log in results:
            if log:
                sys.stderr.write(log)
    if force or _stale(lib, objs):
        tmp = lib + ".tmp%d" % os.getpid()
        # cudart is linked statically; the driver API (tensor-map encoding) is reached
        # through cudaGetDriverEntryPointByVersion, so libcuda is not a link dependency
        cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n%s\n%s" % (" ".join(cmd), r.stderr))
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
