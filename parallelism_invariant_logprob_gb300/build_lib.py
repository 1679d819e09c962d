"""Build step for the CUDA library: compiles ``csrc/*.cu`` and ``csrc/*.cpp``
for sm_103a with nvcc (translation units in parallel) and links
``libiso.so`` in-tree beside this file.  No CMake, no torch extension
machinery: the library is plain C ABI.

``build(debug=True)`` builds ``libiso_debug.so`` from the same sources with
``-DISO_DEBUG``: the same entry points, with device-side bounds checks that
record ISO_ERR_DEVICE_CHECK in the status word and skip the access instead of
trapping (a stand-in for a memory checker)."""
from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "csrc")
_OBJ = os.path.join(_HERE, "_build")
_OBJ_DEBUG = os.path.join(_HERE, "_build_debug")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def library_path(debug: bool = False) -> str:
    return os.path.join(_HERE, "libiso_debug.so" if debug else "libiso.so")


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _sources():
    return sorted(f for f in os.listdir(_SRC) if f.endswith((".cu", ".cpp")))


def _headers_mtime() -> float:
    hs = [os.path.join(_SRC, f) for f in os.listdir(_SRC) if f.endswith((".h", ".cuh"))]
    hs.append(os.path.join(os.path.dirname(_HERE), "include", "iso.h"))
    return max(os.path.getmtime(h) for h in hs)


def _compile(src: str, verbose: bool, debug: bool = False) -> str:
    obj = os.path.join(_OBJ_DEBUG if debug else _OBJ, src + ".o")
    defs = ["-DISO_DEBUG"] if debug else []
    cmd = [_nvcc(), ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
           "--expt-relaxed-constexpr", "-Xptxas", "-v" if verbose else "-O3"] + defs + ["-c",
                                                                                       os.path.join(_SRC, src), "-o", obj]
    if src.endswith(".cpp"):
        cmd = [_nvcc(), "-O2", "-std=c++17", "-Xcompiler", "-fPIC", "-x", "cu"] + defs + [
            "-c", os.path.join(_SRC, src), "-o", obj, ARCH]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    if verbose and (r.stdout or r.stderr):
        print(r.stdout + r.stderr)
    return obj


def build(verbose: bool = False, force: bool = False, debug: bool = False) -> str:
    out = library_path(debug)
    srcs = _sources()
    newest = max([os.path.getmtime(os.path.join(_SRC, s)) for s in srcs] + [_headers_mtime()])
    if not force and os.path.exists(out) and os.path.getmtime(out) >= newest:
        return out
    os.makedirs(_OBJ_DEBUG if debug else _OBJ, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose, debug), srcs))
    tmp = out + f".tmp{os.getpid()}"
    cmd = [_nvcc(), ARCH, "-shared", "-o", tmp] + objs + ["-lcudart_static", "-ldl", "-lpthread", "-lrt"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    import sys
    print(build(verbose="-v" in sys.argv, force=True))
