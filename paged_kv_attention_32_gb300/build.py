"""Build the C-ABI shared library ``libpka.so`` in-tree for sm_103a.

Every translation unit under ``csrc/`` is compiled in parallel with nvcc
(one ``-gencode arch=compute_103a,code=sm_103a``), then linked into
``paged_kv_attention_32_gb300/_lib/libpka.so``.  Object files go to
``_build/`` at the repository root.  Run ``python -m
paged_kv_attention_32_gb300.build`` (or ``__graft_entry__.build()``).
"""

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build", "pka")
LIB_DIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIB_DIR, "libpka.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-I", CSRC, "-I", INCLUDE]
CUDA_FLAGS = ARCH + ["-lineinfo", "--expt-relaxed-constexpr"]


def _nvcc():
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(home, "bin", "nvcc")
    return cand if os.path.exists(cand) else (shutil.which("nvcc") or "nvcc")


def _sources():
    return sorted(f for f in os.listdir(CSRC) if f.endswith((".cu", ".cpp")))


def _compile(src, verbose):
    obj = os.path.join(BUILD, src + ".o")
    cmd = [_nvcc()] + COMMON + (CUDA_FLAGS if src.endswith(".cu") else ["-x", "cu"] + ARCH)
    if verbose and src.endswith(".cu"):
        cmd += ["-Xptxas", "-v"]
    cmd += ["-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    return src, obj, r.returncode, r.stdout + r.stderr


def build(verbose=False):
    """Compile and link ``libpka.so``; return its path.  Raises on failure."""
    os.makedirs(BUILD, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)
    srcs = _sources()
    objs, errors = [], []
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        for src, obj, rc, log in ex.map(lambda s: _compile(s, verbose), srcs):
            if verbose and log.strip():
                print(f"--- {src}\n{log}", file=sys.stderr)
            if rc != 0:
                errors.append(f"--- {src} failed:\n{log}")
            objs.append(obj)
    if errors:
        raise RuntimeError("nvcc failed:\n" + "\n".join(errors))
    tmp = LIB + ".tmp"
    cmd = [_nvcc()] + ARCH + ["-shared", "-o", tmp] + objs + ["-lcudart_static", "-ldl", "-lrt", "-lpthread"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stdout + r.stderr)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
