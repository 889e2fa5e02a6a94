"""Build the in-tree shared library libtq_gb300.so for sm_103a with nvcc.

Each translation unit compiles in parallel to an object file under
``_build/`` next to this file; the objects link into one shared library (static
CUDA runtime) beside the package sources.
"""

import concurrent.futures
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT = os.path.join(HERE, "libtq_gb300.so")
SOURCES = ["tq_host.cpp", "tq_store.cu", "tq_store_tc.cu", "tq_decode.cu", "tq_decode_noalloc.cu"] + [
    f"tq_decode_split_{d}_{kb}.cu" for d in (128, 256) for kb in (2, 3, 4)
] + ["tq_decode_split_128_3u.cu"] + [f"tq_extend_prefix_{k}.cu" for k in ("2", "3", "3u", "4u")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc():
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libtq_gb300.so")
    return path


def _flags():
    return ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O3", "-I", INCLUDE, "-I", CSRC] + ARCH


def _compile(src, obj, extra):
    cmd = [nvcc(), "-c", os.path.join(CSRC, src), "-o", obj] + _flags() + extra
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return r.stderr


def build(verbose=False, extra_flags=()):
    """Compile and link; returns the path of the shared library."""
    bdir = os.path.join(HERE, "_build")
    os.makedirs(bdir, exist_ok=True)
    objs = [os.path.join(bdir, os.path.splitext(s)[0] + ".o") for s in SOURCES]
    with concurrent.futures.ThreadPoolExecutor(len(SOURCES)) as ex:
        logs = list(ex.map(lambda so: _compile(so[0], so[1], list(extra_flags)), zip(SOURCES, objs)))
    tmp = OUT + ".tmp"
    cmd = [nvcc(), "-shared", "-o", tmp] + objs + ARCH + ["-lcudart_static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, OUT)
    if verbose:
        for log in logs:
            if log.strip():
                print(log)
    return OUT


if __name__ == "__main__":
    print(build(verbose=True))
