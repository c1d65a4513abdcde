"""Build ``libpp.so`` (the tick's kernels + C ABI) in-tree for sm_103a with nvcc.

Each ``csrc/*.cu`` (and host-only ``csrc/*.cpp``) compiles to an object in parallel; the objects link into one shared
library next to this file.  The CUDA runtime is linked statically.
"""
import concurrent.futures
import glob
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
OBJ = os.path.join(HERE, "_build")
SO = os.path.join(HERE, "libpp.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xptxas", "-v"]


def _sources():
    # kernels (.cu) and host-only runtime code (.cpp), both through nvcc
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + [os.path.join(INCLUDE, "pp.h")]


def stale():
    if not os.path.exists(SO):
        return True
    t = os.path.getmtime(SO)
    return any(os.path.getmtime(p) > t for p in _deps())


def _compile(src, log):
    obj = os.path.join(OBJ, os.path.splitext(os.path.basename(src))[0] + ".o")
    cmd = [NVCC] + ARCH + FLAGS + ["-I", INCLUDE, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    log.append((src, r.stdout + r.stderr))
    if r.returncode != 0:
        raise RuntimeError("nvcc failed on %s:\n%s" % (src, r.stdout + r.stderr))
    return obj


def build(force=False, verbose=False):
    if not force and not stale():
        return SO
    os.makedirs(OBJ, exist_ok=True)
    log = []
    with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, os.cpu_count() or 1)) as ex:
        objs = list(ex.map(lambda s: _compile(s, log), _sources()))
    tmp = SO + ".tmp"
    subprocess.check_call([NVCC] + ARCH + ["-shared", "-o", tmp] + objs)
    os.replace(tmp, SO)
    if verbose:
        for src, text in log:
            print("==", os.path.basename(src))
            print(text)
    return SO


if __name__ == "__main__":
    build(force=True, verbose=True)
