"""Build the seeded input generator libraries in-tree.

``libppsynth_host.so`` (gcc, OpenMP) fills host arrays; ``libppsynth_dev.so`` (nvcc,
sm_103a) fills device arrays with the same bits.  Both are test and bench
infrastructure; the tick itself never loads them.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
HOST_SO = os.path.join(HERE, "libppsynth_host.so")
DEV_SO = os.path.join(HERE, "libppsynth_dev.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(os.path.join(HERE, d)) > t for d in deps)


def host_cmd():
    return ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
            os.path.join(HERE, "synth.c"), "-o", HOST_SO, "-lm"]


def dev_cmd():
    return [NVCC, "-O3", "-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo",
            "-Xcompiler", "-fPIC", "-shared", os.path.join(HERE, "synth.cu"), "-o", DEV_SO]


def build(host=True, device=True, force=False):
    """Compile what is missing or stale; returns the list of Popen objects waited on."""
    procs = []
    if host and (force or _stale(HOST_SO, ["synth.c", "synth.h", "synth_core.h"])):
        procs.append(subprocess.Popen(host_cmd()))
    if device and (force or _stale(DEV_SO, ["synth.cu", "synth.h", "synth_core.h"])):
        procs.append(subprocess.Popen(dev_cmd()))
    for p in procs:
        if p.wait() != 0:
            raise RuntimeError("synth build failed: %s" % " ".join(p.args))
    return procs


if __name__ == "__main__":
    build(force=True)
