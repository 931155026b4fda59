"""Build the aggregation library libfedavg.so for sm_103a with nvcc.

Translation units compile in parallel; the result lands in
server_side_fedavg_gb300/_build/ (git-ignored).  cudart is linked as a shared
library so that a process that already loaded torch's libcudart.so.13 shares
one runtime with this library."""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
SO = os.path.join(BUILD, "libfedavg.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["accumulate.cu", "reduce.cu", "gather.cu", "finalize.cu", "noalloc.cu", "fedavg.cpp",
           "ledger.cpp", "partition.cpp", "gather_plan.cpp"]


def _common():
    return ["-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "include"),
            "-I", CSRC]


def compile_commands(extra=None):
    os.makedirs(BUILD, exist_ok=True)
    cmds = []
    for src in SOURCES:
        obj = os.path.join(BUILD, src.rsplit(".", 1)[0] + ".o")
        cmd = [NVCC] + _common() + (extra or [])
        if src.endswith(".cu"):
            cmd += ARCH + ["-lineinfo", "-Xptxas", "-v"]
        else:
            cmd += ["-x", "c++", "-Xcompiler", "-ffp-contract=off"]
        cmd += ["-c", os.path.join(CSRC, src), "-o", obj]
        cmds.append((obj, cmd))
    return cmds


def cmd_is_cuda(cmd):
    """True for the compile command of a CUDA source (its ptxas -v report is kept)."""
    return any(str(a).endswith(".cu") for a in cmd)


def link_command(objs):
    return [NVCC, "-shared"] + ARCH + objs + ["-cudart", "shared",
                                              "-Xlinker", "-rpath,/usr/local/cuda/lib64",
                                              "-o", SO]


def build(verbose: bool = False) -> str:
    procs = []
    for obj, cmd in compile_commands():
        procs.append((obj, cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    objs, ptxas = [], []
    for obj, cmd, p in procs:
        log = p.communicate()[0].decode(errors="replace")
        if p.returncode != 0:
            raise RuntimeError(f"build failed: {' '.join(cmd)}\n{log}")
        if verbose and log.strip():
            print(log)
        if cmd_is_cuda(cmd):
            ptxas.append(log)
        objs.append(obj)
    with open(os.path.join(BUILD, "ptxas.txt"), "w") as f:
        f.write("".join(ptxas))
    r = subprocess.run(link_command(objs), stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stdout.decode(errors="replace"))
    return SO


if __name__ == "__main__":
    print(build(verbose=True))
