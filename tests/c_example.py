"""Builds tests/c_abi_forward.c, a C program that calls the library through
include/gbmoe.h alone, against the in-tree libgbmoe.so and the CUDA runtime."""
from __future__ import annotations

import glob
import os
import shutil
import subprocess

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_abi_forward.c")


def cuda_home() -> str:
    return os.environ.get("CUDA_HOME", "/usr/local/cuda")


def cudart_dir() -> str | None:
    home = cuda_home()
    for d in [os.path.join(home, "lib64")] + sorted(glob.glob(os.path.join(home, "targets", "*", "lib"))):
        if os.path.exists(os.path.join(d, "libcudart.so")):
            return d
    return None


def build(out_dir: str) -> str:
    """Compile and link the example into out_dir; return the executable's path.
    Raises RuntimeError (with the compiler's output) when it does not build."""
    import mixture_experts_layer_count_gb300 as g
    cc = shutil.which("gcc")
    rt = cudart_dir()
    if cc is None or rt is None:
        raise FileNotFoundError("gcc or libcudart.so not found")
    g.load()  # builds libgbmoe.so if it is missing or stale
    libdir = os.path.dirname(g.lib_path())
    exe = os.path.join(out_dir, "c_abi_forward")
    cmd = [cc, "-std=c99", "-O1", "-Wall", "-Wextra", "-Werror",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda_home(), "include"),
           SRC, "-o", exe, "-L", libdir, "-L", rt, "-lgbmoe", "-lcudart", "-lm",
           f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{rt}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(" ".join(cmd) + "\n" + r.stdout + r.stderr)
    return exe
