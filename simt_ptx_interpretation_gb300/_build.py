"""Builds libks.so in-tree: the sm_103a interpreter (nvcc) and the host
decoder / C ABI (g++), compiled in parallel and linked with nvcc."""
from __future__ import annotations

import os
import shutil
import subprocess
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libks.so")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"
_lock = threading.Lock()


def _cuda_home() -> str:
    home = os.environ.get("CUDA_HOME") or "/usr/local/cuda"
    if not os.path.exists(os.path.join(home, "bin", "nvcc")):
        nvcc = shutil.which("nvcc")
        if nvcc:
            home = os.path.dirname(os.path.dirname(nvcc))
    return home


def _sources():
    return [os.path.join(CSRC, f) for f in sorted(os.listdir(CSRC)) if f.endswith((".cu", ".cuh", ".cpp", ".h"))] + [
        os.path.join(os.path.dirname(PKG), "include", "ks.h")]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(s) <= t for s in _sources())


def build_native(force: bool = False, verbose: bool = False) -> str:
    with _lock:
        if not force and up_to_date():
            return LIB
        os.makedirs(BUILD, exist_ok=True)
        home = _cuda_home()
        nvcc = os.path.join(home, "bin", "nvcc")
        inc = os.path.join(home, "include")
        jobs = []
        objs = []
        for f in sorted(os.listdir(CSRC)):
            src = os.path.join(CSRC, f)
            obj = os.path.join(BUILD, f + ".o")
            if f.endswith(".cu"):
                cmd = [nvcc, ARCH, "-lineinfo", "-O3", "-std=c++17", "--fmad=false", "-Xcompiler", "-fPIC",
                       "-Xptxas", "-v", "-c", src, "-o", obj]
            elif f.endswith(".cpp"):
                cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-Wall", f"-I{inc}", "-c", src, "-o", obj]
            else:
                continue
            objs.append(obj)
            jobs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
        failed = []
        for cmd, p in jobs:
            out, _ = p.communicate()
            if verbose or p.returncode:
                print(" ".join(cmd))
                print(out)
            if p.returncode:
                failed.append(cmd[-3])
        if failed:
            raise RuntimeError(f"libks build failed: {failed}")
        tmp = LIB + f".tmp{os.getpid()}"
        link = [nvcc, ARCH, "-shared", "-o", tmp] + objs + ["-lpthread"]
        r = subprocess.run(link, capture_output=True, text=True)
        if r.returncode:
            raise RuntimeError("libks link failed:\n" + r.stdout + r.stderr)
        os.replace(tmp, LIB)
        return LIB
