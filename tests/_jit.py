"""Runs a PTX kernel natively through the CUDA driver's JIT (cuModuleLoadData
and cuLaunchKernel via ctypes), as an implementation of the PTX semantics that
is independent of both the interpreter and the oracle."""
from __future__ import annotations

import ctypes
import struct

import torch

_cuda = None


def _lib():
    global _cuda
    if _cuda is None:
        _cuda = ctypes.CDLL("libcuda.so.1")
    return _cuda


def _ck(rc, what):
    if rc != 0:
        name = ctypes.c_char_p()
        _lib().cuGetErrorName(rc, ctypes.byref(name))
        raise RuntimeError(f"{what} failed: {rc} {name.value}")


def run_native(ptx: str, kernel: str, grid: int, block: int, param_layout, param_values, stream=None):
    """param_layout: [(offset, size)]; param_values: ints in declaration order."""
    cu = _lib()
    torch.cuda.init()
    torch.cuda.synchronize()
    _ck(cu.cuInit(0), "cuInit")
    mod = ctypes.c_void_p()
    log = ctypes.create_string_buffer(8192)
    # options: CU_JIT_ERROR_LOG_BUFFER (5), CU_JIT_ERROR_LOG_BUFFER_SIZE_BYTES (6)
    opts = (ctypes.c_int * 2)(5, 6)
    vals = (ctypes.c_void_p * 2)(ctypes.cast(log, ctypes.c_void_p), ctypes.c_void_p(len(log)))
    rc = cu.cuModuleLoadDataEx(ctypes.byref(mod), ptx.encode() + b"\0", 2, opts, vals)
    if rc != 0:
        raise RuntimeError(f"JIT failed ({rc}): {log.value.decode(errors='replace')}")
    try:
        fn = ctypes.c_void_p()
        _ck(cu.cuModuleGetFunction(ctypes.byref(fn), mod, kernel.encode()), "cuModuleGetFunction")
        holders = []
        for (off, size), v in zip(param_layout, param_values):
            holders.append(ctypes.c_uint64(v) if size == 8 else ctypes.c_uint32(v & 0xFFFFFFFF))
        args = (ctypes.c_void_p * max(1, len(holders)))(*[ctypes.cast(ctypes.byref(h), ctypes.c_void_p) for h in holders])
        s = stream.cuda_stream if stream is not None else torch.cuda.current_stream().cuda_stream
        _ck(cu.cuLaunchKernel(fn, grid, 1, 1, block, 1, 1, 0, ctypes.c_void_p(s), args, None), "cuLaunchKernel")
        torch.cuda.synchronize()
    finally:
        cu.cuModuleUnload(mod)


def unpack_params(blob: bytes, layout):
    vals = []
    for off, size in layout:
        vals.append(struct.unpack_from("<Q" if size == 8 else "<I", blob, off)[0])
    return vals
