"""Tiny PTX kernels used by the pins and parity tests.

op_kernel: every thread loads up to three operands from 8-byte slots of three
input buffers, runs one instruction, and stores its result to an 8-byte slot
of the output buffer. Used to check single-instruction semantics lane by lane.
"""
from __future__ import annotations

import numpy as np

from simt_ptx_interpretation_gb300 import workloads as wl

HEADER = wl.HEADER

# operand register per (position, width)
_REG32 = ["%r5", "%r6", "%r7"]
_REGF = ["%f1", "%f2", "%f3"]
_REG64 = ["%rd11", "%rd12", "%rd13"]
_ADDR = ["%rd7", "%rd8", "%rd9"]


def _reg(kind: str, i: int) -> str:
    return {"u": _REG32, "f": _REGF, "w": _REG64, "p": ["%p1", "%p2", "%p3"]}[kind][i]


def op_kernel(name: str, op: str, srcs: str, dst: str, imm: str | None = None) -> str:
    """srcs: operand kinds per source position: 'u' 32-bit int reg, 'f' f32 reg,
    'w' 64-bit reg, 'p' predicate (loaded as u32, true when nonzero), 'i' immediate.
    dst: 'u', 'f', 'w' or 'p' (a predicate result is stored as 0/1 u32)."""
    lines = [
        f".visible .entry {name}(",
        "    .param .u64 k_out, .param .u64 k_a, .param .u64 k_b, .param .u64 k_c",
        ")",
        "{",
        "    .reg .pred %p<5>;",
        "    .reg .b32 %r<12>;",
        "    .reg .f32 %f<6>;",
        "    .reg .b64 %rd<16>;",
        "    ld.param.u64 %rd1, [k_out];",
        "    ld.param.u64 %rd2, [k_a];",
        "    ld.param.u64 %rd3, [k_b];",
        "    ld.param.u64 %rd4, [k_c];",
        "    mov.u32 %r1, %ctaid.x;",
        "    mov.u32 %r2, %ntid.x;",
        "    mov.u32 %r3, %tid.x;",
        "    mad.lo.s32 %r4, %r1, %r2, %r3;",
        "    cvt.u64.u32 %rd5, %r4;",
        "    shl.b64 %rd6, %rd5, 3;",
        "    add.s64 %rd7, %rd2, %rd6;",
        "    add.s64 %rd8, %rd3, %rd6;",
        "    add.s64 %rd9, %rd4, %rd6;",
        "    add.s64 %rd10, %rd1, %rd6;",
    ]
    operands = []
    for i, k in enumerate(srcs):
        if k == "i":
            operands.append(imm)
        elif k == "u":
            lines.append(f"    ld.global.u32 {_REG32[i]}, [{_ADDR[i]}];")
            operands.append(_REG32[i])
        elif k == "f":
            lines.append(f"    ld.global.f32 {_REGF[i]}, [{_ADDR[i]}];")
            operands.append(_REGF[i])
        elif k == "w":
            lines.append(f"    ld.global.u64 {_REG64[i]}, [{_ADDR[i]}];")
            operands.append(_REG64[i])
        elif k == "p":
            lines.append(f"    ld.global.u32 %r{8 + i}, [{_ADDR[i]}];")
            lines.append(f"    setp.ne.u32 %p{1 + i}, %r{8 + i}, 0;")
            operands.append(f"%p{1 + i}")
        else:
            raise ValueError(k)
    d = {"u": "%r11", "f": "%f5", "w": "%rd14", "p": "%p4"}[dst]
    lines.append(f"    {op} {', '.join([d] + operands)};")
    if dst == "u":
        lines.append("    st.global.u32 [%rd10], %r11;")
    elif dst == "f":
        lines.append("    st.global.f32 [%rd10], %f5;")
    elif dst == "w":
        lines.append("    st.global.u64 [%rd10], %rd14;")
    else:
        lines.append("    selp.u32 %r11, 1, 0, %p4;")
        lines.append("    st.global.u32 [%rd10], %r11;")
    lines += ["    ret;", "}", ""]
    return HEADER + "\n".join(lines)


def op_workload(name: str, op: str, srcs: str, dst: str, a, b=None, c=None, imm=None,
                block: int = 256) -> wl.Workload:
    """Inputs a, b, c: uint64 arrays (one 8-byte slot per thread)."""
    n = len(a)
    assert n % block == 0
    z = np.zeros(n, dtype=np.uint64)
    arrs = [np.ascontiguousarray(np.asarray(x if x is not None else z, dtype=np.uint64)) for x in (a, b, c)]
    out = np.zeros(n, dtype=np.uint64)
    bufs = wl.place([("out", out, True), ("a", arrs[0], False), ("b", arrs[1], False), ("c", arrs[2], False)])
    params = wl.pack_params([("u64", x.sim_base) for x in bufs])
    return wl.Workload(name, op_kernel(name, op, srcs, dst, imm), name, n // block, block, params, bufs)


def straight_line(name: str, body: list[str], regs: str = "") -> str:
    """A kernel with no parameters: body lines, then ret."""
    decl = regs or "    .reg .pred %p<8>;\n    .reg .b32 %r<32>;\n    .reg .f32 %f<32>;\n    .reg .b64 %rd<16>;"
    return HEADER + f".visible .entry {name}()\n{{\n{decl}\n" + "\n".join("    " + x for x in body) + "\n    ret;\n}\n"
