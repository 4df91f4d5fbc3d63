"""Hand-written kernels for the L1/L2 hit model (KernelScope backend doc,
simulator/engine.py — "Cache parameters", SimpleCache, _execute_instruction;
the access order follows the page's step()). Shared by the oracle pins and
the GPU parity tests; PTX text and inputs only."""
from __future__ import annotations

import numpy as np

from simt_ptx_interpretation_gb300 import workloads as wl

BASE_IN = 0x1000_0000
BASE_OUT = 0x4000_0000


def _kernel(name: str, params: str, body: str) -> str:
    return wl.HEADER + f""".visible .entry {name}({params})
{{
    .reg .pred %p<4>;
    .reg .b32 %r<8>;
    .reg .f32 %f<8>;
    .reg .b64 %rd<8>;
{body}
}}
"""


# One warp loads one word twice (the second load depends on nothing new),
# each load feeding an add, then stores the sum: DRAM, then an L1 hit.
REUSE = _kernel("reuse", ".param .u64 p_in, .param .u64 p_out", """
    ld.param.u64    %rd1, [p_in];
    ld.param.u64    %rd2, [p_out];
    ld.global.f32   %f1, [%rd1];
    add.f32         %f2, %f1, %f1;
    ld.global.f32   %f3, [%rd1];
    add.f32         %f2, %f3, %f2;
    st.global.f32   [%rd2], %f2;
    ret;""")

# Loads at in, in + off, in, in + off (four independent loads).
PAIR = _kernel("pair", ".param .u64 p_in, .param .u64 p_off", """
    ld.param.u64    %rd1, [p_in];
    ld.param.u64    %rd2, [p_off];
    add.s64         %rd3, %rd1, %rd2;
    ld.global.f32   %f1, [%rd1];
    ld.global.f32   %f2, [%rd3];
    ld.global.f32   %f3, [%rd1];
    ld.global.f32   %f4, [%rd3];
    ret;""")


def order_kernel(delay_warp0: int, delay_warp1: int) -> str:
    """Two warps of one CTA load the same word; warp w first runs delay_w extra
    adds, so warp 0 loads at step 6 + delay_0 and warp 1 at 6 + delay_1."""
    a = "\n".join("    add.u32         %r2, %r2, 1;" for _ in range(delay_warp0))
    b = "\n".join("    add.u32         %r2, %r2, 1;" for _ in range(delay_warp1))
    return _kernel("order", ".param .u64 p_in", f"""
    mov.u32         %r1, %tid.x;
    mov.u32         %r2, 0;
    setp.ge.u32     %p1, %r1, 32;
    @%p1 bra        W1;
{a}
    bra.uni         LOAD;
W1:
{b}
    bra.uni         LOAD;
LOAD:
    ld.param.u64    %rd1, [p_in];
    ld.global.f32   %f1, [%rd1];
    ret;""")


# Each lane addresses its own line (in + 128 * tid); the first load skips
# lane 0, so its representative is lane 1's line; the second load is lane
# 0's address + 128 in every lane, the line lane 1 brought in: an L1 hit.
REPRESENTATIVE = _kernel("rep", ".param .u64 p_in", """
    ld.param.u64    %rd1, [p_in];
    mov.u32         %r1, %tid.x;
    cvt.u64.u32     %rd2, %r1;
    shl.b64         %rd2, %rd2, 7;
    add.s64         %rd3, %rd1, %rd2;
    setp.ne.u32     %p1, %r1, 0;
    @%p1 ld.global.f32 %f1, [%rd3];
    ld.global.f32   %f2, [%rd1+128];
    ret;""")

# A store installs its line: the load of the same word that follows hits L1.
STORE_THEN_LOAD = _kernel("stld", ".param .u64 p_out", """
    ld.param.u64    %rd1, [p_out];
    mov.u32         %r1, 7;
    st.global.u32   [%rd1], %r1;
    ld.global.u32   %r2, [%rd1+4];
    st.global.u32   [%rd1+8], %r2;
    ret;""")

# Warp 0 runs three adds before bar.sync (arrives at step 6), warp 1 arrives
# at step 3; both resume at step 7 and load the same word at step 8.
BARRIER = _kernel("barrier", ".param .u64 p_in", """
    mov.u32         %r1, %tid.x;
    setp.lt.u32     %p1, %r1, 32;
    @!%p1 bra       BAR;
    add.u32         %r2, %r1, 1;
    add.u32         %r2, %r2, 1;
    add.u32         %r2, %r2, 1;
BAR:
    bar.sync        0;
    ld.param.u64    %rd1, [p_in];
    ld.global.f32   %f1, [%rd1];
    ret;""")

# Warp 1 never reaches the barrier: five adds then ret (its last instruction
# at step 8); warp 0 waits from step 3 and resumes at step 9, loading at 10.
BARRIER_EXIT = _kernel("barrier_exit", ".param .u64 p_in", """
    mov.u32         %r1, %tid.x;
    setp.lt.u32     %p1, %r1, 32;
    @%p1 bra        W0;
    add.u32         %r2, %r1, 1;
    add.u32         %r2, %r2, 1;
    add.u32         %r2, %r2, 1;
    add.u32         %r2, %r2, 1;
    add.u32         %r2, %r2, 1;
    ret;
W0:
    bar.sync        0;
    ld.param.u64    %rd1, [p_in];
    ld.global.f32   %f1, [%rd1];
    ret;""")

# Two accesses per thread (cap tests) and a control flow that reads back
# what the thread stored (the first pass, which stores nothing, takes the
# other path and makes one more access).
READ_BACK = _kernel("read_back", ".param .u64 p_in, .param .u64 p_out", """
    ld.param.u64    %rd1, [p_in];
    ld.param.u64    %rd2, [p_out];
    mov.u32         %r1, %tid.x;
    cvt.u64.u32     %rd3, %r1;
    shl.b64         %rd3, %rd3, 2;
    add.s64         %rd4, %rd2, %rd3;
    mov.u32         %r2, 1;
    st.global.u32   [%rd4], %r2;
    ld.global.u32   %r3, [%rd4];
    setp.eq.u32     %p1, %r3, 1;
    @%p1 bra        DONE;
    ld.global.u32   %r4, [%rd1];
DONE:
    ret;""")


def f32_buffer(n_words: int, seed: int = 11) -> np.ndarray:
    return wl.uniform_f32(n_words, -1.0, 1.0, seed)


def u64(*vals) -> bytes:
    return b"".join(int(v).to_bytes(8, "little") for v in vals)
