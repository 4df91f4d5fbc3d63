"""Seeded synthetic workloads: PTX program text, launch shapes and input buffers.

This module is shared by the GPU path's tests and bench and by the oracle
checks. It holds none of the interpreter's arithmetic: it writes programs and
draws inputs, and never executes or predicts anything.

Workloads (sizes as the simulator's headline configurations state them):
  * vector_add  — KernelScope backend doc, "PTX Parser" example kernel:
    params u64 a, b, c and u32 n; index ctaid*ntid+tid by mad.lo.s32;
    setp.ge.s32 bounds check then @p bra to the exit; two ld.global.f32,
    add.f32, st.global.f32, ret. Written here from that description.
  * ffma        — SASS 프로브 방법론 §4 / §14: 4096 outer iterations around 32
    fma.rn.f32, loop overhead add/setp/bra; 1 accumulator (dependent) or k
    rotating accumulators (independent).
  * gather      — out[i] = in[i*s] in f32 (coalescing study of the KernelScope
    page's "global memory coalescing" section, swept over the stride).
  * divergent   — data-dependent trip count per thread with a lane-dependent
    branch inside the loop body.
  * fuzz        — random structured programs over the whole supported subset.

Inputs are drawn with torch's CPU generator, U[lo, hi) = lo + (hi - lo) * rand.
"""
from __future__ import annotations

import random
import struct
from dataclasses import dataclass, field

import numpy as np
import torch

SIM_BASE0 = 0x1000_0000
SIM_GAP = 1 << 16
HEADER = ".version 8.0\n.target sm_90\n.address_size 64\n\n"
F32_2POW_M20 = "0f35800000"  # 2^-20


@dataclass
class Buffer:
    name: str
    sim_base: int
    data: np.ndarray  # C-contiguous host array (inputs filled, outputs zero)
    output: bool = False


@dataclass
class Workload:
    name: str
    ptx: str
    kernel: str
    grid: int
    block: int
    params: bytes
    buffers: list[Buffer]
    max_ts: int = 0
    meta: dict = field(default_factory=dict)

    @property
    def warps(self) -> int:
        return self.grid * ((self.block + 31) // 32)

    def buffer(self, name: str) -> Buffer:
        for b in self.buffers:
            if b.name == name:
                return b
        raise KeyError(name)

    def fresh_buffers(self) -> list[Buffer]:
        """Copies of the buffers (outputs zeroed) so two runs start alike."""
        return [Buffer(b.name, b.sim_base, b.data.copy(), b.output) for b in self.buffers]


def place(arrays: list[tuple[str, np.ndarray, bool]]) -> list[Buffer]:
    """Assigns 4 KiB-aligned, non-overlapping simulated base addresses."""
    out, base = [], SIM_BASE0
    for name, arr, is_out in arrays:
        arr = np.ascontiguousarray(arr)
        out.append(Buffer(name, base, arr, is_out))
        base += (arr.nbytes + 4095) // 4096 * 4096 + SIM_GAP
    return out


_PFMT = {"u32": "<I", "s32": "<i", "b32": "<I", "f32": "<f", "u64": "<Q", "s64": "<q", "b64": "<Q"}


def pack_params(decl: list[tuple[str, object]]) -> bytes:
    """Packs (ptx_type, value) pairs in declaration order, each at its natural
    alignment (the layout of a PTX .param list)."""
    blob = bytearray()
    for ty, val in decl:
        size = 8 if ty.endswith("64") else 4
        while len(blob) % size:
            blob.append(0)
        blob += struct.pack(_PFMT[ty], val)
    return bytes(blob)


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def uniform_f32(n: int, lo: float, hi: float, seed: int) -> np.ndarray:
    r = torch.rand(n, generator=_gen(seed), dtype=torch.float32)
    return (lo + (hi - lo) * r).numpy()


def randint_u32(n: int, lo: int, hi: int, seed: int) -> np.ndarray:
    return torch.randint(lo, hi, (n,), generator=_gen(seed), dtype=torch.int64).numpy().astype(np.uint32)


def random_u32(n: int, seed: int) -> np.ndarray:
    return randint_u32(n, 0, 1 << 32, seed)


# --------------------------------------------------------------- vector_add --

def vector_add_ptx() -> str:
    return HEADER + """.visible .entry vector_add(
    .param .u64 va_a,
    .param .u64 va_b,
    .param .u64 va_c,
    .param .u32 va_n
)
{
    .reg .pred  %p<2>;
    .reg .b32   %r<6>;
    .reg .f32   %f<4>;
    .reg .b64   %rd<9>;

    //@iket range_start kernel
    ld.param.u64    %rd1, [va_a];
    ld.param.u64    %rd2, [va_b];
    ld.param.u64    %rd3, [va_c];
    ld.param.u32    %r1, [va_n];
    mov.u32         %r2, %ctaid.x;
    mov.u32         %r3, %ntid.x;
    mov.u32         %r4, %tid.x;
    mad.lo.s32      %r5, %r2, %r3, %r4;
    setp.ge.s32     %p1, %r5, %r1;
    @%p1 bra        VA_EXIT;
    //@iket mark body
    cvt.s64.s32     %rd4, %r5;
    shl.b64         %rd5, %rd4, 2;
    add.s64         %rd6, %rd1, %rd5;
    add.s64         %rd7, %rd2, %rd5;
    add.s64         %rd8, %rd3, %rd5;
    ld.global.f32   %f1, [%rd6];
    ld.global.f32   %f2, [%rd7];
    add.rn.f32      %f3, %f1, %f2;
    st.global.f32   [%rd8], %f3;
VA_EXIT:
    //@iket range_end kernel
    ret;
}
"""


def vector_add(n: int = 4000, block: int = 256, grid: int | None = None, seed: int = 0,
               max_ts: int = 8) -> Workload:
    if grid is None:
        grid = (n + block - 1) // block
    g = _gen(seed)
    a = (-1.0 + 2.0 * torch.rand(n, generator=g, dtype=torch.float32)).numpy()
    b = (-1.0 + 2.0 * torch.rand(n, generator=g, dtype=torch.float32)).numpy()
    c = np.zeros(n, dtype=np.float32)
    bufs = place([("a", a, False), ("b", b, False), ("c", c, True)])
    params = pack_params([("u64", bufs[0].sim_base), ("u64", bufs[1].sim_base),
                          ("u64", bufs[2].sim_base), ("u32", n)])
    return Workload("vector_add", vector_add_ptx(), "vector_add", grid, block, params, bufs,
                    max_ts=max_ts, meta={"n": n})


# -------------------------------------------------------------------- ffma --

def ffma_ptx(acc: int = 1, iters: int = 4096, per_iter: int = 32, name: str | None = None) -> str:
    """FFMA latency probe: `iters` outer iterations of `per_iter` fma.rn.f32
    over `acc` rotating accumulators, then a left-to-right add.rn.f32
    reduction and one store per thread."""
    name = name or f"ffma_acc{acc}"
    nf = 2 + acc
    lines = [
        f".visible .entry {name}(",
        "    .param .u64 fp_out,",
        "    .param .u64 fp_mul,",
        "    .param .u64 fp_add",
        ")",
        "{",
        "    .reg .pred  %p<2>;",
        "    .reg .b32   %r<8>;",
        f"    .reg .f32   %f<{nf}>;",
        "    .reg .b64   %rd<8>;",
        "",
        "    ld.param.u64    %rd1, [fp_out];",
        "    ld.param.u64    %rd2, [fp_mul];",
        "    ld.param.u64    %rd3, [fp_add];",
        "    mov.u32         %r1, %ctaid.x;",
        "    mov.u32         %r2, %ntid.x;",
        "    mov.u32         %r3, %tid.x;",
        "    mad.lo.s32      %r4, %r1, %r2, %r3;",
        "    cvt.u64.u32     %rd4, %r4;",
        "    shl.b64         %rd4, %rd4, 2;",
        "    add.s64         %rd5, %rd2, %rd4;",
        "    add.s64         %rd6, %rd3, %rd4;",
        "    add.s64         %rd7, %rd1, %rd4;",
        "    ld.global.f32   %f0, [%rd5];",
        "    ld.global.f32   %f1, [%rd6];",
    ]
    for j in range(acc):
        lines += [
            f"    add.u32         %r5, %r4, {j};",
            f"    cvt.rn.f32.u32  %f{2 + j}, %r5;",
            f"    mul.rn.f32      %f{2 + j}, %f{2 + j}, {F32_2POW_M20};",
        ]
    lines += ["    mov.u32         %r6, 0;", "    //@iket range_start loop", "FP_LOOP:"]
    for i in range(per_iter):
        a = 2 + (i % acc)
        lines.append(f"    fma.rn.f32      %f{a}, %f{a}, %f0, %f1;")
    lines += [
        "    add.u32         %r6, %r6, 1;",
        f"    setp.lt.u32     %p1, %r6, {iters};",
        "    @%p1 bra        FP_LOOP;",
        "    //@iket range_end loop",
    ]
    for j in range(1, acc):
        lines.append(f"    add.rn.f32      %f2, %f2, %f{2 + j};")
    lines += ["    st.global.f32   [%rd7], %f2;", "    ret;", "}", ""]
    return HEADER + "\n".join(lines)


def ffma(acc: int = 1, iters: int = 4096, per_iter: int = 32, grid: int = 132, block: int = 128,
         seed: int = 2, max_ts: int = 8) -> Workload:
    n = grid * block
    g = _gen(seed)
    m = (0.5 + 1.0 * torch.rand(n, generator=g, dtype=torch.float32)).numpy()
    c = (-1e-3 + 2e-3 * torch.rand(n, generator=g, dtype=torch.float32)).numpy()
    out = np.zeros(n, dtype=np.float32)
    bufs = place([("out", out, True), ("mul", m, False), ("add", c, False)])
    params = pack_params([("u64", bufs[0].sim_base), ("u64", bufs[1].sim_base), ("u64", bufs[2].sim_base)])
    name = f"ffma_acc{acc}"
    return Workload(name, ffma_ptx(acc, iters, per_iter, name), name, grid, block, params, bufs,
                    max_ts=max_ts, meta={"acc": acc, "iters": iters, "per_iter": per_iter})


# ------------------------------------------------------------------ gather --

def gather_ptx() -> str:
    return HEADER + """.visible .entry gather(
    .param .u64 ga_in,
    .param .u64 ga_out,
    .param .u32 ga_s
)
{
    .reg .b32   %r<6>;
    .reg .f32   %f<2>;
    .reg .b64   %rd<9>;

    ld.param.u64    %rd1, [ga_in];
    ld.param.u64    %rd2, [ga_out];
    ld.param.u32    %r1, [ga_s];
    mov.u32         %r2, %ctaid.x;
    mov.u32         %r3, %ntid.x;
    mov.u32         %r4, %tid.x;
    mad.lo.s32      %r5, %r2, %r3, %r4;
    cvt.u64.u32     %rd3, %r5;
    cvt.u64.u32     %rd4, %r1;
    mul.lo.u64      %rd5, %rd3, %rd4;
    shl.b64         %rd5, %rd5, 2;
    add.s64         %rd6, %rd1, %rd5;
    ld.global.f32   %f1, [%rd6];
    shl.b64         %rd7, %rd3, 2;
    add.s64         %rd8, %rd2, %rd7;
    st.global.f32   [%rd8], %f1;
    ret;
}
"""


def gather(stride: int, n_out: int = 1 << 24, block: int = 256, seed: int = 1) -> Workload:
    assert n_out % block == 0
    src = uniform_f32(n_out * stride, -1.0, 1.0, seed)
    out = np.zeros(n_out, dtype=np.float32)
    bufs = place([("in", src, False), ("out", out, True)])
    params = pack_params([("u64", bufs[0].sim_base), ("u64", bufs[1].sim_base), ("u32", stride)])
    return Workload(f"gather_s{stride}", gather_ptx(), "gather", n_out // block, block, params, bufs,
                    max_ts=0, meta={"stride": stride, "n_out": n_out})


# ------------------------------------------------------------ smem_reduce --

def smem_reduce_ptx(block: int) -> str:
    """Per-CTA u32 sum in shared memory: every thread stores its element,
    then a tree over halving strides s (threads tid < s add sdata[tid + s]),
    bar.sync 0 between the steps; thread 0 writes the CTA's sum."""
    return HEADER + f""".visible .entry smem_reduce(
    .param .u64 rd_in,
    .param .u64 rd_out
)
{{
    .reg .pred  %p<3>;
    .reg .b32   %r<12>;
    .reg .b64   %rd<6>;
    .shared .align 4 .b8 sdata[{4 * block}];

    ld.param.u64    %rd1, [rd_in];
    ld.param.u64    %rd2, [rd_out];
    mov.u32         %r1, %tid.x;
    mov.u32         %r2, %ctaid.x;
    mov.u32         %r3, %ntid.x;
    mad.lo.s32      %r4, %r2, %r3, %r1;
    cvt.u64.u32     %rd3, %r4;
    shl.b64         %rd3, %rd3, 2;
    add.s64         %rd4, %rd1, %rd3;
    ld.global.u32   %r5, [%rd4];
    mov.u32         %r6, sdata;
    shl.b32         %r7, %r1, 2;
    add.u32         %r8, %r6, %r7;
    st.shared.u32   [%r8], %r5;
    bar.sync 0;
    shr.u32         %r9, %r3, 1;
    //@iket range_start tree
RD_LOOP:
    setp.eq.u32     %p1, %r9, 0;
    @%p1 bra        RD_DONE;
    setp.lt.u32     %p2, %r1, %r9;
    @!%p2 bra       RD_SKIP;
    shl.b32         %r10, %r9, 2;
    add.u32         %r10, %r8, %r10;
    ld.shared.u32   %r11, [%r10];
    ld.shared.u32   %r5, [%r8];
    add.u32         %r5, %r5, %r11;
    st.shared.u32   [%r8], %r5;
RD_SKIP:
    bar.sync 0;
    shr.u32         %r9, %r9, 1;
    bra             RD_LOOP;
RD_DONE:
    //@iket range_end tree
    setp.ne.u32     %p1, %r1, 0;
    @%p1 bra        RD_EXIT;
    cvt.u64.u32     %rd3, %r2;
    shl.b64         %rd3, %rd3, 2;
    add.s64         %rd5, %rd2, %rd3;
    st.global.u32   [%rd5], %r5;
RD_EXIT:
    ret;
}}
"""


def smem_reduce(n: int = 1 << 22, block: int = 256, seed: int = 5, max_ts: int = 4) -> Workload:
    """Shared-memory tree reduction: one u32 sum per CTA of `block` threads
    (block a power of two, at most 1024)."""
    assert block & (block - 1) == 0 and 2 <= block <= 1024 and n % block == 0
    x = randint_u32(n, 0, 1 << 31, seed)
    out = np.zeros(n // block, dtype=np.uint32)
    bufs = place([("in", x, False), ("out", out, True)])
    params = pack_params([("u64", bufs[0].sim_base), ("u64", bufs[1].sim_base)])
    return Workload(f"smem_reduce_b{block}", smem_reduce_ptx(block), "smem_reduce", n // block, block, params,
                    bufs, max_ts=max_ts, meta={"n": n, "block": block})


# ---------------------------------------------------------- fuzz_shared --

def fuzz_shared_ptx(seed: int, block: int) -> str:
    """A random program over shared memory and bar.sync, race-free by
    construction and defined natively (no word is read before it is
    written). A .shared array holds two halves of 2*block u32 words and a
    u64 area. Thread x starts from in[gtid] and stores it and a second word to
    half 0 at tid and tid + block; then each phase (separated by bar.sync 0)
    reads the half written last at a random index map (tid*A + B) &
    (2*block - 1) — so lanes of a warp hit the same bank on different words,
    or share a word — combines it with x, may run a divergent then-block, and
    stores x and a second word to the other half; the half offset toggles in
    a register, so phases can sit in uniform loops. Some phases write the u64
    area with 8-byte stores and read a neighbour's entry after the barrier.
    Every barrier is in convergent code. The result goes to out[gtid]."""
    assert block & (block - 1) == 0 and 32 <= block <= 1024
    rng = random.Random(seed)
    words = 2 * block
    half = 4 * words
    lines = [
        f".visible .entry fuzz_sh(",
        "    .param .u64 fs_in,",
        "    .param .u64 fs_out",
        ")",
        "{",
        "    .reg .pred  %p<4>;",
        "    .reg .b32   %r<24>;",
        "    .reg .b64   %rd<10>;",
        f"    .shared .align 8 .b8 sw[{2 * half}];",
        f"    .shared .align 8 .b8 sd[{8 * words}];",
        "    ld.param.u64    %rd1, [fs_in];",
        "    ld.param.u64    %rd2, [fs_out];",
        "    mov.u32         %r1, %tid.x;",
        "    mov.u32         %r2, %ctaid.x;",
        "    mov.u32         %r3, %ntid.x;",
        "    mad.lo.s32      %r4, %r2, %r3, %r1;",
        "    cvt.u64.u32     %rd3, %r4;",
        "    shl.b64         %rd3, %rd3, 2;",
        "    add.s64         %rd4, %rd1, %rd3;",
        "    ld.global.u32   %r5, [%rd4];",
        "    mov.u32         %r6, sw;",
        "    mov.u32         %r7, sd;",
        "    shl.b32         %r8, %r1, 2;",
        "    add.u32         %r9, %r6, %r8;",
        "    st.shared.u32   [%r9], %r5;",
        "    xor.b32         %r19, %r5, 1431655765;",
        f"    st.shared.u32   [%r9+{4 * block}], %r19;",
        "    mov.u32         %r10, 0;",   # byte offset of the half written last
        "    bar.sync 0;",
    ]
    label = [0]

    def phase(out):
        a, b = rng.randrange(0, 2 * words), rng.randrange(0, words)
        out += [
            f"    mul.lo.u32      %r11, %r1, {a};",
            f"    add.u32         %r11, %r11, {b};",
            f"    and.b32         %r11, %r11, {words - 1};",
            "    shl.b32         %r11, %r11, 2;",
            "    add.u32         %r11, %r11, %r10;",
            "    add.u32         %r11, %r11, %r6;",
            "    ld.shared.u32   %r12, [%r11];",
        ]
        op = rng.choice(["xor", "add", "mad"])
        if op == "xor":
            out.append("    xor.b32         %r5, %r5, %r12;")
        elif op == "add":
            out.append("    add.u32         %r5, %r5, %r12;")
        else:
            out.append(f"    mad.lo.u32      %r5, %r12, {rng.randrange(1, 1 << 31) | 1}, %r5;")
        if rng.random() < 0.4:  # a divergent then-block
            label[0] += 1
            m = rng.choice([1, 3, 7, 15, 31])
            out += [
                f"    and.b32         %r13, %r1, {m};",
                "    setp.ne.u32     %p1, %r13, 0;",
                f"    @%p1 bra        FS_SKIP{label[0]};",
                f"    mul.lo.u32      %r5, %r5, {rng.randrange(3, 1 << 20) | 1};",
                f"    add.u32         %r5, %r5, {rng.randrange(0, 1 << 30)};",
                f"FS_SKIP{label[0]}:",
            ]
        wrote64 = rng.random() < 0.3
        if wrote64:  # the u64 area: written here, read back through a map after the barrier
            out += [
                "    cvt.u64.u32     %rd5, %r5;",
                "    shl.b64         %rd5, %rd5, 7;",
                "    cvt.u64.u32     %rd6, %r12;",
                "    xor.b64         %rd5, %rd5, %rd6;",
                "    shl.b32         %r14, %r1, 3;",
                "    add.u32         %r14, %r14, %r7;",
                "    st.shared.u64   [%r14], %rd5;",
            ]
        # write x and a second word to the other half (every word of a half is
        # written before it is read), then the barrier
        out += [
            f"    xor.b32         %r10, %r10, {half};",
            "    add.u32         %r15, %r8, %r10;",
            "    add.u32         %r15, %r15, %r6;",
            "    st.shared.u32   [%r15], %r5;",
            f"    add.u32         %r19, %r5, {rng.randrange(1, 1 << 31)};",
            f"    st.shared.u32   [%r15+{4 * block}], %r19;",
            "    bar.sync 0;",
        ]
        if wrote64 and rng.random() < 0.7:  # read the u64 area of a neighbour
            c = rng.choice([1, 3, 5, 33])
            out += [
                f"    mul.lo.u32      %r16, %r1, {c};",
                f"    and.b32         %r16, %r16, {block - 1};",
                "    shl.b32         %r16, %r16, 3;",
                "    add.u32         %r16, %r16, %r7;",
                "    ld.shared.u64   %rd7, [%r16];",
                "    cvt.u32.u64     %r17, %rd7;",
                "    add.u32         %r5, %r5, %r17;",
                "    bar.sync 0;",  # the u64 area may be written again next phase
            ]

    for _ in range(rng.randint(3, 6)):
        if rng.random() < 0.3:  # a uniform loop of phases
            label[0] += 1
            loop = label[0]
            trips = rng.randint(2, 4)
            lines += ["    mov.u32         %r18, 0;", "    //@iket range_start loop", f"FS_LOOP{loop}:"]
            phase(lines)
            lines += ["    add.u32         %r18, %r18, 1;", f"    setp.lt.u32     %p2, %r18, {trips};",
                      f"    @%p2 bra        FS_LOOP{loop};", "    //@iket range_end loop"]
        else:
            phase(lines)
    lines += [
        "    add.s64         %rd8, %rd2, %rd3;",
        "    st.global.u32   [%rd8], %r5;",
        "    ret;",
        "}",
        "",
    ]
    return HEADER + "\n".join(lines)


def fuzz_shared(i: int, grid: int = 64, block: int = 128, seed_base: int = 2000, data_seed: int = 6,
                max_ts: int = 16) -> Workload:
    """Random shared-memory / barrier program i (seed seed_base + i)."""
    n = grid * block
    x = randint_u32(n, 0, 1 << 31, data_seed)
    out = np.zeros(n, dtype=np.uint32)
    bufs = place([("in", x, False), ("out", out, True)])
    params = pack_params([("u64", bufs[0].sim_base), ("u64", bufs[1].sim_base)])
    return Workload(f"fuzz_shared_{seed_base + i}", fuzz_shared_ptx(seed_base + i, block), "fuzz_sh", grid, block,
                    params, bufs, max_ts=max_ts, meta={"seed": seed_base + i})


# --------------------------------------------------------------- divergent --

DIVERGENT_BODY_OPS = 16
DIVERGENT_THEN_OPS = 5


def divergent_ptx() -> str:
    return HEADER + """.visible .entry divergent(
    .param .u64 dv_in,
    .param .u64 dv_out,
    .param .u32 dv_k
)
{
    .reg .pred  %p<4>;
    .reg .b32   %r<22>;
    .reg .b64   %rd<6>;

    ld.param.u64    %rd1, [dv_in];
    ld.param.u64    %rd2, [dv_out];
    ld.param.u32    %r1, [dv_k];
    mov.u32         %r2, %ctaid.x;
    mov.u32         %r3, %ntid.x;
    mov.u32         %r4, %tid.x;
    mad.lo.s32      %r5, %r2, %r3, %r4;
    cvt.u64.u32     %rd3, %r5;
    shl.b64         %rd3, %rd3, 2;
    add.s64         %rd4, %rd1, %rd3;
    add.s64         %rd5, %rd2, %rd3;
    ld.global.u32   %r6, [%rd4];
    and.b32         %r7, %r4, 31;
    sub.u32         %r8, %r1, 1;
    mov.u32         %r9, %r5;
    mov.u32         %r10, 0;
    //@iket range_start loop
DV_HEAD:
    setp.ge.u32     %p1, %r10, %r6;
    @%p1 bra        DV_DONE;
    mul.lo.u32      %r11, %r9, 0x9E3779B1;
    xor.b32         %r11, %r11, %r10;
    shl.b32         %r12, %r11, 3;
    shr.u32         %r13, %r11, 5;
    xor.b32         %r14, %r12, %r13;
    and.b32         %r15, %r14, 0xFFFF;
    add.u32         %r9, %r9, %r15;
    setp.lt.u32     %p2, %r15, 0x8000;
    selp.u32        %r16, %r14, %r13, %p2;
    add.u32         %r9, %r9, %r16;
    mul.lo.u32      %r9, %r9, 0x01000193;
    xor.b32         %r9, %r9, %r6;
    shr.u32         %r17, %r9, 5;
    shl.b32         %r18, %r17, 3;
    add.u32         %r9, %r9, %r18;
    and.b32         %r19, %r7, %r8;
    setp.eq.u32     %p3, %r19, 0;
    @!%p3 bra       DV_SKIP;
    mul.lo.u32      %r20, %r9, 3;
    add.u32         %r20, %r20, %r10;
    xor.b32         %r9, %r9, %r20;
    shr.u32         %r21, %r9, 7;
    add.u32         %r9, %r9, %r21;
DV_SKIP:
    add.u32         %r10, %r10, 1;
    bra.uni         DV_HEAD;
DV_DONE:
    //@iket range_end loop
    st.global.u32   [%rd5], %r9;
    ret;
}
"""


def divergent(k: int, n: int = 1 << 20, block: int = 128, seed: int = 3, max_ts: int = 8) -> Workload:
    assert k in (1, 2, 4, 8, 16, 32) and n % block == 0
    trips = randint_u32(n, 0, 64, seed)
    out = np.zeros(n, dtype=np.uint32)
    bufs = place([("in", trips, False), ("out", out, True)])
    params = pack_params([("u64", bufs[0].sim_base), ("u64", bufs[1].sim_base), ("u32", k)])
    return Workload(f"divergent_k{k}", divergent_ptx(), "divergent", n // block, block, params, bufs,
                    max_ts=max_ts, meta={"k": k, "n": n})


# -------------------------------------------------------------------- fuzz --
# Random structured programs. Construction rules that make them valid for
# both interpreters and for the driver JIT, race-free and bounded:
#   * every register is written at entry from gtid before any use;
#   * loads only from inF / inU at (s*gtid + c + sum d_i*loop_i) & (2^20-1);
#   * stores only to `out` at perm_s(gtid) + T*k, T = 2^18, k in 0..3, where
#     perm_s interleaves lanes with stride s inside groups of s warps, so each
#     thread owns four private words;
#   * addresses never depend on loaded data;
#   * f32 add/sub/mul carry .rn so a JIT compiler cannot contract them;
#   * loops are counted (trip <= 16, possibly lane-dependent) and nest <= 4
#     deep, with the product of enclosing trips bounded so that the dynamic
#     instruction count per thread stays under the budget;
#   * range_start / range_end pseudo-ops surround every loop.

FUZZ_N = 1 << 20       # words per fuzz buffer (4 MiB)
FUZZ_T = 1 << 18       # threads in a fuzz launch (1024 x 256)
FUZZ_INT = 20          # %r0..%r19   32-bit integer pool
FUZZ_FLT = 8           # %f0..%f7    32-bit float pool
FUZZ_WIDE = 4          # %rd0..%rd3  64-bit integer pool


class _FuzzGen:
    def __init__(self, seed: int, n_static: int, budget: int, early_exit: bool):
        self.rng = random.Random(seed)
        self.n_static = n_static
        self.budget = budget
        self.early_exit = early_exit
        self.lines: list[str] = []
        self.count = 0          # static instructions emitted
        self.label_no = 0
        self.loop_no = 0
        self.mult = 1           # product of the enclosing loops' maximum trips
        self.dynamic = 0        # upper bound of instructions one thread issues

    # -- helpers --
    def emit(self, text: str):
        self.lines.append("    " + text)
        self.count += 1
        self.dynamic += self.mult

    def label(self, stem: str) -> str:
        self.label_no += 1
        return f"FZ_{stem}{self.label_no}"

    def ri(self) -> str:
        return f"%r{self.rng.randrange(FUZZ_INT)}"

    def rf(self) -> str:
        return f"%f{self.rng.randrange(FUZZ_FLT)}"

    def rw(self) -> str:
        return f"%rd{self.rng.randrange(FUZZ_WIDE)}"

    def imm32(self) -> str:
        c = self.rng.random()
        if c < 0.4:
            return str(self.rng.randrange(0, 64))
        if c < 0.7:
            return hex(self.rng.getrandbits(32))
        return str(-self.rng.randrange(1, 1 << 31))

    def fimm(self) -> str:
        # a modest-magnitude float literal (sign, exponent in [-8, 8])
        sign = self.rng.random() < 0.3
        e = self.rng.randrange(-8, 9)
        mant = self.rng.getrandbits(23)
        bits = (int(sign) << 31) | ((127 + e) << 23) | mant
        return f"0f{bits:08X}"

    # -- instruction makers --
    def int_op(self, guard: str = ""):
        r = self.rng
        d, a = self.ri(), self.ri()
        b = self.ri() if r.random() < 0.7 else self.imm32()
        op = r.choice(["add.u32", "add.s32", "sub.u32", "sub.s32", "mul.lo.u32", "mul.lo.s32",
                       "mad.lo.u32", "mad.lo.s32", "and.b32", "or.b32", "xor.b32", "shl.b32",
                       "shr.u32", "shr.s32", "shr.b32", "selp.u32", "mov.u32", "cvt.rzi.s32.f32",
                       "cvt.rni.u32.f32", "cvt.rmi.s32.f32", "cvt.rpi.u32.f32", "mov.b32"])
        if op.startswith("mad"):
            self.emit(f"{guard}{op} {d}, {a}, {b}, {self.ri()};")
        elif op.startswith(("shl", "shr")):
            amt = self.ri() if r.random() < 0.3 else str(r.randrange(0, 40))
            self.emit(f"{guard}{op} {d}, {a}, {amt};")
        elif op == "selp.u32":
            self.emit(f"{guard}{op} {d}, {a}, {b}, %p{r.randrange(4)};")
        elif op == "mov.u32":
            self.emit(f"{guard}{op} {d}, {b};")
        elif op == "mov.b32":
            self.emit(f"{guard}{op} {d}, {self.rf()};")
        elif op.startswith("cvt"):
            self.emit(f"{guard}{op} {d}, {self.rf()};")
        else:
            self.emit(f"{guard}{op} {d}, {a}, {b};")

    def flt_op(self, guard: str = ""):
        r = self.rng
        d, a = self.rf(), self.rf()
        b = self.rf() if r.random() < 0.75 else self.fimm()
        op = r.choice(["add.rn.f32", "sub.rn.f32", "mul.rn.f32", "fma.rn.f32", "fma.rn.f32",
                       "div.rn.f32", "sqrt.rn.f32", "cvt.rn.f32.u32", "cvt.rn.f32.s32",
                       "selp.f32", "mov.f32", "mov.b32"])
        if op == "fma.rn.f32":
            self.emit(f"{guard}{op} {d}, {a}, {b}, {self.rf()};")
        elif op == "sqrt.rn.f32":
            self.emit(f"{guard}{op} {d}, {a};")
        elif op.startswith("cvt"):
            self.emit(f"{guard}{op} {d}, {self.ri()};")
        elif op == "selp.f32":
            self.emit(f"{guard}{op} {d}, {a}, {b}, %p{r.randrange(4)};")
        elif op == "mov.f32":
            self.emit(f"{guard}{op} {d}, {b};")
        elif op == "mov.b32":
            self.emit(f"{guard}{op} {d}, {self.ri()};")
        else:
            self.emit(f"{guard}{op} {d}, {a}, {b};")

    def wide_op(self, guard: str = ""):
        r = self.rng
        d, a = self.rw(), self.rw()
        op = r.choice(["add.u64", "sub.s64", "mul.lo.u64", "xor.b64", "and.b64", "or.b64",
                       "shl.b64", "shr.s64", "shr.u64", "cvt.u64.u32", "cvt.s64.s32",
                       "cvt.u32.u64", "cvt.rn.f32.s64", "cvt.rzi.s64.f32", "selp.b64", "mad.lo.s64"])
        if op.startswith(("shl", "shr")):
            self.emit(f"{guard}{op} {d}, {a}, {r.randrange(0, 70)};")
        elif op in ("cvt.u64.u32", "cvt.s64.s32"):
            self.emit(f"{guard}{op} {d}, {self.ri()};")
        elif op == "cvt.u32.u64":
            self.emit(f"{guard}{op} {self.ri()}, {a};")
        elif op == "cvt.rn.f32.s64":
            self.emit(f"{guard}{op} {self.rf()}, {a};")
        elif op == "cvt.rzi.s64.f32":
            self.emit(f"{guard}{op} {d}, {self.rf()};")
        elif op == "selp.b64":
            self.emit(f"{guard}{op} {d}, {a}, {self.rw()}, %p{r.randrange(4)};")
        elif op == "mad.lo.s64":
            self.emit(f"{guard}{op} {d}, {a}, {self.rw()}, {self.rw()};")
        else:
            b = self.rw() if r.random() < 0.7 else str(r.randrange(-1000, 100000))
            self.emit(f"{guard}{op} {d}, {a}, {b};")

    def setp_op(self, p: int, guard: str = ""):
        r = self.rng
        c = r.random()
        if c < 0.5:
            cmp = r.choice(["eq", "ne", "lt", "le", "gt", "ge"])
            ty = r.choice(["u32", "s32"])
            b = self.ri() if r.random() < 0.5 else self.imm32()
            self.emit(f"{guard}setp.{cmp}.{ty} %p{p}, {self.ri()}, {b};")
        elif c < 0.8:
            cmp = r.choice(["eq", "ne", "lt", "le", "gt", "ge"])
            self.emit(f"{guard}setp.{cmp}.f32 %p{p}, {self.rf()}, {self.rf()};")
        else:
            op = r.choice(["and", "or", "xor"])
            self.emit(f"{guard}{op}.pred %p{p}, %p{r.randrange(4)}, %p{r.randrange(4)};")

    def guard(self) -> str:
        if self.rng.random() < 0.15:
            neg = "!" if self.rng.random() < 0.5 else ""
            return f"@{neg}%p{self.rng.randrange(4)} "
        return ""

    def index_expr(self, loops: list[str]):
        """%ra <- (s*gtid + c + sum d_i*loop_i) & mask (in %ra), returns nothing."""
        r = self.rng
        s = r.randrange(1, 65)
        c = r.randrange(0, FUZZ_N)
        self.emit(f"mul.lo.u32 %ra, %gt, {s};")
        self.emit(f"add.u32 %ra, %ra, {c};")
        for lv in loops:
            if r.random() < 0.6:
                self.emit(f"mad.lo.u32 %ra, {lv}, {r.randrange(1, 65)}, %ra;")

    def load(self, loops: list[str]):
        r = self.rng
        self.index_expr(loops)
        kind = r.random()
        if kind < 0.45:
            self.emit("and.b32 %ra, %ra, 1048575;")
            self._addr("%inF", 4)
            self.emit(f"ld.global.f32 {self.rf()}, [%aa];")
        elif kind < 0.85:
            self.emit("and.b32 %ra, %ra, 1048575;")
            self._addr("%inU", 4)
            self.emit(f"ld.global.u32 {self.ri()}, [%aa];")
        else:
            self.emit("and.b32 %ra, %ra, 1048574;")
            self._addr("%inU", 4)
            self.emit(f"ld.global.u64 {self.rw()}, [%aa];")

    def _addr(self, base: str, scale: int):
        self.emit("cvt.u64.u32 %aa, %ra;")
        self.emit(f"shl.b64 %aa, %aa, {scale.bit_length() - 1};")
        self.emit(f"add.s64 %aa, {base}, %aa;")

    def store(self, loops: list[str]):
        r = self.rng
        # k = (affine in loop counters) & 3, slot = perm + T*k
        self.emit(f"mov.u32 %ra, {r.randrange(0, 4)};")
        for lv in loops:
            if r.random() < 0.5:
                self.emit(f"add.u32 %ra, %ra, {lv};")
        self.emit("and.b32 %ra, %ra, 3;")
        self.emit(f"mad.lo.u32 %ra, %ra, {FUZZ_T}, %pm;")
        self._addr("%outp", 4)
        if r.random() < 0.5:
            self.emit(f"{self.guard()}st.global.u32 [%aa], {self.ri()};")
        else:
            self.emit(f"{self.guard()}st.global.f32 [%aa], {self.rf()};")

    # -- structure --
    def block(self, depth: int, loops: list[str], mult: int, room: int):
        """Emits straight-line code and nested structures, about `room` insts."""
        r = self.rng
        end = self.count + room
        while self.count < end:
            c = r.random()
            left = end - self.count
            if c < 0.08 and depth < 4 and left > 14:
                self.loop(depth, loops, mult, r.randrange(6, max(7, min(left, 60))))
            elif c < 0.15 and left > 10:
                self.if_block(depth, loops, mult, r.randrange(3, max(4, min(left, 30))))
            elif c < 0.22:
                self.load(loops)
            elif c < 0.27:
                self.store(loops)
            elif c < 0.33:
                self.setp_op(r.randrange(4), self.guard())
            elif c < 0.34 and self.early_exit and depth > 0:
                self.emit(f"@%p{r.randrange(4)} ret;")
            elif c < 0.55:
                self.flt_op(self.guard())
            elif c < 0.65:
                self.wide_op(self.guard())
            else:
                self.int_op(self.guard())

    def if_block(self, depth, loops, mult, room):
        r = self.rng
        p = r.randrange(4)
        self.setp_op(p)
        neg = "!" if r.random() < 0.5 else ""
        if r.random() < 0.5:
            skip = self.label("skip")
            self.emit(f"@{neg}%p{p} bra {skip};")
            self.block(depth, loops, mult, room)
            self.lines.append(f"{skip}:")
        else:
            other, join = self.label("else"), self.label("join")
            self.emit(f"@{neg}%p{p} bra {other};")
            self.block(depth, loops, mult, room // 2)
            self.emit(f"bra.uni {join};")
            self.lines.append(f"{other}:")
            self.block(depth, loops, mult, room - room // 2)
            self.lines.append(f"{join}:")

    def loop(self, depth, loops, mult, room):
        r = self.rng
        # bound the trip so that mult * trip * room stays within the budget
        max_trip = max(1, min(16, self.budget // max(1, mult * (room + 8))))
        trip = r.randrange(1, max_trip + 1)
        lv = f"%lc{depth}"
        tr = f"%lt{depth}"
        lane_dep = r.random() < 0.5 and trip > 1
        self.loop_no += 1
        name = f"loop{self.loop_no}"
        head = self.label("loop")
        self.emit(f"mov.u32 {lv}, 0;")
        if lane_dep:
            # trip in 1..trip, varying per lane
            self.emit(f"and.b32 {tr}, %gt, {(1 << (trip.bit_length() - 1)) - 1};")
            self.emit(f"add.u32 {tr}, {tr}, 1;")
        else:
            self.emit(f"mov.u32 {tr}, {trip};")
        self.lines.append(f"    //@iket range_start {name}")
        self.lines.append(f"{head}:")
        outer_mult = self.mult
        self.mult = mult * trip
        brk = None
        if r.random() < 0.15:
            brk = self.label("brk")
            p = r.randrange(4)
            self.setp_op(p)
            self.emit(f"@%p{p} bra {brk};")
        self.block(depth + 1, loops + [lv], mult * trip, room)
        self.emit(f"add.u32 {lv}, {lv}, 1;")
        self.emit(f"setp.lt.u32 %pl, {lv}, {tr};")
        self.emit(f"@%pl bra {head};")
        self.mult = outer_mult
        if brk:
            self.lines.append(f"{brk}:")
        self.lines.append(f"    //@iket range_end {name}")

    def program(self, name: str) -> str:
        r = self.rng
        s_perm = 1 << r.randrange(0, 7)  # 1..64
        self.s_perm = s_perm
        body_start = len(self.lines)
        # prologue: gtid, buffer pointers, perm_s(gtid), register pool init
        pro = [
            "ld.param.u64 %inF, [fz_inf];",
            "ld.param.u64 %inU, [fz_inu];",
            "ld.param.u64 %outp, [fz_out];",
            "mov.u32 %ra, %ctaid.x;",
            "mov.u32 %rb, %ntid.x;",
            "mov.u32 %gt, %tid.x;",
            "mad.lo.s32 %gt, %ra, %rb, %gt;",
            # perm_s(g) = (g & ~(32s-1)) | ((g & 31) * s) | ((g >> 5) & (s-1))
            f"and.b32 %pm, %gt, {0xFFFFFFFF ^ (32 * s_perm - 1)};",
            "and.b32 %ra, %gt, 31;",
            f"mul.lo.u32 %ra, %ra, {s_perm};",
            "or.b32 %pm, %pm, %ra;",
            "shr.u32 %ra, %gt, 5;",
            f"and.b32 %ra, %ra, {s_perm - 1};",
            "or.b32 %pm, %pm, %ra;",
        ]
        for t in pro:
            self.emit(t)
        for i in range(FUZZ_INT):
            self.emit(f"mad.lo.u32 %r{i}, %gt, {r.getrandbits(32) | 1}, {r.getrandbits(31)};")
        for i in range(FUZZ_FLT):
            self.emit(f"cvt.rn.f32.u32 %f{i}, %r{i};")
            self.emit(f"mul.rn.f32 %f{i}, %f{i}, {F32_2POW_M20};")
        for i in range(FUZZ_WIDE):
            self.emit(f"cvt.u64.u32 %rd{i}, %r{FUZZ_INT - 1 - i};")
        for i in range(4):
            self.emit(f"setp.lt.u32 %p{i}, %r{i + 4}, {hex(r.getrandbits(32))};")
        self.emit("setp.eq.u32 %pl, %gt, 0;")
        for d in range(4):
            self.emit(f"mov.u32 %lc{d}, 0;")
            self.emit(f"mov.u32 %lt{d}, 0;")
        self.emit("mov.u64 %aa, 0;")
        room = max(8, self.n_static - self.count - 8)
        self.block(0, [], 1, room)
        # final stores so every thread leaves a result
        self.store([])
        self.emit("ret;")
        body = "\n".join(self.lines[body_start:])
        decl = "\n".join([
            "    .reg .pred %p<4>;",
            "    .reg .pred %pl;",
            f"    .reg .b32 %r<{FUZZ_INT}>;",
            f"    .reg .f32 %f<{FUZZ_FLT}>;",
            f"    .reg .b64 %rd<{FUZZ_WIDE}>;",
            "    .reg .b32 %ra, %rb, %gt, %pm;",
            "    .reg .b32 %lc<4>;",
            "    .reg .b32 %lt<4>;",
            "    .reg .b64 %inF, %inU, %outp, %aa;",
        ])
        return HEADER + (f".visible .entry {name}(\n    .param .u64 fz_inf,\n    .param .u64 fz_inu,\n"
                         f"    .param .u64 fz_out\n)\n{{\n{decl}\n\n{body}\n}}\n")


def fuzz_program(seed: int, n_static: int = 256, budget: int = 20000, early_exit: bool = True):
    """A random program named fuzz_<seed>, redrawn (with a derived stream)
    until its static bound on per-thread issued instructions fits `budget`.
    Returns (ptx, s) where s is the lane-interleave stride of its stores."""
    for attempt in range(100):
        g = _FuzzGen(seed * 1000 + attempt, n_static, budget, early_exit)
        text = g.program(f"fuzz_{seed}")
        if g.dynamic <= budget:
            return text, g.s_perm
    raise RuntimeError("fuzz generator could not meet the dynamic budget")


def fuzz_ptx(seed: int, n_static: int = 256, budget: int = 20000, early_exit: bool = True) -> str:
    return fuzz_program(seed, n_static, budget, early_exit)[0]


def fuzz_store_words(gtid: np.ndarray, s_perm: int) -> np.ndarray:
    """The four `out` words thread gtid may store to (perm_s(gtid) + T*k)."""
    g = gtid.astype(np.int64)
    perm = (g & ~(32 * s_perm - 1)) | ((g & 31) * s_perm) | ((g >> 5) & (s_perm - 1))
    return (perm[:, None] + FUZZ_T * np.arange(4)[None, :]).reshape(-1)


def fuzz(i: int, grid: int = 1024, block: int = 256, data_seed: int = 4, max_ts: int = 64,
         n_static: int = 256, early_exit: bool = True) -> Workload:
    seed = 1000 + i
    ptx, s_perm = fuzz_program(seed, n_static=n_static, early_exit=early_exit)
    inf = uniform_f32(FUZZ_N, -2.0, 2.0, data_seed)
    inu = random_u32(FUZZ_N, data_seed + 1)
    out = np.zeros(FUZZ_N, dtype=np.uint32)
    bufs = place([("inF", inf, False), ("inU", inu, False), ("out", out, True)])
    params = pack_params([("u64", bufs[0].sim_base), ("u64", bufs[1].sim_base), ("u64", bufs[2].sim_base)])
    return Workload(f"fuzz_{seed}", ptx, f"fuzz_{seed}", grid, block, params, bufs, max_ts=max_ts,
                    meta={"seed": seed, "s_perm": s_perm})
