"""Pins the oracle's single-instruction semantics to arithmetic that does not
come from the oracle: exact rationals rounded by the IEEE 754 rule (f32),
Python big integers masked to the register width (integers), and the PTX ISA
rules for shifts, saturating conversions and ordered comparisons.

Each case runs one instruction per thread over 256 threads with operands
chosen to hit edge values (zeros of both signs, subnormals, infinities, NaN,
extreme integers) plus seeded random bits.
"""
import random
import struct

import numpy as np
import pytest

import oracle
from tests import _exact as X
from tests._kernels import op_workload

N = 256
M32 = (1 << 32) - 1
M64 = (1 << 64) - 1

F32_EDGE = [0x00000000, 0x80000000, 0x00000001, 0x80000001, 0x007FFFFF, 0x00800000, 0x7F7FFFFF,
            0xFF7FFFFF, 0x7F800000, 0xFF800000, 0x7FC00000, 0x7F800001, 0x3F800000, 0xBF800000,
            0x3F000000, 0x4B000000, 0x4B000001, 0xCB000000, 0x3EFFFFFF, 0x3FC00000, 0x40200000,
            0x4F000000, 0xCF000000, 0x4F800000, 0x5F000000, 0xDF000000, 0x5F800000, 0x34000000]
I32_EDGE = [0, 1, 2, 31, 32, 33, 63, 64, 0x7FFFFFFF, 0x80000000, 0xFFFFFFFF, 0xFFFFFFFE, 0x12345678]
I64_EDGE = [0, 1, 63, 64, 65, 0x7FFFFFFFFFFFFFFF, 0x8000000000000000, M64, 0xFFFFFFFF, 0x100000000]


def f32_operands(seed):
    rng = random.Random(seed)
    vals = list(F32_EDGE)
    while len(vals) < N:
        c = rng.random()
        if c < 0.5:
            vals.append(rng.getrandbits(32))
        elif c < 0.8:  # moderate magnitudes so that sums/products stay finite and inexact
            e = rng.randrange(110, 145)
            vals.append((rng.getrandbits(1) << 31) | (e << 23) | rng.getrandbits(23))
        else:  # near-subnormal
            vals.append((rng.getrandbits(1) << 31) | rng.getrandbits(24))
    rng.shuffle(vals)
    return vals[:N]


def int_operands(seed, width):
    rng = random.Random(seed)
    edge = I32_EDGE if width == 32 else I64_EDGE
    vals = list(edge)
    while len(vals) < N:
        vals.append(rng.getrandbits(width) if rng.random() < 0.7 else rng.randrange(0, 80))
    rng.shuffle(vals)
    return vals[:N]


def run_op(name, op, srcs, dst, a, b=None, c=None, imm=None):
    w = op_workload(name, op, srcs, dst, np.array(a, dtype=np.uint64),
                    None if b is None else np.array(b, dtype=np.uint64),
                    None if c is None else np.array(c, dtype=np.uint64), imm=imm)
    bufs = w.fresh_buffers()
    r = oracle.run(w.ptx, w.kernel, w.grid, w.block, w.params, [(x.sim_base, x.data) for x in bufs])
    assert r.status == 0
    return [int(v) for v in bufs[0].data]


def sx(v, w):
    v &= (1 << w) - 1
    return v - (1 << w) if v >> (w - 1) else v


# ------------------------------------------------------------------ f32 ----

@pytest.mark.parametrize("opname", ["add", "sub", "mul", "div"])
def test_f32_binary_exact(opname):
    a = f32_operands(1)
    b = f32_operands(2)
    op = {"add": "add.rn.f32", "sub": "sub.rn.f32", "mul": "mul.rn.f32", "div": "div.rn.f32"}[opname]
    got = run_op(f"k_{opname}", op, "ff", "f", a, b)
    for x, y, g in zip(a, b, got):
        if opname == "add":
            want = X.add(x, y)
        elif opname == "sub":
            want = X.add(x, y, sub=True)
        elif opname == "mul":
            want = X.mul(x, y)
        else:
            want = X.div(x, y)
        assert g == want, (opname, hex(x), hex(y), hex(g), hex(want))


def test_f32_add_without_rounding_suffix_is_rn():
    a, b = f32_operands(3), f32_operands(4)
    got = run_op("k_addplain", "add.f32", "ff", "f", a, b)
    assert got == [X.add(x, y) for x, y in zip(a, b)]


def test_f32_fma_exact():
    a, b, c = f32_operands(5), f32_operands(6), f32_operands(7)
    got = run_op("k_fma", "fma.rn.f32", "fff", "f", a, b, c)
    for x, y, z, g in zip(a, b, c, got):
        assert g == X.fma(x, y, z), (hex(x), hex(y), hex(z), hex(g))


def test_f32_sqrt_exact():
    a = f32_operands(8)
    got = run_op("k_sqrt", "sqrt.rn.f32", "f", "f", a)
    for x, g in zip(a, got):
        assert g == X.sqrt(x), (hex(x), hex(g))


def test_f32_immediate_operand():
    a = f32_operands(9)
    got = run_op("k_addimm", "add.rn.f32", "fi", "f", a, imm="0f3FC00000")  # 1.5
    assert got == [X.add(x, 0x3FC00000) for x in a]


def test_nan_results_are_canonical():
    a = [0x7F800000, 0xFF800000, 0x7FC00001, 0xFFFFFFFF] * (N // 4)
    b = [0xFF800000, 0x7F800000, 0x3F800000, 0x3F800000] * (N // 4)
    got = run_op("k_nan", "add.rn.f32", "ff", "f", a, b)
    assert set(got) == {0x7FFFFFFF}


@pytest.mark.parametrize("cmp", ["eq", "ne", "lt", "le", "gt", "ge"])
def test_setp_f32_ordered(cmp):
    a, b = f32_operands(10), f32_operands(11)
    a[:8] = [0x7FC00000, 0x3F800000, 0x7FC00000, 0, 0x80000000, 0x7F800000, 0xFF800000, 1]
    b[:8] = [0x3F800000, 0x7FC00000, 0x7FC00000, 0x80000000, 0, 0x7F800000, 0x7F800000, 0]
    got = run_op(f"k_setpf_{cmp}", f"setp.{cmp}.f32", "ff", "p", a, b)
    assert got == [int(X.cmp_f32(x, y, cmp)) for x, y in zip(a, b)]


# ------------------------------------------------------------- integers ----

INT_BINARY = {
    "add": lambda a, b, w: a + b,
    "sub": lambda a, b, w: a - b,
    "mul.lo": lambda a, b, w: a * b,
}


@pytest.mark.parametrize("ty", ["u32", "s32", "u64", "s64"])
@pytest.mark.parametrize("op", ["add", "sub", "mul.lo"])
def test_int_arith_bigint(op, ty):
    w = int(ty[1:])
    kind = "u" if w == 32 else "w"
    a, b = int_operands(20, w), int_operands(21, w)
    got = run_op(f"k_{op.replace('.', '')}{ty}", f"{op}.{ty}", kind * 2, kind, a, b)
    mask = (1 << w) - 1
    assert got == [INT_BINARY[op](x, y, w) & mask for x, y in zip(a, b)]


@pytest.mark.parametrize("ty", ["u32", "s32", "u64", "s64"])
def test_mad_lo_bigint(ty):
    w = int(ty[1:])
    kind = "u" if w == 32 else "w"
    a, b, c = int_operands(22, w), int_operands(23, w), int_operands(24, w)
    got = run_op(f"k_mad{ty}", f"mad.lo.{ty}", kind * 3, kind, a, b, c)
    mask = (1 << w) - 1
    assert got == [(x * y + z) & mask for x, y, z in zip(a, b, c)]


@pytest.mark.parametrize("ty", ["b32", "b64"])
@pytest.mark.parametrize("op", ["and", "or", "xor"])
def test_logic_bigint(op, ty):
    w = int(ty[1:])
    kind = "u" if w == 32 else "w"
    a, b = int_operands(25, w), int_operands(26, w)
    got = run_op(f"k_{op}{ty}", f"{op}.{ty}", kind * 2, kind, a, b)
    f = {"and": lambda x, y: x & y, "or": lambda x, y: x | y, "xor": lambda x, y: x ^ y}[op]
    assert got == [f(x, y) for x, y in zip(a, b)]


@pytest.mark.parametrize("op,ty", [("shl", "b32"), ("shl", "b64"), ("shr", "b32"), ("shr", "u32"),
                                   ("shr", "s32"), ("shr", "b64"), ("shr", "u64"), ("shr", "s64")])
def test_shifts_clamp(op, ty):
    """PTX ISA: shift amounts at or above the width give 0 (logical) or the
    sign fill (arithmetic); the amount is an unsigned 32-bit operand."""
    w = int(ty[1:])
    kind = "u" if w == 32 else "w"
    a = int_operands(27, w)
    b = [random.Random(28 + i).choice([0, 1, 5, w - 1, w, w + 1, 100, 0xFFFFFFFF, random.Random(i).getrandbits(32)])
         for i in range(N)]
    got = run_op(f"k_{op}{ty}", f"{op}.{ty}", kind + "u", kind, a, b)
    mask = (1 << w) - 1
    for x, s, g in zip(a, b, got):
        if op == "shl":
            want = 0 if s >= w else (x << s) & mask
        elif ty.startswith("s"):
            v = sx(x, w)
            want = (-1 if v < 0 else 0) & mask if s >= w else (v >> s) & mask
        else:
            want = 0 if s >= w else x >> s
        assert g == want, (op, ty, hex(x), s, hex(g), hex(want))


@pytest.mark.parametrize("ty", ["u32", "s32", "u64", "s64"])
@pytest.mark.parametrize("cmp", ["eq", "ne", "lt", "le", "gt", "ge"])
def test_setp_int(cmp, ty):
    w = int(ty[1:])
    kind = "u" if w == 32 else "w"
    a = int_operands(30, w)
    b = int_operands(31, w)
    b[: N // 4] = a[: N // 4]  # plenty of equal pairs
    got = run_op(f"k_setp{cmp}{ty}", f"setp.{cmp}.{ty}", kind * 2, "p", a, b)
    conv = (lambda v: sx(v, w)) if ty[0] == "s" else (lambda v: v)
    ops = {"eq": lambda x, y: x == y, "ne": lambda x, y: x != y, "lt": lambda x, y: x < y,
           "le": lambda x, y: x <= y, "gt": lambda x, y: x > y, "ge": lambda x, y: x >= y}
    assert got == [int(ops[cmp](conv(x), conv(y))) for x, y in zip(a, b)]


@pytest.mark.parametrize("cmp,ref", [("lo", "lt"), ("ls", "le"), ("hi", "gt"), ("hs", "ge")])
def test_setp_unsigned_names(cmp, ref):
    a, b = int_operands(32, 32), int_operands(33, 32)
    got = run_op(f"k_setp{cmp}", f"setp.{cmp}.u32", "uu", "p", a, b)
    ops = {"lt": lambda x, y: x < y, "le": lambda x, y: x <= y, "gt": lambda x, y: x > y, "ge": lambda x, y: x >= y}
    assert got == [int(ops[ref](x, y)) for x, y in zip(a, b)]


def test_selp_and_pred_logic():
    a, b = int_operands(34, 32), int_operands(35, 32)
    p = [random.Random(36).getrandbits(1) for _ in range(N)]
    got = run_op("k_selp", "selp.u32", "uup", "u", a, b, p)
    assert got == [x if c else y for x, y, c in zip(a, b, p)]
    p1 = [random.Random(37 + i).getrandbits(1) for i in range(N)]
    p2 = [random.Random(900 + i).getrandbits(1) for i in range(N)]
    for op, f in (("and", lambda x, y: x & y), ("or", lambda x, y: x | y), ("xor", lambda x, y: x ^ y)):
        got = run_op(f"k_{op}pred", f"{op}.pred", "pp", "p", p1, p2)
        assert got == [f(x, y) for x, y in zip(p1, p2)]


def test_integer_immediates_truncate():
    a = int_operands(38, 32)
    got = run_op("k_addneg", "add.u32", "ui", "u", a, imm="-5")
    assert got == [(x - 5) & M32 for x in a]
    got = run_op("k_addhex", "add.s64", "wi", "w", int_operands(39, 64), imm="0xFFFFFFFFFFFFFFF0")
    assert got == [(x + 0xFFFFFFFFFFFFFFF0) & M64 for x in int_operands(39, 64)]


# ------------------------------------------------------------------ cvt ----

@pytest.mark.parametrize("src", ["u32", "s32", "u64", "s64"])
def test_cvt_int_to_f32_exact(src):
    w = int(src[1:])
    a = int_operands(40, w)
    rng = random.Random(41)
    a[:64] = [rng.getrandbits(rng.randrange(1, w + 1)) for _ in range(64)]
    got = run_op(f"k_cvtf{src}", f"cvt.rn.f32.{src}", "u" if w == 32 else "w", "f", a)
    conv = (lambda v: sx(v, w)) if src[0] == "s" else (lambda v: v)
    assert got == [X.int_to_f32(conv(x)) for x in a]


@pytest.mark.parametrize("dst", ["u32", "s32", "u64", "s64"])
@pytest.mark.parametrize("mode", ["rni", "rzi", "rmi", "rpi"])
def test_cvt_f32_to_int_saturates(mode, dst):
    w = int(dst[1:])
    a = f32_operands(42)
    rng = random.Random(43)
    for i in range(64):  # values near integers and halfway points
        a[i] = X.f32_bits(rng.randrange(-40, 40) + rng.choice([0.0, 0.5, -0.5, 0.25, 0.75]))
    got = run_op(f"k_cvt{mode}{dst}", f"cvt.{mode}.{dst}.f32", "f", "u" if w == 32 else "w", a)
    assert got == [X.f32_to_int(x, mode, w, dst[0] == "s") for x in a]


@pytest.mark.parametrize("dst,src", [("u64", "u32"), ("s64", "s32"), ("u64", "s32"), ("s64", "u32"),
                                     ("u32", "u64"), ("s32", "s64"), ("u32", "s32"), ("s32", "u32")])
def test_cvt_int_to_int(dst, src):
    ws, wd = int(src[1:]), int(dst[1:])
    a = int_operands(44, ws)
    got = run_op(f"k_cvt{dst}{src}", f"cvt.{dst}.{src}", "u" if ws == 32 else "w", "u" if wd == 32 else "w", a)
    want = [(sx(x, ws) if src[0] == "s" else x) & ((1 << wd) - 1) for x in a]
    assert got == want


def test_mov_special_registers():
    """%tid.x is the thread's index in its CTA (not the lane), %laneid the lane."""
    from simt_ptx_interpretation_gb300 import workloads as wl
    ptx = wl.HEADER + """.visible .entry sp(.param .u64 o)
{
    .reg .b32 %r<8>;
    .reg .b64 %rd<6>;
    ld.param.u64 %rd1, [o];
    mov.u32 %r1, %tid.x;
    mov.u32 %r2, %ntid.x;
    mov.u32 %r3, %ctaid.x;
    mov.u32 %r4, %nctaid.x;
    mov.u32 %r5, %laneid;
    mov.u32 %r6, %tid.y;
    mad.lo.u32 %r7, %r3, %r2, %r1;
    cvt.u64.u32 %rd2, %r7;
    shl.b64 %rd2, %rd2, 4;
    add.s64 %rd3, %rd1, %rd2;
    st.global.u32 [%rd3], %r1;
    st.global.u32 [%rd3+4], %r4;
    st.global.u32 [%rd3+8], %r5;
    st.global.u32 [%rd3+12], %r6;
    ret;
}
"""
    grid, block = 3, 96
    out = np.zeros(grid * block * 4, dtype=np.uint32)
    r = oracle.run(ptx, "sp", grid, block, struct.pack("<Q", 0x10000000), [(0x10000000, out)])
    assert r.status == 0
    o = out.reshape(-1, 4)
    g = np.arange(grid * block)
    assert np.array_equal(o[:, 0], g % block)
    assert np.all(o[:, 1] == grid)
    assert np.array_equal(o[:, 2], g % 32)
    assert np.all(o[:, 3] == 0)
