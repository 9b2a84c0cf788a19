"""Generate interp_asm.cuh: the compute-op interpreter loop as inline PTX.

For S slots of V 32-bit elements per thread, the loop reads a program word
from constant memory, jumps through a brx.idx table indexed by the word's
case number (the fused encoding of cmd_internal.h) and updates the
destination slot's registers in place. The slots are the asm's "+r"
operands, so each case names its registers directly and the dispatch moves
no data. A store or end word leaves the loop and is returned to the caller,
which performs the store in C++ and re-enters at the next word.

Division (int32, and binary32 rounded to nearest) takes a long instruction
sequence per element, so it is not expanded in every (dst, src) case: for each element the case copies the two
operands into a pair of staging registers, records a return-site number and
branches to one shared body, which returns through a second jump table to
the site, where the quotient is moved into the destination register. One
element at a time keeps only two staging registers live beside the slots
(no spills), and one shared body keeps the generated code small.

Comparisons and selects read the staging slot X (the tier's last slot,
filled by the word before): `d = d rel X`, `d = d rel scalar`,
`d = X != 0 ? d : s` and `d = X != 0 ? d : scalar`, S cases each.

Division by a scalar has its own cases: constants the host derives per
launch (a reciprocal, or a multiply-high constant and shift) replace the
division for a warp whose elements all lie in range; otherwise the warp
branches to the general scalar-division case.

Each tier is emitted twice: the extended variant has the division,
comparison and select cases; in the base variant those cases exit like the
end word, so its loop carries none of their code (the host runs a program
on the base variant only when it has none of them).

The wide tiers (16 and 32 slots, the wide encoding of cmd_internal.h) are
emitted once each (gen_wide): a fused table would need S^2 cases per op
(for 16 slots about 7000, which took minutes to compile), so each word
takes two jumps, the first on the source slot (copying it, or a broadcast
scalar, into V staging registers), the second on (op, destination). Only
the arithmetic, min/max and unary words run there; every other word leaves
the loop for the caller.

Run: python gen_interp.py  (writes interp_asm.cuh next to this file)
"""
from __future__ import annotations

import os

HERE = os.path.dirname(os.path.abspath(__file__))
OUT = os.path.join(HERE, "interp_asm.cuh")

TIERS = [(2, 8), (2, 16), (4, 8), (4, 16), (8, 8), (8, 4)]

N_BIN = 16
N_UN = 7
N_ST = 5   # store types (f32, f16, bf16, i32, packed bits)

# Binary ops d = d (op) x, in BinOp order of cmd_internal.h. A string is an
# inline body ("{d}" destination, "{x}" source); a tuple ("staged", name,
# reversed) goes through the shared body `name` with operands (d, x), or
# (x, d) when reversed.
BIN = [
    "add.rn.f32 {d}, {d}, {x};",
    "sub.rn.f32 {d}, {d}, {x};",
    "sub.rn.f32 {d}, {x}, {d};",
    "mul.rn.f32 {d}, {d}, {x};",
    "add.u32 {d}, {d}, {x};",
    "sub.u32 {d}, {d}, {x};",
    "sub.u32 {d}, {x}, {d};",
    "mul.lo.u32 {d}, {d}, {x};",
    ("staged", "fdiv", False),
    ("staged", "fdiv", True),
    ("staged", "idiv", False),
    ("staged", "idiv", True),
    # IEEE minimumNumber / maximumNumber: min.f32 / max.f32 without .ftz
    # return the number when one operand is NaN and order -0 below +0
    "min.f32 {d}, {d}, {x};",
    "max.f32 {d}, {d}, {x};",
    "min.s32 {d}, {d}, {x};",
    "max.s32 {d}, {d}, {x};",
]
assert len(BIN) == N_BIN

# Unary ops d = f(x), in UnOp order.
UN = [
    "xor.b32 {d}, {x}, 0x80000000;",
    "neg.s32 {d}, {x};",
    "mov.b32 {d}, {x};",
    "and.b32 {d}, {x}, 0x7fffffff;",
    # |x| modulo 2^32: (x ^ s) - s with s = x >> 31 (arithmetic)
    "shr.s32 %%t, {x}, 31; xor.b32 {d}, {x}, %%t; sub.s32 {d}, {d}, %%t;",
    "cvt.rn.f32.s32 {d}, {x};",
    # truncation toward zero; the conversion saturates and maps NaN to 0
    "cvt.rzi.s32.f32 {d}, {x};",
]
assert len(UN) == N_UN

# Comparisons d = (d rel x) ? 1 : 0, in CmpOp order: float (ordered, so false
# on NaN, except ne, which is the unordered-or-not-equal test and so true on
# NaN: the IEEE != ), signed int, unsigned int.
CMP = [f"{rel}.f32" for rel in ("lt", "le", "gt", "ge", "eq", "neu")] + \
      [f"{rel}.s32" for rel in ("lt", "le", "gt", "ge", "eq", "ne")] + \
      [f"{rel}.u32" for rel in ("lt", "le", "gt", "ge")]
N_CMP = len(CMP)
assert N_CMP == 16


def staged_body(name: str) -> str:
    """Result in %%xa from operands %%xa, %%xb (one element)."""
    if name == "fdiv":
        # IEEE binary32 division, rounded once to nearest even
        return "div.rn.f32 %%xa, %%xa, %%xb;"
    assert name == "idiv"
    # truncating division; b == 0 gives -1 and b == -1 gives 0 - a (which
    # wraps INT_MIN onto itself); the divide itself never sees 0 or -1
    return ("setp.eq.s32 %%p0, %%xb, 0; setp.eq.s32 %%p1, %%xb, -1; "
            "selp.b32 %%t, 1, %%xb, %%p0; selp.b32 %%t, 1, %%t, %%p1; "
            "div.s32 %%t, %%xa, %%t; neg.s32 %%xb, %%xa; selp.b32 %%t, %%xb, %%t, %%p1; "
            "selp.b32 %%xa, -1, %%t, %%p0;")


def gen_tier(S: int, V: int, ext: bool) -> str:
    def reg(i, v):
        return f"%{i * V + v}"

    end = (N_BIN + N_UN) * S * S + (N_BIN + 1 + N_ST) * S
    n_cases = end + 1 + 2 * N_CMP * S + S * S + S + 2 * S
    X = S - 1  # the staging slot compares and selects read
    slot_ops = S * V
    o_idx = slot_ops        # "+r" program index (words)
    o_word = slot_ops + 1   # "=r" the word that left the loop
    o_prog = slot_ops + 2   # "l" generic address of the program
    o_scal = slot_ops + 3   # "l" generic address of the scalar array
    load_k = f"shr.u32 %%aux, %%wc, 16; mad.wide.u32 %%sa, %%aux, 4, %{o_scal}; ld.u32 %%k, [%%sa];"

    labels, bodies = [], []
    staged_used = set()
    ret_sites = []

    def staged_case(name, rev, d, src_regs):
        """Per element: stage (d, x) (or (x, d) when reversed), branch to the
        shared body and take the result back at this element's site."""
        staged_used.add(name)
        parts = []
        for v in range(V):
            first, second = (src_regs[v], reg(d, v)) if rev else (reg(d, v), src_regs[v])
            site = len(ret_sites)
            ret_sites.append(f"$LR{site}")
            parts.append(f"mov.b32 %%xa, {first}; mov.b32 %%xb, {second}; mov.u32 %%rd, {site}; "
                         f"bra.uni $Lbody_{name}; $LR{site}: mov.b32 {reg(d, v)}, %%xa;")
        return " ".join(parts) + " bra.uni $Lloop;"

    # binary slot-slot
    for b in range(N_BIN):
        for d in range(S):
            for s in range(S):
                lab = f"$LB{b}_{d}_{s}"
                labels.append(lab)
                op = BIN[b]
                if isinstance(op, tuple) and not ext:
                    labels[-1] = "$Lexit"
                    continue
                if isinstance(op, tuple):
                    body = staged_case(op[1], op[2], d, [reg(s, v) for v in range(V)])
                else:
                    body = " ".join(op.format(d=reg(d, v), x=reg(s, v)) for v in range(V)) + " bra.uni $Lloop;"
                bodies.append(f"{lab}: {body}")
    # unary
    for u in range(N_UN):
        for d in range(S):
            for s in range(S):
                lab = f"$LU{u}_{d}_{s}"
                labels.append(lab)
                if u == 2 and d == s:
                    bodies.append(f"{lab}: bra.uni $Lloop;")
                else:
                    ops = " ".join(UN[u].format(d=reg(d, v), x=reg(s, v)) for v in range(V))
                    bodies.append(f"{lab}: {ops} bra.uni $Lloop;")
    # binary with scalar source
    for b in range(N_BIN):
        for d in range(S):
            lab = f"$LS{b}_{d}"
            labels.append(lab)
            op = BIN[b]
            if isinstance(op, tuple) and not ext:
                labels[-1] = "$Lexit"
                continue
            if isinstance(op, tuple):
                body = load_k + " " + staged_case(op[1], op[2], d, ["%%k"] * V)
            else:
                body = load_k + " " + " ".join(op.format(d=reg(d, v), x="%%k") for v in range(V)) + \
                    " bra.uni $Lloop;"
            bodies.append(f"{lab}: {body}")
    # broadcast scalar
    for d in range(S):
        lab = f"$LM{d}"
        labels.append(lab)
        ops = " ".join(f"mov.b32 {reg(d, v)}, %%k;" for v in range(V))
        bodies.append(f"{lab}: {load_k} {ops} bra.uni $Lloop;")
    # stores and end leave the loop
    labels += ["$Lexit"] * (N_ST * S + 1)
    # comparisons with the staging slot, then with a scalar; selects on the
    # staging slot with a slot, then with a scalar. An op that reads the
    # staging slot never has it as destination or source (the lowering keeps
    # it free): those cases exit, and the host encoder never emits them.
    for c in range(N_CMP):
        for d in range(S):
            if d == X or not ext:
                labels.append("$Lexit")
                continue
            lab = f"$LCX{c}_{d}"
            labels.append(lab)
            ops = " ".join(f"setp.{CMP[c]} %%p0, {reg(d, v)}, {reg(X, v)}; selp.u32 {reg(d, v)}, 1, 0, %%p0;"
                           for v in range(V))
            bodies.append(f"{lab}: {ops} bra.uni $Lloop;")
    for c in range(N_CMP):
        for d in range(S):  # (no staging slot read: every destination is valid)
            if not ext:
                labels.append("$Lexit")
                continue
            lab = f"$LCS{c}_{d}"
            labels.append(lab)
            ops = " ".join(f"setp.{CMP[c]} %%p0, {reg(d, v)}, %%k; selp.u32 {reg(d, v)}, 1, 0, %%p0;"
                           for v in range(V))
            bodies.append(f"{lab}: {load_k} {ops} bra.uni $Lloop;")
    for d in range(S):
        for s_ in range(S):
            if d == X or s_ == X or not ext:
                labels.append("$Lexit")
                continue
            lab = f"$LSEL{d}_{s_}"
            labels.append(lab)
            ops = " ".join(f"setp.ne.u32 %%p0, {reg(X, v)}, 0; selp.b32 {reg(d, v)}, {reg(d, v)}, {reg(s_, v)}, %%p0;"
                           for v in range(V))
            bodies.append(f"{lab}: {ops} bra.uni $Lloop;")
    for d in range(S):
        if d == X or not ext:
            labels.append("$Lexit")
            continue
        lab = f"$LSELS{d}"
        labels.append(lab)
        ops = " ".join(f"setp.ne.u32 %%p0, {reg(X, v)}, 0; selp.b32 {reg(d, v)}, {reg(d, v)}, %%k, %%p0;"
                       for v in range(V))
        bodies.append(f"{lab}: {load_k} {ops} bra.uni $Lloop;")
    # division of d by a scalar through constants the host derives at launch
    # (scalars aux, aux + 1, aux + 2): the whole warp takes the fast sequence
    # or, when any of its elements (or the divisor) is outside its range, the
    # general scalar-division case of the same destination, which reads the
    # divisor at aux
    for o in range(2):
        for d in range(S):
            if not ext:
                labels.append("$Lexit")
                continue
            lab = f"$LSD{o}_{d}"
            labels.append(lab)
            head = f"shr.u32 %%aux, %%wc, 16; mad.wide.u32 %%sa, %%aux, 4, %{o_scal};"
            if o == 0:
                # binary32: q0 = x r, then twice q += (x - q s) r with the
                # residual formed exactly by an FMA (r = RN(1/s), Markstein)
                parts = [head, "ld.u32 %%k, [%%sa]; ld.u32 %%t, [%%sa+4]; setp.ne.b32 %%p1, %%t, 0;"]
                for v in range(V):
                    x = reg(d, v)
                    parts.append(f"abs.f32 %%xa, {x}; setp.ge.f32 %%p0, %%xa, 0f21800000; and.pred %%p1, %%p1, %%p0; "
                                 f"setp.le.f32 %%p0, %%xa, 0f5D800000; and.pred %%p1, %%p1, %%p0;")
                parts.append(f"activemask.b32 %%aux; vote.sync.all.pred %%p1, %%p1, %%aux; @!%%p1 bra.uni $LS8_{d};")
                for v in range(V):
                    x = reg(d, v)
                    parts.append(f"mul.rn.f32 %%xa, {x}, %%t; neg.f32 %%xb, %%xa; fma.rn.f32 %%xb, %%xb, %%k, {x}; "
                                 f"fma.rn.f32 %%xa, %%xb, %%t, %%xa; neg.f32 %%xb, %%xa; fma.rn.f32 %%xb, %%xb, %%k, {x}; "
                                 f"fma.rn.f32 {x}, %%xb, %%t, %%xa;")
            else:
                # int32 (Granlund and Montgomery, signed, truncating): q =
                # ((((n + mulhi(m, n)) >> sh) - (n >> 31)) ^ ds) - ds, ds = d >> 31
                parts = [head, f"ld.u32 %%t, [%%sa+8]; setp.lt.s32 %%p1, %%t, 0; @%%p1 bra.uni $LS10_{d};",
                         "ld.u32 %%k, [%%sa+4]; ld.u32 %%rd, [%%sa]; shr.s32 %%rd, %%rd, 31;"]
                for v in range(V):
                    x = reg(d, v)
                    parts.append(f"mul.hi.s32 %%xa, {x}, %%k; add.s32 %%xa, %%xa, {x}; shr.s32 %%xa, %%xa, %%t; "
                                 f"shr.s32 %%xb, {x}, 31; sub.s32 %%xa, %%xa, %%xb; xor.b32 %%xa, %%xa, %%rd; "
                                 f"sub.s32 {x}, %%xa, %%rd;")
            bodies.append(f"{lab}: " + " ".join(parts) + " bra.uni $Lloop;")
    # the table is padded to a power of two with exits so that masking the
    # case number keeps every jump inside it
    assert len(labels) == n_cases
    size = 1
    while size < n_cases:
        size *= 2
    labels += ["$Lexit"] * (size - n_cases)

    # shared bodies of the staged ops; they return through the site table
    for name in sorted(staged_used):
        bodies.append(f"$Lbody_{name}: {staged_body(name)} brx.idx.uni %%rd, $Lret;")

    lines = ["{"]
    lines.append(".reg .b32 %%w, %%wc, %%c, %%aux, %%k, %%t, %%rd, %%xa, %%xb;")
    lines.append(".reg .b64 %%cbase, %%ca, %%sa;")
    lines.append(".reg .pred %%p0, %%p1;")
    tbl = []
    for i in range(0, len(labels), 16):
        tbl.append(", ".join(labels[i:i + 16]))
    lines.append("$Ltable: .branchtargets " + ",\n".join(tbl) + ";")
    if ret_sites:
        lines.append("$Lret: .branchtargets " + ",\n".join(
            ", ".join(ret_sites[i:i + 16]) for i in range(0, len(ret_sites), 16)) + ";")
    lines.append(f"cvta.to.const.u64 %%cbase, %{o_prog};")
    lines.append(f"mad.wide.u32 %%ca, %{o_idx}, 4, %%cbase;")
    lines.append("ld.const.u32 %%w, [%%ca];")
    lines.append("$Lloop:")
    # the case number, masked to the table; the next word is fetched while
    # this one's case runs (the host keeps every program shorter than its
    # constant-memory row, so that read stays inside the row)
    lines.append(f"and.b32 %%c, %%w, {size - 1};")
    lines.append("mov.b32 %%wc, %%w;")
    lines.append("add.u64 %%ca, %%ca, 4;")
    lines.append("ld.const.u32 %%w, [%%ca];")
    lines.append("brx.idx.uni %%c, $Ltable;")
    lines += bodies
    lines.append("$Lexit:")
    lines.append(f"mov.b32 %{o_word}, %%wc;")
    # the index of the word after the one that left the loop
    lines.append("sub.u64 %%ca, %%ca, %%cbase;")
    lines.append(f"cvt.u32.u64 %{o_idx}, %%ca;")
    lines.append(f"shr.u32 %{o_idx}, %{o_idx}, 2;")
    lines.append("}")
    asm = "\n".join(lines)

    def cstr(text):
        out = []
        for ln in text.split("\n"):
            out.append('    "' + ln.replace("\\", "\\\\").replace('"', '\\"') + '\\n"')
        return "\n".join(out)

    outs = ", ".join(f'"+r"(r[{i}][{v}])' for i in range(S) for v in range(V))
    return f"""
template <>
struct AsmInterp<{S}, {V}, {"true" if ext else "false"}> {{
  // Run compute words from prog[idx] on; return the first store or end word
  // (idx then points past it).{"" if ext else " Extended words (division, comparison, select) are not in this variant: they leave the loop like an end word."}
  static __device__ __forceinline__ uint32_t run(uint32_t (&r)[{S}][{V}], uint32_t& idx, const uint32_t* prog,
                                                 const uint32_t* scal) {{
    uint32_t word;
    asm volatile(
{cstr(asm)}
        : {outs}, "+r"(idx), "=r"(word)
        : "l"(prog), "l"(scal)
        : "memory");
    return word;
  }}
}};
"""


# Kinds of the wide encoding (cmd_internal.h WideKind): binary ops at
# 0 .. N_BIN - 1, unary ops at N_BIN .. N_BIN + N_UN - 1; everything from
# N_BIN + N_UN on (stores, end, comparisons, select, division by a scalar)
# and the staged binary ops leave the loop.
W_BASE_KINDS = N_BIN + N_UN
W_SCALAR = 0x40


def gen_wide(S: int, V: int) -> str:
    """A wide tier (16 or 32 slots): word = kind << 24 | d << 16 | s << 8 |
    aux. The source operand (slot s, or scalar aux when the kind has the
    scalar flag) is copied into V staging registers by a first jump table on
    s; a second table on (kind, d) applies the op to the destination's
    registers. Words this loop does not run leave it and are returned to the
    caller."""

    def reg(i, v):
        return f"%{i * V + v}"

    slot_ops = S * V
    o_idx, o_word, o_prog, o_scal = slot_ops, slot_ops + 1, slot_ops + 2, slot_ops + 3
    xs = [f"%%x{v}" for v in range(V)]
    fetch_labels, fetch_bodies = [], []
    for s in range(S):
        lab = f"$LF{s}"
        fetch_labels.append(lab)
        fetch_bodies.append(f"{lab}: " + " ".join(f"mov.b32 {xs[v]}, {reg(s, v)};" for v in range(V)) +
                            " bra.uni $Lop;")
    op_labels, op_bodies = [], []
    for kind in range(W_BASE_KINDS):
        for d in range(S):
            if kind < N_BIN:
                op = BIN[kind]
                if isinstance(op, tuple):
                    op_labels.append("$Lexit")
                    continue
                body = " ".join(op.format(d=reg(d, v), x=xs[v]) for v in range(V))
            else:
                u = kind - N_BIN
                body = " ".join(UN[u].format(d=reg(d, v), x=xs[v]) for v in range(V))
            lab = f"$LO{kind}_{d}"
            op_labels.append(lab)
            op_bodies.append(f"{lab}: {body} bra.uni $Lloop;")

    def table(name, labels):
        return f"{name}: .branchtargets " + ",\n".join(
            ", ".join(labels[i:i + 16]) for i in range(0, len(labels), 16)) + ";"

    lines = ["{"]
    lines.append(".reg .b32 %%w, %%wc, %%c, %%kd, %%aux, %%k, %%t, " + ", ".join(xs) + ";")
    lines.append(".reg .b64 %%cbase, %%ca, %%sa;")
    lines.append(".reg .pred %%p0;")
    lines.append(table("$Lfetch", fetch_labels))
    lines.append(table("$Lops", op_labels))
    lines.append(f"cvta.to.const.u64 %%cbase, %{o_prog};")
    lines.append(f"mad.wide.u32 %%ca, %{o_idx}, 4, %%cbase;")
    lines.append("ld.const.u32 %%w, [%%ca];")
    lines.append("$Lloop:")
    lines.append("mov.b32 %%wc, %%w;")
    lines.append("add.u64 %%ca, %%ca, 4;")
    lines.append("ld.const.u32 %%w, [%%ca];")
    # kind without the scalar flag; kinds past the unary ops leave the loop
    lines.append("shr.u32 %%kd, %%wc, 24;")
    lines.append(f"and.b32 %%c, %%kd, {W_SCALAR - 1};")
    lines.append(f"setp.ge.u32 %%p0, %%c, {W_BASE_KINDS};")
    lines.append("@%%p0 bra.uni $Lexit;")
    lines.append(f"and.b32 %%t, %%kd, {W_SCALAR};")
    lines.append("setp.ne.u32 %%p0, %%t, 0;")
    lines.append("@%%p0 bra.uni $Lscalar;")
    lines.append("bfe.u32 %%t, %%wc, 8, 8;")
    lines.append("brx.idx.uni %%t, $Lfetch;")
    lines += fetch_bodies
    lines.append(f"$Lscalar: and.b32 %%aux, %%wc, 255; mad.wide.u32 %%sa, %%aux, 4, %{o_scal}; ld.u32 %%k, [%%sa]; " +
                 " ".join(f"mov.b32 {xs[v]}, %%k;" for v in range(V)))
    lines.append("$Lop:")
    lines.append("bfe.u32 %%t, %%wc, 16, 8;")
    lines.append(f"mad.lo.u32 %%t, %%c, {S}, %%t;")
    lines.append("brx.idx.uni %%t, $Lops;")
    lines += op_bodies
    lines.append("$Lexit:")
    lines.append(f"mov.b32 %{o_word}, %%wc;")
    lines.append("sub.u64 %%ca, %%ca, %%cbase;")
    lines.append(f"cvt.u32.u64 %{o_idx}, %%ca;")
    lines.append(f"shr.u32 %{o_idx}, %{o_idx}, 2;")
    lines.append("}")
    asm = "\n".join(lines)
    out_lines = []
    for ln in asm.split("\n"):
        out_lines.append('    "' + ln.replace("\\", "\\\\").replace('"', '\\"') + '\\n"')
    outs = ", ".join(f'"+r"(r[{i}][{v}])' for i in range(S) for v in range(V))
    return f"""
template <>
struct AsmWide<{S}, {V}> {{
  // Run the arithmetic, min/max and unary words from prog[idx] on; return
  // the first other word (a store, the end, a division, comparison or
  // select), with idx pointing past it.
  static __device__ __forceinline__ uint32_t run(uint32_t (&r)[{S}][{V}], uint32_t& idx, const uint32_t* prog,
                                                 const uint32_t* scal) {{
    uint32_t word;
    asm volatile(
{chr(10).join(out_lines)}
        : {outs}, "+r"(idx), "=r"(word)
        : "l"(prog), "l"(scal)
        : "memory");
    return word;
  }}
}};
"""


WIDE = [(32, 2), (16, 4)]


def main():
    parts = [
        "// interp_asm.cuh - GENERATED by gen_interp.py; do not edit by hand.\n"
        "// The compute-op interpreter loop as inline PTX for each fused tier.\n"
        "#pragma once\n\n#include <cstdint>\n\nnamespace cmdx {\n\n"
        "// EXT selects the variant with the extended ops (division, comparisons,\n"
        "// select); programs without them run the base variant, whose loop\n"
        "// carries none of their code.\n"
        "template <int S, int V, bool EXT>\nstruct AsmInterp;\n"
    ]
    for S, V in TIERS:
        for ext in (False, True):
            parts.append(gen_tier(S, V, ext))
    parts.append("\n// The loop of a wide tier of S slots, V elements per slot.\n"
                 "template <int S, int V>\nstruct AsmWide;\n")
    for S, V in WIDE:
        parts.append(gen_wide(S, V))
    parts.append("\n}  // namespace cmdx\n")
    with open(OUT, "w") as f:
        f.write("".join(parts))
    print(OUT)


if __name__ == "__main__":
    main()
