"""Generate interp_asm.cuh: the compute-op interpreter loop as inline PTX.

For S slots of V 32-bit elements per thread, the loop reads a program word
from constant memory, jumps through a brx.idx table indexed by the word's
case number (the fused encoding of cmd_internal.h) and updates the
destination slot's registers in place. The slots are the asm's "+r"
operands, so each case names its registers directly and the dispatch moves
no data. A store or end word leaves the loop and is returned to the caller,
which performs the store in C++ and re-enters at the next word.

Run: python gen_interp.py  (writes interp_asm.cuh next to this file)
"""
from __future__ import annotations

import os

HERE = os.path.dirname(os.path.abspath(__file__))
OUT = os.path.join(HERE, "interp_asm.cuh")

TIERS = [(2, 8), (2, 16), (4, 8), (4, 16), (8, 8), (8, 4)]

# binary ops d = d (op) x, in BinOp order; "{d}" destination, "{x}" source
BIN = [
    "add.rn.f32 {d}, {d}, {x};",
    "sub.rn.f32 {d}, {d}, {x};",
    "sub.rn.f32 {d}, {x}, {d};",
    "mul.rn.f32 {d}, {d}, {x};",
    "add.u32 {d}, {d}, {x};",
    "sub.u32 {d}, {d}, {x};",
    "sub.u32 {d}, {x}, {d};",
    "mul.lo.u32 {d}, {d}, {x};",
]
# unary ops d = f(x), in UnOp order
UN = [
    "xor.b32 {d}, {x}, 0x80000000;",
    "neg.s32 {d}, {x};",
    "mov.b32 {d}, {x};",
]


def gen_tier(S: int, V: int) -> str:
    def reg(i, v):
        return f"%{i * V + v}"

    n_bin = 8 * S * S
    n_un = 3 * S * S
    base_bs = 11 * S * S
    base_movs = base_bs + 8 * S
    base_st = base_movs + S
    end = 11 * S * S + 13 * S
    n_cases = end + 1
    slot_ops = S * V
    o_idx = slot_ops        # "+r" program index (words)
    o_word = slot_ops + 1   # "=r" the word that left the loop
    o_prog = slot_ops + 2   # "l" generic address of the program
    o_scal = slot_ops + 3   # "l" generic address of the scalar array

    labels = []
    bodies = []
    # binary slot-slot
    for b in range(8):
        for d in range(S):
            for s in range(S):
                lab = f"$LB{b}_{d}_{s}"
                labels.append(lab)
                ops = " ".join(BIN[b].format(d=reg(d, v), x=reg(s, v)) for v in range(V))
                bodies.append(f"{lab}: {ops} bra.uni $Lloop;")
    # unary
    for u in range(3):
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
    for b in range(8):
        for d in range(S):
            lab = f"$LS{b}_{d}"
            labels.append(lab)
            ops = " ".join(BIN[b].format(d=reg(d, v), x="%%k") for v in range(V))
            bodies.append(f"{lab}: shr.u32 %%aux, %%wc, 16; mad.wide.u32 %%sa, %%aux, 4, %{o_scal}; "
                          f"ld.u32 %%k, [%%sa]; {ops} bra.uni $Lloop;")
    # broadcast scalar
    for d in range(S):
        lab = f"$LM{d}"
        labels.append(lab)
        ops = " ".join(f"mov.b32 {reg(d, v)}, %%k;" for v in range(V))
        bodies.append(f"{lab}: shr.u32 %%aux, %%wc, 16; mad.wide.u32 %%sa, %%aux, 4, %{o_scal}; "
                      f"ld.u32 %%k, [%%sa]; {ops} bra.uni $Lloop;")
    # stores and end leave the loop; the table is padded to a power of two
    # with exits so that masking the case number keeps every jump inside it
    labels += ["$Lexit"] * (4 * S + 1)
    assert len(labels) == n_cases
    size = 1
    while size < n_cases:
        size *= 2
    labels += ["$Lexit"] * (size - n_cases)

    lines = []
    lines.append("{")
    lines.append(".reg .b32 %%w, %%wc, %%c, %%aux, %%k;")
    lines.append(".reg .b64 %%cbase, %%ca, %%sa;")
    # branch table, 16 labels per line
    tbl = []
    for i in range(0, len(labels), 16):
        tbl.append(", ".join(labels[i:i + 16]))
    lines.append("$Ltable: .branchtargets " + ",\n".join(tbl) + ";")
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

    def cstr(s):
        out = []
        for ln in s.split("\n"):
            out.append('    "' + ln.replace("\\", "\\\\").replace('"', '\\"') + '\\n"')
        return "\n".join(out)

    outs = ", ".join(f'"+r"(r[{i}][{v}])' for i in range(S) for v in range(V))
    return f"""
template <>
struct AsmInterp<{S}, {V}> {{
  // Run compute words from prog[idx] on; return the first store or end word
  // (idx then points past it).
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


def main():
    parts = [
        "// interp_asm.cuh - GENERATED by gen_interp.py; do not edit by hand.\n"
        "// The compute-op interpreter loop as inline PTX for each fused tier.\n"
        "#pragma once\n\n#include <cstdint>\n\nnamespace cmdx {\n\n"
        "template <int S, int V>\nstruct AsmInterp;\n"
    ]
    for S, V in TIERS:
        parts.append(gen_tier(S, V))
    parts.append("\n}  // namespace cmdx\n")
    with open(OUT, "w") as f:
        f.write("".join(parts))
    print(OUT)


if __name__ == "__main__":
    main()
