"""Planted mistakes: each is a plausible error in the oracle, compiled from a
patched copy of ``oracle.c`` on the CPU; the pins must catch every one.

This shows that the pins are strong enough that the oracle cannot drift
from the pages' arithmetic unnoticed.
"""
import os

import numpy as np
import pytest

import oracle
from tests.libcasts import lib_reduce, lib_round, lib_widen, mismatches
from tests.test_oracle_casts import _golden_rows
from tests.test_oracle_fold import edgy_f32

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    "fold starts from zero": (
        "float acc = wire_operand(dst_dtype, wire_dtype, srcs[0], i);",
        "float acc = 0.0f + wire_operand(dst_dtype, wire_dtype, srcs[0], i);"),
    "rank 0 skips the wire cast": (
        "float acc = wire_operand(dst_dtype, wire_dtype, srcs[0], i);",
        "float acc = orc_widen(dst_dtype, load_bits(dst_dtype, srcs[0], i));"),
    "fold in descending rank order": (
        "float acc = wire_operand(dst_dtype, wire_dtype, srcs[0], i);\n"
        "        for (int r = 1; r < R; ++r) {\n"
        "            acc = acc + wire_operand(dst_dtype, wire_dtype, srcs[r], i);",
        "float acc = wire_operand(dst_dtype, wire_dtype, srcs[R - 1], i);\n"
        "        for (int r = R - 2; r >= 0; --r) {\n"
        "            acc = acc + wire_operand(dst_dtype, wire_dtype, srcs[r], i);"),
    "accumulates in double": (
        "float acc = wire_operand(dst_dtype, wire_dtype, srcs[0], i);",
        "double acc = wire_operand(dst_dtype, wire_dtype, srcs[0], i);"),
    "ties round up": (
        "r = (fmod(below, 2.0) == 0.0) ? below : below + 1.0;",
        "r = below + 1.0;"),
    "ties round down": (
        "r = (fmod(below, 2.0) == 0.0) ? below : below + 1.0;",
        "r = below;"),
    "flushes subnormals": (
        "if (e < f->emin) e = f->emin;",
        "if (e < f->emin) return sign;"),
    "overflow one binade late": (
        "if (y >= ldexp(1.0, f->emax + 1)) return sign | exp_all_ones;",
        "if (y >= ldexp(1.0, f->emax + 2)) return sign | exp_all_ones;"),
    "f16 precision off by one": (
        "static const orc_format FMT_F16 = {11, -14, 15, 5};",
        "static const orc_format FMT_F16 = {10, -14, 15, 5};"),
    "bf16 bias off by one": (
        "static const orc_format FMT_BF16 = {8, -126, 127, 8};",
        "static const orc_format FMT_BF16 = {8, -126, 126, 8};"),
    "widen drops the sign": (
        "return negative ? -v : v;",
        "return v;"),
    "only the first destination is written": (
        "for (int d = 0; d < n_dsts; ++d) store_bits(dst_dtype, dsts[d], i, y);",
        "for (int d = 0; d < 1; ++d) store_bits(dst_dtype, dsts[d], i, y);"),
    "inactive rank omitted instead of +0": (
        "w = orc_widen(wire_dtype, orc_round(wire_dtype, 0.0f));",
        "continue;"),
    "residual rounded through the wire": (
        "acc = acc + orc_widen(dst_dtype, load_bits_at(dst_dtype, residual, off, i));",
        "acc = acc + orc_widen(wire_dtype, orc_round(wire_dtype, orc_widen(dst_dtype, load_bits_at(dst_dtype, residual, off, i))));"),
    "residual added before the ranks": (
        "acc = (r == 0) ? w : acc + w;",
        "acc = (r == 0) ? (residual ? orc_widen(dst_dtype, load_bits_at(dst_dtype, residual, (long long)j * residual_stride, i)) + w : w) : acc + w;"),
    "destination stride ignored": (
        "store_bits(dst_dtype, (char *)dsts[d] + (long long)j * stride, i, y);",
        "store_bits(dst_dtype, (char *)dsts[d] + (long long)j * packed + 0 * stride, i, y);"),
    "pack skips the wire cast": (
        "store_bits(wire_dtype, wire, i, orc_round(wire_dtype, v));",
        "store_bits(wire_dtype, wire, i, wire_dtype == ORC_F32 ? orc_round(wire_dtype, v) : orc_round(dst_dtype, v));"),
    "final cast truncates": (
        "const uint32_t y = orc_round(dst_dtype, acc);\n        for (int d = 0; d < n_dsts; ++d) store_bits",
        "uint32_t y = orc_round(dst_dtype, acc);\n"
        "        if (dst_dtype == ORC_BF16) { uint32_t b; memcpy(&b, &acc, 4); y = b >> 16; }\n"
        "        for (int d = 0; d < n_dsts; ++d) store_bits"),
}


def _battery(orc: oracle.Oracle) -> list:
    """Run every pin quickly; return the names of the ones that fail."""
    failed = []
    L = orc.lib
    for kind, name, inp, exp, _ in _golden_rows():
        code = oracle.DTYPES[name]
        if kind == "round":
            got = L.orc_round(code, float(np.array([inp], np.uint32).view(np.float32)[0]))
        else:
            got = int(np.float32(L.orc_widen(code, inp)).view(np.uint32))
        if got != exp:
            failed.append("closed forms")
            break
    rng = np.random.Generator(np.random.PCG64(5))
    for dst in ("f32", "f16", "bf16"):
        for wire in ("f32", "f16", "bf16"):
            srcs = [lib_round(dst, edgy_f32(rng, 4000)) for _ in range(3)]
            if mismatches(orc.reduce(srcs, 1, dst, wire)[0], lib_reduce(srcs, dst, wire), dst).size:
                failed.append(f"library formula {dst}/{wire}")
            x = srcs[0]
            exp = lib_round(dst, lib_widen(wire, lib_round(wire, lib_widen(dst, x))))
            if mismatches(orc.reduce([x], 1, dst, wire)[0], exp, dst).size:
                failed.append(f"R=1 {dst}/{wire}")
    one = [np.array([v], dtype=np.float32) for v in (1e8, 1.0, -1e8)]
    two = [np.array([v], dtype=np.float32) for v in (1e8, -1e8, 1.0)]
    if orc.reduce(one, 1, "f32", "f32")[0][0] != 0.0 or orc.reduce(two, 1, "f32", "f32")[0][0] != 1.0:
        failed.append("rank order")
    z = orc.reduce([np.array([-0.0], np.float32)], 1, "f32", "bf16")[0]
    if int(z.view(np.uint32)[0]) != 0x80000000:
        failed.append("signed zero")
    outs = orc.reduce([lib_round("f32", edgy_f32(rng, 100))] * 2, 3, "f32", "f16")
    if any(mismatches(o, outs[0], "f32").size for o in outs[1:]):
        failed.append("destinations identical")
    failed += _battery_2d(orc, rng)
    return failed


def _battery_2d(orc, rng):
    from tests.test_oracle_2d import embed, extract, lib_fold_f32
    failed = []
    ne0, ne1 = 40, 5
    for dst, wire in (("f32", "bf16"), ("bf16", "f16"), ("f16", "f32")):
        es = 4 if dst == "f32" else 2
        srcs = [lib_round(dst, edgy_f32(rng, ne0 * ne1)) for _ in range(3)]
        flat = orc.reduce(srcs, 1, dst, wire)[0]
        st = ne0 + 3
        emb = [embed(s, ne0, st, 1) for s in srcs]
        out = [embed(np.zeros(ne0 * ne1, dtype=srcs[0].dtype), ne0, st, 2)]
        orc.reduce_2d(emb, 1, dst, wire, ne0, ne1, src_strides=[st * es] * 3, dst_strides=[st * es], out=out)
        if mismatches(extract(out[0], ne0, ne1, st), flat, dst).size:
            failed.append(f"2-D strides {dst}/{wire}")
        zeroed = [srcs[0], np.zeros_like(srcs[1]), srcs[2]]
        got = orc.reduce_2d([srcs[0], None, srcs[2]], 1, dst, wire, ne0 * ne1, 1, inactive=(1,))[0]
        if mismatches(got, orc.reduce(zeroed, 1, dst, wire)[0], dst).size:
            failed.append(f"2-D inactive {dst}/{wire}")
        res = lib_round(dst, edgy_f32(rng, ne0 * ne1))
        got = orc.reduce_2d(srcs, 1, dst, wire, ne0, ne1, residual=res)[0]
        with np.errstate(over="ignore", invalid="ignore"):
            acc = (lib_fold_f32(srcs, dst, wire) + lib_widen(dst, res)).astype(np.float32)
        if mismatches(got, lib_round(dst, acc), dst).size:
            failed.append(f"2-D residual {dst}/{wire}")
        if mismatches(orc.wire_pack(srcs[0], dst, wire), lib_round(wire, lib_widen(dst, srcs[0])), wire).size:
            failed.append(f"pack {dst}/{wire}")
    a = np.array([-0.0, -0.0], dtype=np.float32)
    if orc.reduce_2d([a, None], 1, "f32", "bf16", 2, 1, inactive=(1,))[0].view(np.uint32).tolist() != [0, 0]:
        failed.append("inactive is +0")
    return failed


def test_real_oracle_passes_battery():
    assert _battery(oracle.default()) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name!r} not found exactly once"
    mutated = tmp_path / "oracle_mutant.c"
    mutated.write_text(src.replace(old, new))
    so = oracle.compile_to(str(mutated), str(tmp_path / "liboracle_mutant.so"))
    failed = _battery(oracle.Oracle(so))
    assert failed, f"mutant {name!r} passed every pin"
