"""Writes norm_rope_rounding.txt: one Q/K head row through the RMSNorm + RoPE
reading of the fused boundary, evaluated in exact rational arithmetic with an
explicit IEEE round-to-nearest-even after every fp32 and bf16 step.

The pages name the Q/K norm + RoPE boundary ("Laguna S 2.1 INT4 -- calibrated
FP8 KV on Intel B70", section "Initial optimization order", item 3) but fix
none of its arithmetic; the reading adopted (and documented with
fp8kv_qk_norm_rope_insert) is, per row x of 128 bf16 values, weights w,
table row (c, s) and eps:

    part_l = fma(x3, x3, fma(x2, x2, fma(x1, x1, x0 * x0)))    x_i = x[4l + i]
    parts summed pairwise: l + (l + 16), then + 8, + 4, + 2, + 1
    r      = 1 / sqrt(ss / 128 + eps)
    y_i    = bf16( bf16(x_i * r) * w_i )
    o_k    = bf16( fma(y_k,      c_k, -(y_k+64 * s_k)) )
    o_k+64 = bf16( fma(y_k+64,   c_k,   y_k    * s_k ) )

This script does not call the oracle or the CUDA library: every operation is
rewritten here on Python Fractions, so the stored row pins the C oracle
against an independent evaluation.  It searches seeded rows for one whose
output bits change under each of three plausible misreadings, so a mistake
of that kind in either implementation fails the check:

    no_bf16_after_norm   y_i = bf16(fp32(x_i * r) * w_i)
    sequential_sum       ss = (((part_0 + part_1) + part_2) + ... ) + part_31
    rope_without_fma     o_k = bf16(fp32(y_k c_k) - fp32(y_k+64 s_k)), likewise o_k+64

    python tests/golden/make_norm_rope_rounding.py     (rewrites the fixture)
"""
from __future__ import annotations

import math
import os
import struct
from fractions import Fraction

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
OUT = os.path.join(HERE, "norm_rope_rounding.txt")
D, THETA, EPS_DOUBLE = 128, 1e6, 1e-6


def round_to(x: Fraction, mant_bits: int, min_exp: int) -> Fraction:
    """x rounded to nearest, ties to even, on the binary grid with mant_bits
    significant bits and smallest normal exponent min_exp (subnormals below)."""
    if x == 0:
        return Fraction(0)
    sign = -1 if x < 0 else 1
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    e = max(e, min_exp)                                  # binade [2^e, 2^(e+1)) (or subnormal)
    step = Fraction(2) ** (e - mant_bits + 1)
    q, rem = divmod(a, step)
    q = int(q)
    if rem * 2 > step or (rem * 2 == step and q % 2 == 1):
        q += 1
    return sign * q * step


def f32(x):
    return round_to(Fraction(x), 24, -126)


def bf16(x):
    return round_to(Fraction(x), 8, -126)


def f32_sqrt(a: Fraction) -> Fraction:
    """Correctly rounded fp32 square root of a >= 0."""
    c = f32(Fraction(math.sqrt(float(a))))               # within an ulp; fixed exactly below
    for _ in range(4):
        up = _next_up(c)
        dn = _next_down(c)
        if ((c + up) / 2) ** 2 < a:
            c = up
        elif ((c + dn) / 2) ** 2 > a:
            c = dn
        else:
            break
    mid_up, mid_dn = (c + _next_up(c)) / 2, (c + _next_down(c)) / 2
    if mid_up ** 2 == a or mid_dn ** 2 == a:
        raise ValueError("sqrt tie: pick another row")
    return c


def _bits(x: Fraction) -> int:
    return struct.unpack("<I", struct.pack("<f", float(x)))[0]


def _from_bits(u: int) -> Fraction:
    return Fraction(struct.unpack("<f", struct.pack("<I", u))[0])


def _next_up(c: Fraction) -> Fraction:
    return _from_bits(_bits(c) + 1)


def _next_down(c: Fraction) -> Fraction:
    return _from_bits(_bits(c) - 1)


def norm_rope(x, w, cs, eps, variant=None):
    """Output row (Fractions) of the adopted reading, or of a misreading."""
    parts = []
    for l in range(32):
        xs = x[4 * l:4 * l + 4]
        acc = f32(xs[0] * xs[0])
        for xi in xs[1:]:
            acc = f32(xi * xi + acc)                     # fma: one rounding
        parts.append(acc)
    if variant == "sequential_sum":
        ss = parts[0]
        for p in parts[1:]:
            ss = f32(ss + p)
    else:
        width = 16
        while width >= 1:
            for l in range(width):
                parts[l] = f32(parts[l] + parts[l + width])
            width //= 2
        ss = parts[0]
    r = f32(1 / f32_sqrt(f32(f32(ss / 128) + eps)))
    if variant == "no_bf16_after_norm":
        y = [bf16(f32(f32(xi * r) * wi)) for xi, wi in zip(x, w)]
    else:
        y = [bf16(f32(bf16(f32(xi * r)) * wi)) for xi, wi in zip(x, w)]
    h = D // 2
    out = [None] * D
    for k in range(h):
        c, s = cs[k], cs[h + k]
        if variant == "rope_without_fma":
            out[k] = bf16(f32(f32(y[k] * c) - f32(y[k + h] * s)))
            out[k + h] = bf16(f32(f32(y[k + h] * c) + f32(y[k] * s)))
        else:
            out[k] = bf16(f32(y[k] * c - f32(y[k + h] * s)))     # fma(y_k, c, -(y' s)): one fp32 rounding
            out[k + h] = bf16(f32(y[k + h] * c + f32(y[k] * s)))
    return out, ss, r


def bf16_hex(v: Fraction) -> str:
    return f"{_bits(v) >> 16:04x}"


def f32_hex(v: Fraction) -> str:
    return f"{_bits(v):08x}"


def table_row(pos):
    """The rotary table row as the input generator builds it: cos and sin of
    pos * theta^(-2k/128) in float64, rounded once to fp32."""
    k = np.arange(D // 2, dtype=np.float64)
    ang = pos * np.power(THETA, -2.0 * k / D)
    row = np.concatenate([np.cos(ang), np.sin(ang)]).astype(np.float32)
    return [Fraction(float(v)) for v in row]


def _bf16_np(a):
    """float32 array rounded to bf16 (nearest, ties to even), as float32."""
    u = a.astype(np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def _screen(x):
    """Fast float32 pre-screen of a batch of rows [n][128]: True where the two
    summation orders give different ss and that moves some bf16(x_i * r).
    Only a filter; every row kept is then evaluated exactly."""
    sq = x.astype(np.float64).reshape(-1, 32, 4)
    acc = (sq[:, :, 0] * sq[:, :, 0]).astype(np.float32)
    for i in range(1, 4):
        acc = (sq[:, :, i] * sq[:, :, i] + acc.astype(np.float64)).astype(np.float32)
    p = acc.copy()
    width = 16
    while width >= 1:
        p[:, :width] = p[:, :width] + p[:, width:2 * width]
        width //= 2
    seq = acc[:, 0].copy()
    for l in range(1, 32):
        seq = seq + acc[:, l]
    eps = np.float32(EPS_DOUBLE)
    r1 = np.float32(1) / np.sqrt(p[:, 0] / np.float32(128) + eps)
    r2 = np.float32(1) / np.sqrt(seq / np.float32(128) + eps)
    n1 = _bf16_np(x * r1[:, None])
    n2 = _bf16_np(x * r2[:, None])
    return (p[:, 0] != seq) & (n1 != n2).any(axis=1)


def main():
    rng = np.random.default_rng(20261203)
    eps = f32(Fraction(EPS_DOUBLE))
    variants = ("no_bf16_after_norm", "sequential_sum", "rope_without_fma")
    found = None
    for batch in range(200):
        xf = rng.standard_normal((20000, D)).astype(np.float32)
        xf = _bf16_np(xf * rng.choice(np.float32([0.05, 1.0, 30.0]), size=(20000, 1)))
        wf = _bf16_np((0.5 + rng.random((20000, D))).astype(np.float32))
        pos_all = rng.integers(1, 32768, 20000)
        for i in np.nonzero(_screen(xf))[0]:
            x = [Fraction(float(v)) for v in xf[i]]
            w = [Fraction(float(v)) for v in wf[i]]
            pos = int(pos_all[i])
            cs = table_row(pos)
            try:
                ref, ss, r = norm_rope(x, w, cs, eps)
            except ValueError:
                continue
            diffs = {v: sum(a != b for a, b in zip(norm_rope(x, w, cs, eps, v)[0], ref)) for v in variants}
            if all(diffs.values()):
                found = (batch, int(i))
                break
        if found:
            break
    if not found:
        raise SystemExit("no row found")
    attempt = f"batch {found[0]}, row {found[1]}"
    with open(OUT, "w") as f:
        f.write("# One RMSNorm + rotate-half RoPE head row of the fused Q/K boundary, evaluated\n"
                "# in exact rational arithmetic with IEEE round-to-nearest-even after every fp32\n"
                "# and bf16 step (tests/golden/make_norm_rope_rounding.py, which does not call the\n"
                "# oracle or the CUDA library).  Reading: eps 1e-6, per-lane fma chains of four\n"
                "# squares summed pairwise (16, 8, 4, 2, 1), r = 1/sqrt(ss/128 + eps), bf16 after\n"
                "# the normalisation and after the weight, RoPE with one fma per output.\n"
                f"# Seeded search: {attempt} of seed 20261203, position {pos}.  Output elements that\n"
                "# differ from this row under each misreading (each must be > 0):\n")
        for v in variants:
            f.write(f"#   {v}: {diffs[v]}\n")
        f.write("# Intermediates (fp32 hex): ss and r, for a reader checking by hand.\n")
        f.write(f"ss {f32_hex(ss)}\nr {f32_hex(r)}\neps {f32_hex(eps)}\npos {pos}\n")
        f.write("x " + " ".join(bf16_hex(v) for v in x) + "\n")
        f.write("w " + " ".join(bf16_hex(v) for v in w) + "\n")
        f.write("cs " + " ".join(f32_hex(v) for v in cs) + "\n")
        f.write("out " + " ".join(bf16_hex(v) for v in ref) + "\n")
    print(OUT, attempt, diffs)


if __name__ == "__main__":
    main()
