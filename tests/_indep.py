"""An independent, pure-Python restatement of the method for pinning the oracle.

It shares no code with ``oracle/kvoracle.c`` and is written differently on
purpose, so that a slip in one is unlikely to be repeated in the other:
  * bf16 rounding uses exact rational arithmetic (``fractions.Fraction``) and
    encodes the result from the bf16 format definition (1 sign, 8 exponent,
    7 fraction bits; IEEE 754 roundTiesToEven);
  * the rotation R(δ) is complex multiplication: with rotate-half pairing,
    z_j = x[j] + i·x[j+d/2] becomes z_j·exp(i·δ·θ_j), θ_j = base^(-2j/d);
  * a splice is list slicing on the logical sequence:
    old[:s_start] + stub + [R(Δ) row for row in old[s_end:]];
  * the patch product is a numpy matmul (a library primitive).
Slow by design; for tiny cases only.
"""
from __future__ import annotations

import cmath
import math
import struct
from fractions import Fraction

import numpy as np

BF16_MAX = Fraction(255 * 2 ** 120)


def bf16_bits_to_float(b: int) -> float:
    return struct.unpack("<f", struct.pack("<I", (int(b) & 0xFFFF) << 16))[0]


def round_bf16(v: float) -> int:
    """Nearest bf16 bit pattern to the double ``v`` (ties to even), exactly."""
    if math.isnan(v):
        return 0x7FC0
    sign = 0x8000 if math.copysign(1.0, v) < 0 else 0
    if math.isinf(v):
        return sign | 0x7F80
    a = Fraction(abs(v))
    if a == 0:
        return sign
    # E with 2^E <= a < 2^(E+1)
    E = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** E > a:
        E -= 1
    assert Fraction(2) ** E <= a < Fraction(2) ** (E + 1)
    E = max(E, -126)
    q = E - 7
    n = round(a / Fraction(2) ** q)          # Fraction.__round__: ties to even
    value = n * Fraction(2) ** q
    if value > BF16_MAX:
        return sign | 0x7F80
    if n == 0:
        return sign
    if n < 128:                               # subnormal: exponent field 0
        return sign | n
    if n == 256:                              # carried into the next binade
        n, q = 128, q + 1
    exp_field = q + 7 + 127
    assert 1 <= exp_field <= 254 and 128 <= n < 256
    return sign | (exp_field << 7) | (n - 128)


def theta(base: float, j: int, d: int) -> float:
    return base ** (-2.0 * j / d)


def rotate_exact(x, delta: int, base: float, il: bool = False):
    """R(δ)·x for a real rotary vector x (list of floats), as complex products:
    z_j = x[j] + i·x[j+d/2] (rotate-half) or x[2j] + i·x[2j+1] (il)."""
    d = len(x)
    h = d // 2
    out = [0.0] * d
    for j in range(h):
        re, im = (2 * j, 2 * j + 1) if il else (j, j + h)
        z = complex(x[re], x[im]) * cmath.exp(1j * (delta * theta(base, j, d)))
        out[re], out[im] = z.real, z.imag
    return out


def rotate_bits(xbits, delta: int, base: float, il: bool = False):
    """bf16 rotation on bit patterns; R(0) keeps the bits."""
    if delta == 0:
        return [int(b) for b in xbits]
    y = rotate_exact([bf16_bits_to_float(b) for b in xbits], delta, base, il)
    return [round_bf16(v) for v in y]


def rotate_row(rowbits, heads: int, d: int, delta: int, base: float, il: bool = False):
    out = []
    for h in range(heads):
        out += rotate_bits(rowbits[h * d:(h + 1) * d], delta, base, il)
    return out


def slot(bt_row, pos: int, block: int) -> int:
    return int(bt_row[pos // block]) * block + pos % block


def relocate(src_copy, src_rot, dst_copy, dst_rot, block, heads, d, base, tok_off, src_slots,
             chunk_req, chunk_dst_pos, delta, bt, patch=None, il=False):
    """Gather + rotate (+ patch) into copies of the destination arrays.

    ``patch`` = (U[2], V[2]) with U[ch] (L, T, m) and V[ch] (L, C, width, m)
    float32 arrays (None entries = channel not patched)."""
    dc, dr = dst_copy.copy(), dst_rot.copy()
    L = src_copy.shape[0]
    for c in range(len(chunk_req)):
        for i in range(int(tok_off[c + 1] - tok_off[c])):
            t = int(tok_off[c]) + i
            s = int(src_slots[t])
            o = slot(bt[chunk_req[c]], int(chunk_dst_pos[c]) + i, block)
            for l in range(L):
                cp = [int(b) for b in src_copy[l, s]]
                if patch is not None and patch[0][0] is not None:
                    add = np.asarray(patch[0][0][l, t], np.float64) @ np.asarray(
                        patch[1][0][l, c], np.float64).T
                    cp = [round_bf16(bf16_bits_to_float(b) + float(a)) for b, a in zip(cp, add)]
                dc[l, o] = cp
                rb = [int(b) for b in src_rot[l, s]]
                if patch is not None and patch[0][1] is not None:
                    add = np.asarray(patch[0][1][l, t], np.float64) @ np.asarray(
                        patch[1][1][l, c], np.float64).T
                    ex = []
                    for h in range(heads):
                        seg = [bf16_bits_to_float(b) for b in rb[h * d:(h + 1) * d]]
                        ex += seg if delta[c] == 0 else rotate_exact(seg, int(delta[c]), base, il)
                    dr[l, o] = [round_bf16(e + float(a)) for e, a in zip(ex, add)]
                else:
                    dr[l, o] = rotate_row(rb, heads, d, int(delta[c]), base, il)
    return dc, dr


def splice(copy, rot, block, heads, d, base, bt, seq_lens, s_start, s_end, stub_len, stub_copy,
           stub_rot, il=False):
    """List-slicing restatement of one AMORTIZE directive per sequence."""
    pc, pr = copy.copy(), rot.copy()
    L = copy.shape[0]
    new_lens = []
    off = 0
    for q in range(len(seq_lens)):
        n, a, b, nr = int(seq_lens[q]), int(s_start[q]), int(s_end[q]), int(stub_len[q])
        delta = nr - (b - a)
        for l in range(L):
            old = [(list(pc[l, slot(bt[q], p, block)]), list(pr[l, slot(bt[q], p, block)]))
                   for p in range(n)]
            stub = [(list(stub_copy[l, off + k]), list(stub_rot[l, off + k])) for k in range(nr)]
            moved = [(cpy, rotate_row(rt, heads, d, delta, base, il)) for cpy, rt in old[b:]]
            new = old[:a] + stub + moved
            for p, (cpy, rt) in enumerate(new):
                s = slot(bt[q], p, block)
                pc[l, s] = cpy
                pr[l, s] = rt
        new_lens.append(n + delta)
        off += nr
    return pc, pr, new_lens


def splice_composed(copy, rot, block, heads, d, base, bt, seq_lens, dirs, stub_copy, stub_rot):
    """List-slicing restatement of several directives per sequence, composed.

    ``dirs`` lists the directives in order as (s_start[S], s_end[S],
    stub_len[S]), each in the indexing the previous ones left; stub rows are
    stored directive by directive, then sequence by sequence.  The sequence is
    first edited symbolically -- each entry remembers where its content came
    from and the position it was written at -- and every final row is then
    that content turned once by R(final position - written position)."""
    pc, pr = copy.copy(), rot.copy()
    L = copy.shape[0]
    first_stub, off = {}, 0
    for i, (_, _, nrs) in enumerate(dirs):
        for q, nr in enumerate(nrs):
            first_stub[(i, q)] = off
            off += int(nr)
    new_lens = []
    for q in range(len(seq_lens)):
        seq = [("old", p, p) for p in range(int(seq_lens[q]))]
        for i, (starts, ends, nrs) in enumerate(dirs):
            a, b, nr = int(starts[q]), int(ends[q]), int(nrs[q])
            stub = [("stub", first_stub[(i, q)] + k, a + k) for k in range(nr)]
            seq = seq[:a] + stub + seq[b:]
        for l in range(L):
            rows = []
            for p, (kind, idx, written) in enumerate(seq):
                if kind == "old":
                    s = slot(bt[q], idx, block)
                    cpy, rt = list(copy[l, s]), list(rot[l, s])
                else:
                    cpy, rt = list(stub_copy[l, idx]), list(stub_rot[l, idx])
                rows.append((cpy, rotate_row(rt, heads, d, p - written, base)))
            for p, (cpy, rt) in enumerate(rows):
                s = slot(bt[q], p, block)
                pc[l, s] = cpy
                pr[l, s] = rt
        new_lens.append(len(seq))
    return pc, pr, new_lens
