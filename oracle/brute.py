"""Exact-rational brute force of the Lightning Indexer, used only to pin the fp64 oracle.

TEST INFRASTRUCTURE ONLY. It is deliberately a different computation from ``oracle.cpp``:
every input code is decoded to an exact ``fractions.Fraction`` by its own decoder, the score is
evaluated with no rounding at all, and the Top-k is chosen by rank counting instead of sorting:
key s is kept iff fewer than ``topk`` visible keys beat it, where s' beats s when
I[s'] > I[s], or I[s'] == I[s] and s' < s (ties go to the lower index). The rank itself is the
output slot. Pure-Python loops: tiny inputs only (T, S <= ~32, H, D <= ~8).

Scoring rule restated (the pages name the Lightning Indexer and its Top-512 selection in
"DeepSeek V4 Flash 추론을 1.6초로 줄인 ds4 최적화", sections 섹션별 상세 and 용어 해설):
``I[t,s] = kscale[s] * sum_j w[t,j] * max(0, sum_i q[t,j,i] k[s,i])`` for s <= pos_offset + t.
"""
from __future__ import annotations

import struct
from fractions import Fraction

BF16 = 0
FP8_E4M3 = 1


def bf16_value(bits: int) -> Fraction:
    """bf16 bit pattern -> exact value (via the binary32 it is the top half of)."""
    (f,) = struct.unpack("<f", struct.pack("<I", (int(bits) & 0xFFFF) << 16))
    if f != f or f in (float("inf"), float("-inf")):
        raise ValueError("non-finite bf16")
    return Fraction(f)


def e4m3_value(code: int) -> Fraction:
    """OCP E4M3FN byte -> exact value: (-1)^s * 2^(e-7) * (1 + m/8), subnormal 2^-6 * m/8."""
    code = int(code) & 0xFF
    s, e, m = code >> 7, (code >> 3) & 0xF, code & 0x7
    if e == 0xF and m == 0x7:
        raise ValueError("E4M3 NaN")
    if e == 0:
        v = Fraction(m, 8) * Fraction(1, 2 ** 6)
    else:
        v = (1 + Fraction(m, 8)) * (Fraction(2) ** (e - 7))
    return -v if s else v


def f32_value(x: float) -> Fraction:
    (f,) = struct.unpack("<f", struct.pack("<f", float(x)))
    return Fraction(f)


def exact_scores(dtype, q, w, k, kscale, pos_offset):
    """Dict {(t, s): Fraction} over visible pairs. q: [T][H][D] codes, k: [S][D] codes."""
    dec = bf16_value if dtype == BF16 else e4m3_value
    T, S = len(q), len(k)
    kd = [[dec(c) for c in row] for row in k]
    out = {}
    for t in range(T):
        qd = [[dec(c) for c in head] for head in q[t]]
        wd = [f32_value(x) for x in w[t]]
        p = pos_offset + t
        for s in range(min(p, S - 1) + 1):
            total = Fraction(0)
            for j, qj in enumerate(qd):
                dot = sum((a * b for a, b in zip(qj, kd[s])), Fraction(0))
                total += wd[j] * (dot if dot > 0 else Fraction(0))
            scale = Fraction(1) if dtype == BF16 else f32_value(kscale[s])
            out[(t, s)] = scale * total
    return out


def rank_count_topk(scores, T, S, pos_offset, topk):
    """Selection by rank counting. Returns per-row lists [(idx, Fraction)] in rank order."""
    rows = []
    for t in range(T):
        n = min(pos_offset + t, S - 1) + 1
        row = [scores[(t, s)] for s in range(n)]
        slots = [None] * min(topk, n)
        for s in range(n):
            rank = sum(1 for s2 in range(n)
                       if row[s2] > row[s] or (row[s2] == row[s] and s2 < s))
            if rank < topk:
                slots[rank] = (s, row[s])
        rows.append(slots)
    return rows
