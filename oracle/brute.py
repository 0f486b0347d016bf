"""Scalar pure-Python restatement of one decoder layer and the vocab head.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  Written independently
of ``oracle.forward``: Python floats (IEEE double), explicit loops, the math
module, no torch, no BLAS.  Used on tiny shapes to pin ``oracle.forward``.

Same definitions and readings as ``oracle.forward`` (RMSNorm, rotate-half
RoPE after per-head q/k RMSNorm, 1/sqrt(hd) scale, causal mask with cache
offset, GQA head h -> kv head h // (nq / nkv), SiLU-gated MLP, residual adds),
from [TP] "Tensor parallelism from scratch", tp.py.
"""

from __future__ import annotations

import math
import struct
from typing import Callable, List, Optional, Sequence, Tuple

Vec = List[float]
Mat = List[List[float]]  # row-major [out][in]


def matvec(w: Mat, x: Vec) -> Vec:
    out = []
    for row in w:
        s = 0.0
        for a, b in zip(row, x):
            s += a * b
        out.append(s)
    return out


def rmsnorm(x: Vec, w: Vec, eps: float) -> Vec:
    ss = 0.0
    for v in x:
        ss += v * v
    inv = 1.0 / math.sqrt(ss / len(x) + eps)
    return [x[i] * inv * w[i] for i in range(len(x))]


def rope(u: Vec, p: int, theta: float) -> Vec:
    hd = len(u)
    half = hd // 2
    out = [0.0] * hd
    for d in range(half):
        ang = p * theta ** (-2.0 * d / hd)
        c, s = math.cos(ang), math.sin(ang)
        a, b = u[d], u[d + half]
        out[d] = a * c - b * s
        out[d + half] = b * c + a * s
    return out


def bf16_value(x: float) -> float:
    """x rounded to fp32 (struct's round to nearest), then to bf16: the upper 16 bits
    with round to nearest, ties to even, on the bit pattern; finite inputs."""
    u = struct.unpack("<I", struct.pack("<f", x))[0]
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFFFFFF
    return struct.unpack("<f", struct.pack("<I", u & 0xFFFF0000))[0]


def layer(x_rows: Sequence[Vec], w: dict, nq: int, nkv: int, hd: int, eps: float, theta: float,
          k_cache: Sequence[Sequence[Vec]], v_cache: Sequence[Sequence[Vec]],
          store: Optional[Callable[[float], float]] = None
          ) -> Tuple[List[Vec], List[List[Vec]], List[List[Vec]]]:
    """x_rows: T new tokens (rows of length H).  k_cache[g][p] / v_cache[g][p]:
    cached rows of kv head g at position p.  w: dict of nested lists
    (q, k, v, o, gate, up, down, in_norm, post_norm, q_norm, k_norm).
    store: what the cache keeps of each new K / V element (None: the value)."""
    keep = store if store is not None else (lambda a: a)
    T = len(x_rows)
    ctx = len(k_cache[0]) if nkv else 0
    K = [list(k_cache[g]) for g in range(nkv)]
    V = [list(v_cache[g]) for g in range(nkv)]
    qs = []  # qs[t][h] -> vector
    for t in range(T):
        pos = ctx + t
        h = rmsnorm(x_rows[t], w["in_norm"], eps)
        q = matvec(w["q"], h)
        k = matvec(w["k"], h)
        v = matvec(w["v"], h)
        qh = []
        for head in range(nq):
            qv = rmsnorm(q[head * hd:(head + 1) * hd], w["q_norm"], eps)
            qh.append(rope(qv, pos, theta))
        qs.append(qh)
        for g in range(nkv):
            kv = rmsnorm(k[g * hd:(g + 1) * hd], w["k_norm"], eps)
            K[g].append([keep(a) for a in rope(kv, pos, theta)])
            V[g].append([keep(a) for a in v[g * hd:(g + 1) * hd]])
    group = nq // nkv
    out_rows = []
    for t in range(T):
        last_key = ctx + t
        attn_cat: Vec = []
        for head in range(nq):
            g = head // group
            scores = []
            for j in range(last_key + 1):
                s = 0.0
                for d in range(hd):
                    s += qs[t][head][d] * K[g][j][d]
                scores.append(s / math.sqrt(hd))
            m = max(scores)
            e = [math.exp(s - m) for s in scores]
            z = sum(e)
            o = [0.0] * hd
            for j in range(last_key + 1):
                pj = e[j] / z
                for d in range(hd):
                    o[d] += pj * V[g][j][d]
            attn_cat.extend(o)
        proj = matvec(w["o"], attn_cat)
        x1 = [x_rows[t][i] + proj[i] for i in range(len(proj))]
        h2 = rmsnorm(x1, w["post_norm"], eps)
        gate = matvec(w["gate"], h2)
        up = matvec(w["up"], h2)
        act = [gate[i] / (1.0 + math.exp(-gate[i])) * up[i] for i in range(len(gate))]
        dn = matvec(w["down"], act)
        out_rows.append([x1[i] + dn[i] for i in range(len(dn))])
    return out_rows, K, V


def head_argmax(x_last: Vec, final_norm: Vec, lm: Mat, eps: float) -> Tuple[Vec, int]:
    z = rmsnorm(x_last, final_norm, eps)
    logits = matvec(lm, z)
    best = 0
    for i in range(1, len(logits)):
        if logits[i] > logits[best]:
            best = i
    return logits, best
