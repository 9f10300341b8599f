"""A second, separately written scalar emulation of the rounding chain.

Used only as a bitwise cross-check of the C oracle on tiny contexts (it is a
re-statement of the same chain, so it does not by itself pin the oracle to the
pages; the float64 expanded reference and the closed forms do that).  bf16
rounding here goes through torch's conversion, not the oracle's own routine.
"""
from __future__ import annotations

import math

import numpy as np
import torch

H, NOPE, ROPE, V, LORA, PAGE = 96, 128, 64, 128, 512, 64
ROW = LORA + ROPE


def _w(bits) -> np.float32:
    return np.array([np.uint32(int(bits)) << np.uint32(16)], np.uint32).view(np.float32)[0]


def _land(x: np.float32) -> np.float32:
    """bf16 landing via torch (round to nearest even)."""
    t = torch.tensor([float(x)], dtype=torch.float32).to(torch.bfloat16).to(torch.float32)
    return np.float32(t.item())


def twin_head(q_abs_row, rows, n, w_uv_rows, scale_bits):
    """rows: list of n cache rows (uint16[576]) or None for zero latent.
    Returns (out bf16 values as f32 [128], p [n] as f32, s [n] as f32)."""
    Q = [_w(b) for b in q_abs_row]
    scale = _w(scale_bits)
    s = []
    for t in range(n):
        acc = np.float32(0.0)
        if rows[t] is not None:
            for k in range(ROW):
                acc = np.float32(acc + np.float32(Q[k] * _w(rows[t][k])))
        s.append(_land(np.float32(_land(acc) * scale)))
    m = s[0]
    for x in s[1:]:
        if x > m:
            m = x
    e = [np.float32(math.exp(float(np.float32(x - m)))) for x in s]
    lsum = np.float32(0.0)
    for x in e:
        lsum = np.float32(lsum + x)
    p = [_land(np.float32(x / lsum)) for x in e]
    ol = []
    for j in range(LORA):
        acc = np.float32(0.0)
        for t in range(n):
            c = _w(rows[t][j]) if rows[t] is not None else np.float32(0.0)
            acc = np.float32(acc + np.float32(p[t] * c))
        ol.append(_land(acc))
    out = []
    for v in range(V):
        acc = np.float32(0.0)
        for j in range(LORA):
            acc = np.float32(acc + np.float32(_w(w_uv_rows[v][j]) * ol[j]))
        out.append(_land(acc))
    return np.array(out, np.float32), np.array(p, np.float32), np.array(s, np.float32)
