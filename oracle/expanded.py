"""Float64 expanded-K/V reference: attention WITHOUT absorption.

TEST INFRASTRUCTURE ONLY -- see ``oracle/__init__.py``.

pegainfer PR #869 ("K3: paged latent MLA KV + absorbed decode", M2 commit)
replaces a cache of per-head K and V rows, expanded from the latent by kv_b, with
an absorbed kernel over the latent itself, and notes that the two differ only in
how the score dot is associated: (W_UK^T q)^T c versus q^T (W_UK c).  This module
computes the design it replaced, in float64, for each head h and token t:

    k_nope[t] = W_UK[h] c_t            (128)
    k[t]      = [k_nope[t] ; k_rope_t] (192)
    v[t]      = W_UV[h] c_t            (128)
    s_t       = scale * (q_nope . k_nope[t] + q_rope . k_rope_t)
    p         = softmax(s)             (float64)
    out       = sum_t p_t v[t]

No bf16 landing is applied anywhere, so the difference from the rounding-chain
oracle is the chain's own rounding error; it is an independent check of the
absorption identity and of every index and term in the chain.  A -1 table entry
is a zero latent (zero K nope part, zero rope key, zero V), as in the M2 commit.
"""
from __future__ import annotations

import numpy as np

H, NOPE, ROPE, V, LORA, PAGE = 96, 128, 64, 128, 512, 64
ROW = LORA + ROPE


def bf16_bits_to_f64(a: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    return (np.asarray(a, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def gather_rows(slab: np.ndarray, layer: int, table_row: np.ndarray, n: int) -> np.ndarray:
    """Latent rows of one slot's first n logical tokens as float64 [n, 576]; -1 -> zeros."""
    rows = np.zeros((n, ROW), np.float64)
    for t in range(n):
        pid = int(table_row[t // PAGE])
        if pid >= 0:
            rows[t] = bf16_bits_to_f64(slab[pid, layer, t % PAGE])
    return rows


def decode_expanded_f64(q, slab, layer, block_table, ctx_len, w_kv_b, scale, slots=None):
    """Float64 expanded attention.  q [B,96,192] bf16 bits (NOT absorbed).

    Returns out [B,96,128] float64 and the float64 probabilities' argmax [B,96]
    (lowest t on ties; -1 for an empty context).
    """
    B = q.shape[0]
    w = bf16_bits_to_f64(w_kv_b).reshape(H, NOPE + V, LORA)
    w_uk, w_uv = w[:, :NOPE, :], w[:, NOPE:, :]
    qf = bf16_bits_to_f64(q)
    out = np.zeros((B, H, V), np.float64)
    am = np.full((B, H), -1, np.int64)
    if slots is None:
        slots = range(B)
    for b in slots:
        n = int(ctx_len[b])
        if n <= 0:
            continue
        rows = gather_rows(slab, layer, block_table[b], n)
        c, k_rope = rows[:, :LORA], rows[:, LORA:]
        for h in range(H):
            k_nope = c @ w_uk[h].T                      # [n,128]
            v = c @ w_uv[h].T                           # [n,128]
            s = scale * (k_nope @ qf[b, h, :NOPE] + k_rope @ qf[b, h, NOPE:])
            s = s - s.max()
            e = np.exp(s)
            p = e / e.sum()
            out[b, h] = p @ v
            am[b, h] = int(np.argmax(p))
    return out, am


def expand_pages_f64(slab, layer, w_kv_b, pages) -> np.ndarray:
    """The expanded cache of the listed pages at one layer, in float64, unlanded.

    pegainfer PR #869, M2 commit: kv_b expands each token's latent into per-head
    K and V rows, the cache the absorbed decode does away with.  Returns [len(pages), 64 tokens, 96 heads, 320] with,
    for head h and the token at page position t, the row
        [ W_UK[h] c_t (128) | k_rope_t (64) | W_UV[h] c_t (128) ]
    where c_t and k_rope_t are the first 512 and last 64 values of its latent row.
    """
    w = bf16_bits_to_f64(w_kv_b).reshape(H, NOPE + V, LORA)
    out = np.zeros((len(pages), PAGE, H, NOPE + ROPE + V), np.float64)
    for i, pid in enumerate(pages):
        rows = bf16_bits_to_f64(slab[int(pid), layer])            # [64, 576]
        c, k_rope = rows[:, :LORA], rows[:, LORA:]
        out[i, :, :, :NOPE] = np.einsum("hdj,tj->thd", w[:, :NOPE, :], c)
        out[i, :, :, NOPE:NOPE + ROPE] = k_rope[:, None, :]
        out[i, :, :, NOPE + ROPE:] = np.einsum("hdj,tj->thd", w[:, NOPE:, :], c)
    return out
