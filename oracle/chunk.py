"""Chunked prefill, written out plainly (test infrastructure only).

pegainfer PR #869, "K3: paged latent MLA KV + absorbed decode": its follow-up list
queues chunked prefill in place of the token-by-token loop over a prompt.  A chunk
holds the next n_b tokens of slot b, at positions pos0[b] .. pos0[b] + n_b - 1; its
per-token inputs are packed, slot b's being rows row_start[b] .. row_start[b+1] - 1.

* :func:`append_rows` is the M1 commit's indexed row write, once per token.
* :func:`chunk_views` states the causal mask within the chunk: token j of slot b
  attends over the first pos0[b] + j + 1 tokens of the slot, through the slot's
  block table -- exactly what the token-by-token loop saw when it decoded token j.
"""
from __future__ import annotations

import numpy as np

PAGE, LORA = 64, 512


def append_rows(slab, layer, block_table, pos0, row_start, c_kv, k_rope) -> int:
    """In place: every token's latent row (c_kv | k_rope) into the mapped row of its position.
    Returns the rows skipped (page -1 / out of range, negative position, past the table)."""
    n_pages, max_pages = slab.shape[0], block_table.shape[1]
    skipped = 0
    for b in range(len(pos0)):
        for r in range(int(row_start[b]), int(row_start[b + 1])):
            p = int(pos0[b]) + (r - int(row_start[b]))
            page = int(block_table[b, p // PAGE]) if 0 <= p < max_pages * PAGE else -1
            if not 0 <= page < n_pages:
                skipped += 1
                continue
            slab[page, layer, p % PAGE, :LORA] = c_kv[r, :LORA]
            slab[page, layer, p % PAGE, LORA:] = k_rope[r, :slab.shape[3] - LORA]
    return skipped


def chunk_views(block_table, pos0, row_start, R: int):
    """Per-token (table row, context length) of the packed chunk; rows past the chunk: empty."""
    max_pages = block_table.shape[1]
    vtable = np.full((R, max_pages), -1, np.int32)
    vctx = np.zeros(R, np.int32)
    for b in range(len(pos0)):
        for r in range(int(row_start[b]), min(int(row_start[b + 1]), R)):
            vtable[r] = block_table[b]
            vctx[r] = int(pos0[b]) + (r - int(row_start[b])) + 1
    return vtable, vctx
