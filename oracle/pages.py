"""Whole-page copy on the page-first slab, written out plainly (test infrastructure only).

pegainfer PR #869, "K3: paged latent MLA KV + absorbed decode", M1 commit: a prefilled
sequence is adopted into a decode slot by copying its pages whole.  In the slab
``[page][layer][64][576]`` a page is every layer's 64 rows of one block of tokens, so
the copy moves ``slab[src]`` (all layers) to ``slab[dst]``.  Pairs naming a page
outside their slab are skipped and counted, as the device call skips and flags them.
"""
from __future__ import annotations

import numpy as np


def copy_pages(dst_slab: np.ndarray, src_slab: np.ndarray, src_ids, dst_ids) -> int:
    """In place: dst_slab[dst_ids[i]] = src_slab[src_ids[i]] for every valid pair, in order.
    The slabs are uint16 arrays [n_pages][L][64][576] with the same L.  Returns the pairs skipped."""
    assert dst_slab.shape[1:] == src_slab.shape[1:]
    skipped = 0
    for s, d in zip(np.asarray(src_ids).tolist(), np.asarray(dst_ids).tolist()):
        if not (0 <= s < src_slab.shape[0] and 0 <= d < dst_slab.shape[0]):
            skipped += 1
            continue
        dst_slab[d] = src_slab[s]
    return skipped
