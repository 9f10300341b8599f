"""CPU oracle for paged absorbed-MLA decode.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by the package's
``__graft_entry__.smoke()`` check and by the CPU-baseline leg of ``bench.py``.
The product path (the CUDA library and its Python binding) never imports,
links or calls anything here, and nothing here imports the product path.

* :mod:`oracle.chain` wraps ``k3mla_oracle.c`` -- the rounding chain of
  pegainfer PR #869 ("K3: paged latent MLA KV + absorbed decode", M2 commit),
  written out in plain C.
* :mod:`oracle.expanded` is an independent float64 reference that never
  absorbs: it expands per-head K and V from the latent and runs an ordinary
  softmax attention, so that it checks the absorption identity the M2 commit
  relies on.
* :mod:`oracle.pages` is the whole-page copy of the M1 commit's prefill
  adoption, as numpy assignments.
* :mod:`oracle.chunk` is chunked prefill: the row append once per token and
  the causal view of each token of a chunk.
"""
from .chain import (  # noqa: F401
    absorb,
    append,
    build,
    decode,
    f32_to_bf16,
    MUTATIONS,
)
from .expanded import decode_expanded_f64, expand_pages_f64  # noqa: F401
from .pages import copy_pages  # noqa: F401
from .chunk import append_rows, chunk_views  # noqa: F401
