"""paged_latent_attention_k3mla_gb300 -- paged absorbed-MLA decode for GB300 (sm_103a).

The compute path is the C-ABI library ``libk3mla.so`` (hand-written CUDA for
sm_103a, declared in ``include/k3mla.h``); :mod:`.k3mla` is its thin ctypes
binding.  Importing this package does not load the library; the first call
into :mod:`.k3mla` does, and raises if it is missing.
"""
GEOMETRY = dict(heads=96, qk_nope=128, qk_rope=64, v_head=128, kv_lora=512, page=64, row=576)
