"""Seeded synthetic inputs for paged absorbed-MLA decode.

This module only draws random numbers and builds page tables; it holds none of
the attention arithmetic.  It is the one module that both the CUDA path's
callers (tests, ``bench.py``) and the CPU oracle's callers use, so that both
sides see the same bits.

Geometry and distributions follow the five synthetic workloads the project
benchmarks (96 heads, q_nope 128, q_rope 64, v_head 128, kv_lora 512, page 64,
cache row 576 bf16 -- pegainfer PR #869, "K3: paged latent MLA KV + absorbed
decode", M1 and M2 commits):

* ``tiny``: 1 layer, 1 slot, context 130 (3 pages, last partial), a 16-page pool
  whose ids are randomly permuted into the block table; seed 0.
* ``ragged16``: 16 slots x 24 layers, context uniform in [1, 4096] (the length
  after this step's append), pages from a shuffled free list over a pool sized
  for full coverage; seed 1.
* ``steady64``: 64 slots x 24 layers, every slot at 4096 tokens; seed 2.
* ``long8``: 8 slots x 24 layers at 32768 tokens, each latent row (all 576
  values) multiplied by a per-token factor drawn log-uniform in [0.25, 4];
  seed 3.
* ``padding128``: 128 rows, 40 % padding slots whose tables are all -1 (their
  context drawn like the others), the rest with context uniform in [1, 256],
  random -1 holes inside the mapped range, one slot with context 0; seed 4.

Everything is drawn with torch generators on the requested device: q, c and
k_rope are N(0, 1), w_kv_b is N(0, 1/512), each rounded to bf16 by torch's
round-to-nearest-even conversion.  The softmax scale is bf16(1/sqrt(192)).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

H, NOPE, ROPE, V, LORA, PAGE = 96, 128, 64, 128, 512, 64
ROW = LORA + ROPE
QDIM = NOPE + ROPE
WROWS = H * (NOPE + V)


def bf16_bits(x: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (host copy)."""
    assert x.dtype == torch.bfloat16
    return x.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def from_bf16_bits(a: np.ndarray, device="cpu") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)


def scale_bf16_bits() -> int:
    """bf16(1/sqrt(qk_nope + qk_rope)) = bf16(1/sqrt(192)) as a bit pattern."""
    t = torch.tensor([1.0 / math.sqrt(NOPE + ROPE)], dtype=torch.float32).to(torch.bfloat16)
    return int(bf16_bits(t)[0])


@dataclass
class Workload:
    name: str
    seed: int
    n_layers: int
    B: int
    ctx_len: np.ndarray          # [B] int32, length after this step's append
    block_table: np.ndarray      # [B, max_pages] int32, -1 = unmapped
    n_pages: int
    device: str
    q: torch.Tensor              # [L, B, 96, 192] bf16
    w_kv_b: torch.Tensor         # [L, 24576, 512] bf16
    slab: torch.Tensor           # [n_pages, L, 64, 576] bf16
    new_c: torch.Tensor          # [L, B, 512] bf16: row appended this step
    new_rope: torch.Tensor       # [L, B, 64] bf16
    scale_bits: int = field(default_factory=scale_bf16_bits)

    @property
    def max_pages(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def pos(self) -> np.ndarray:
        """Write position of this step's new token (ctx_len - 1; -1 when empty)."""
        return (self.ctx_len.astype(np.int64) - 1).astype(np.int32)

    def latent_bytes(self) -> int:
        return int(self.ctx_len.astype(np.int64).clip(min=0).sum()) * ROW * 2


def _randn_bf16(shape, g, device, std=1.0, chunk=1 << 28):
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    for s in range(0, flat.numel(), chunk):
        e = min(flat.numel(), s + chunk)
        x = torch.randn(e - s, generator=g, device=device, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        flat[s:e].copy_(x.to(torch.bfloat16))
    return out


def _tables_from_free_list(ctx, max_pages, n_pages, rng):
    """Slots claim pages, in slot order, from a shuffled free list."""
    free = rng.permutation(n_pages).astype(np.int32)
    tbl = np.full((len(ctx), max_pages), -1, np.int32)
    k = 0
    for b, n in enumerate(ctx):
        need = (int(n) + PAGE - 1) // PAGE
        assert need <= max_pages and k + need <= n_pages
        tbl[b, :need] = free[k:k + need]
        k += need
    return tbl


def _finish(name, seed, L, ctx, tbl, n_pages, device, g, row_scale=None):
    B = len(ctx)
    q = _randn_bf16((L, B, H, QDIM), g, device)
    w = _randn_bf16((L, WROWS, LORA), g, device, std=math.sqrt(1.0 / LORA))
    slab = _randn_bf16((n_pages, L, PAGE, ROW), g, device)
    new_c = _randn_bf16((L, B, LORA), g, device)
    new_rope = _randn_bf16((L, B, ROPE), g, device)
    if row_scale is not None:
        # per physical row factor (every row of the slab), so that every logical
        # token -- whichever page it sits on -- carries a heavy-tailed magnitude
        f = torch.exp(torch.empty((n_pages, L, PAGE, 1), device=device, dtype=torch.float32)
                      .uniform_(math.log(row_scale[0]), math.log(row_scale[1]), generator=g))
        for p0 in range(0, n_pages, 256):
            p1 = min(n_pages, p0 + 256)
            slab[p0:p1] = (slab[p0:p1].float() * f[p0:p1]).to(torch.bfloat16)
        fn = torch.exp(torch.empty((L, B, 1), device=device, dtype=torch.float32)
                       .uniform_(math.log(row_scale[0]), math.log(row_scale[1]), generator=g))
        new_c = (new_c.float() * fn).to(torch.bfloat16)
        new_rope = (new_rope.float() * fn).to(torch.bfloat16)
    return Workload(name=name, seed=seed, n_layers=L, B=B, ctx_len=np.asarray(ctx, np.int32),
                    block_table=tbl, n_pages=n_pages, device=str(device), q=q, w_kv_b=w,
                    slab=slab, new_c=new_c, new_rope=new_rope)


def make_workload(name: str, device="cpu", n_layers: int | None = None) -> Workload:
    """One of the five named workloads.  ``n_layers`` may shrink the layer count
    (for tests that only need one layer of a 24-layer workload)."""
    if name == "tiny":
        seed, L = 0, 1
        rng = np.random.default_rng(seed)
        g = torch.Generator(device=device).manual_seed(seed)
        perm = rng.permutation(16).astype(np.int32)
        tbl = np.full((1, 4), -1, np.int32)
        tbl[0, :3] = perm[:3]
        return _finish(name, seed, n_layers or L, np.array([130]), tbl, 16, device, g)
    if name == "ragged16":
        seed, L, B, max_ctx = 1, 24, 16, 4096
        rng = np.random.default_rng(seed)
        g = torch.Generator(device=device).manual_seed(seed)
        ctx = rng.integers(1, max_ctx + 1, size=B)
        max_pages = max_ctx // PAGE
        n_pages = B * max_pages
        tbl = _tables_from_free_list(ctx, max_pages, n_pages, rng)
        return _finish(name, seed, n_layers or L, ctx, tbl, n_pages, device, g)
    if name == "steady64":
        seed, L, B, max_ctx = 2, 24, 64, 4096
        rng = np.random.default_rng(seed)
        g = torch.Generator(device=device).manual_seed(seed)
        ctx = np.full(B, max_ctx)
        max_pages = max_ctx // PAGE
        n_pages = B * max_pages
        tbl = _tables_from_free_list(ctx, max_pages, n_pages, rng)
        return _finish(name, seed, n_layers or L, ctx, tbl, n_pages, device, g)
    if name == "long8":
        seed, L, B, max_ctx = 3, 24, 8, 32768
        rng = np.random.default_rng(seed)
        g = torch.Generator(device=device).manual_seed(seed)
        ctx = np.full(B, max_ctx)
        max_pages = max_ctx // PAGE
        n_pages = B * max_pages
        tbl = _tables_from_free_list(ctx, max_pages, n_pages, rng)
        return _finish(name, seed, n_layers or L, ctx, tbl, n_pages, device, g,
                       row_scale=(0.25, 4.0))
    if name == "padding128":
        seed, L, B, max_ctx = 4, 1, 128, 256
        rng = np.random.default_rng(seed)
        g = torch.Generator(device=device).manual_seed(seed)
        ctx = rng.integers(1, max_ctx + 1, size=B)
        max_pages = max_ctx // PAGE
        n_pages = B * max_pages
        tbl = _tables_from_free_list(ctx, max_pages, n_pages, rng)
        pad = rng.random(B) < 0.4
        tbl[pad] = -1
        holes = (rng.random(tbl.shape) < 0.15) & (tbl >= 0)
        tbl[holes] = -1
        ctx[int(np.flatnonzero(~pad)[0])] = 0   # one empty slot among the real rows
        return _finish(name, seed, n_layers or L, ctx, tbl, n_pages, device, g)
    raise ValueError(f"unknown workload {name!r}")


def make_custom(ctx_lens, n_layers=1, seed=123, device="cpu", max_pages=None, n_pages=None,
                row_scale=None) -> Workload:
    """A small workload with the given per-slot context lengths (tables from a
    shuffled free list over a pool with a few spare pages)."""
    ctx = np.asarray(ctx_lens, np.int64)
    need = (ctx + PAGE - 1) // PAGE
    if max_pages is None:
        max_pages = max(1, int(need.max()) if len(need) else 1)
    if n_pages is None:
        n_pages = int(need.sum()) + 3
    rng = np.random.default_rng(seed)
    g = torch.Generator(device=device).manual_seed(seed)
    tbl = _tables_from_free_list(ctx, max_pages, n_pages, rng)
    return _finish(f"custom{seed}", seed, n_layers, ctx, tbl, n_pages, device, g,
                   row_scale=row_scale)


WORKLOADS = ("tiny", "ragged16", "steady64", "long8", "padding128")
