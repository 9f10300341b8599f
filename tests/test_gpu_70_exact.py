"""The exact-chain decode (k3mla_decode_exact) against the oracle, bit for bit.

The mode follows the chain's summation orders and landings exactly (CUDA-core
sequential sums, double exp rounded once to f32, IEEE quotient), so the whole
output -- out and argmax -- must equal the CPU oracle's bits, not merely fall
within the one-pass kernel's 4-ULP bar: ragged contexts across page and tile
boundaries, -1 holes, a bad page id (flagged, read as zero), an empty context,
heavy-tailed rows, the longest context the mode takes, padding slots, and sampled
slots of the full-size workload."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from paged_latent_attention_k3mla_gb300 import k3mla, synth
from tests.gpu_common import oracle_layer

pytestmark = pytest.mark.gpu


def _exact(wl, layer, table=None, max_ctx=None):
    B = wl.B
    max_ctx = max_ctx or max(64, int(wl.block_table.shape[1]) * 64)
    table = torch.from_numpy(wl.block_table if table is None else table).cuda()
    ctx = torch.from_numpy(wl.ctx_len).cuda()
    ws = torch.empty(k3mla.decode_exact_workspace_bytes(B, max_ctx), dtype=torch.uint8, device="cuda")
    ws.fill_(0xFF)
    out = torch.full((B, 96, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    am = torch.full((B, 96), -7, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    k3mla.decode_exact(wl.q[layer], wl.slab, layer, table, ctx, wl.w_kv_b[layer], wl.scale_bits, out, ws, max_ctx,
                       argmax=am, dev_err=err)
    torch.cuda.synchronize()
    return dict(out=synth.bf16_bits(out), argmax=am.cpu().numpy(), dev_err=int(err.item()))


def _bitwise(g, o, slots=None):
    slots = list(range(g["out"].shape[0])) if slots is None else list(slots)
    same = g["out"][slots] == o["out"]
    assert same.all(), f"{(~same).sum()} of {same.size} output elements differ"
    assert np.array_equal(g["argmax"][slots], o["argmax"])


def test_exact_ragged_holes_and_empty(gpu_lib):
    ctx = [1, 2, 63, 64, 65, 127, 129, 300, 640, 1000, 0]
    wl = synth.make_custom(ctx, n_layers=2, seed=700, device="cuda")
    tbl = wl.block_table.copy()
    tbl[7, 2] = -1                       # a -1 hole inside the context: zero rows that take part
    tbl[9, 5] = wl.n_pages + 3           # a bad id: flagged, read as zero
    wl.block_table = tbl
    g = _exact(wl, 1)
    assert g["dev_err"] == k3mla.DEV_BAD_PAGE
    tbl_o = tbl.copy()
    tbl_o[9, 5] = -1                     # the oracle reads the bad id as the zero row it stands for
    wl.block_table = tbl_o
    _bitwise(g, oracle_layer(wl, 1))
    assert (g["out"][10] == 0).all() and (g["argmax"][10] == -1).all()


def test_exact_heavy_tailed_rows(gpu_lib):
    wl = synth.make_custom([700, 1500, 33], seed=701, device="cuda", row_scale=(0.25, 4.0))
    wl.slab[wl.block_table[0, 9], 0, 5, :] *= 6
    g = _exact(wl, 0)
    assert g["dev_err"] == 0
    _bitwise(g, oracle_layer(wl, 0))


def test_exact_at_the_longest_context(gpu_lib):
    # the mode's largest context (one row's exps fill the softmax kernel's shared memory), heavy-tailed
    # rows, beside a short slot; max_ctx not a whole number of pages
    wl = synth.make_custom([51200, 77], seed=702, device="cuda", row_scale=(0.25, 4.0))
    g = _exact(wl, 0, max_ctx=51200)
    assert g["dev_err"] == 0
    _bitwise(g, oracle_layer(wl, 0))


def test_exact_padding_bucket(gpu_lib):
    wl = synth.make_workload("padding128", device="cuda")
    g = _exact(wl, 0)
    _bitwise(g, oracle_layer(wl, 0))


def test_exact_full_size_sampled(gpu_lib):
    wl = synth.make_workload("steady64", device="cuda", n_layers=1)
    g = _exact(wl, 0, max_ctx=4096)
    assert g["dev_err"] == 0
    _bitwise(g, oracle_layer(wl, 0, slots=[0, 63]), slots=[0, 63])
    del wl
    torch.cuda.empty_cache()
