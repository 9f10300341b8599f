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


def test_the_chains_exp_equals_the_double_exponential_rounded_to_f32(gpu_lib):
    # The mode's e_t = f32 of the double exponential (the chain's definition), evaluated first in f32
    # pairs: wherever the pair decided, the result must be the f32 nearest to e^x, the same bits as
    # numpy's double exp rounded once; where it handed over to the double exp (arguments whose e^x lies
    # close to an f32 rounding boundary, or outside [-87, 0]), the two double exponentials may differ by
    # one f32 unit at most.  Arguments: 4M uniform in [-90, 0.5], every landed score difference s - m of
    # two bf16 values in [-16, 16] against m in a few rows' maxima, and edge values.
    g = np.random.default_rng(701)
    xs = [g.uniform(-90.0, 0.5, size=4 << 20).astype(np.float32)]
    b = np.arange(0, 1 << 16, dtype=np.uint32)
    bf = (b << 16).view(np.float32)
    bf = bf[np.isfinite(bf) & (np.abs(bf) <= 16.0)]
    for m in (np.float32(0.0), np.float32(3.1875), np.float32(7.5), np.float32(15.875)):
        d = (bf[bf <= m] - m).astype(np.float32)
        xs.append(d)
    xs.append(np.array([0.0, -0.0, -1e-30, -1.4e-45, -87.0, -87.00001, -86.99999, -88.7, -103.9, -104.0, 1.0,
                        -0.5, -0.34657359, -0.01083, 0.01083], np.float32))
    x = np.concatenate(xs)
    xt = torch.from_numpy(x).cuda()
    y = torch.empty_like(xt)
    fast = torch.empty(x.size, dtype=torch.int32, device="cuda")
    k3mla.diag_exact_exp(xt, y, fast)
    torch.cuda.synchronize()
    y, fast = y.cpu().numpy(), fast.cpu().numpy().astype(bool)
    with np.errstate(over="ignore", under="ignore"):
        ref = np.exp(x.astype(np.float64)).astype(np.float32)
    yb, rb = y.view(np.uint32).astype(np.int64), ref.view(np.uint32).astype(np.int64)
    assert np.array_equal(yb[fast], rb[fast]), f"{int((yb[fast] != rb[fast]).sum())} fast-path results differ"
    assert np.all(np.abs(yb[~fast] - rb[~fast]) <= 1)
    inside = (x >= -87.0) & (x <= 0.0)
    assert fast[inside].mean() > 0.999, fast[inside].mean()          # the double exp is the exception
    assert not fast[~inside].any()
