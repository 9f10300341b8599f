"""Bitwise invariants of the CUDA path (pegainfer PR #869, "K3: paged latent MLA
KV + absorbed decode", M2 commit: physical page ids never enter the arithmetic, a
-1 entry reads as a zero latent, padding rows behave like a zeroed cache; gates:
paged-vs-permuted and graphs-vs-eager bit-identical)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from paged_latent_attention_k3mla_gb300 import k3mla, synth
from tests.gpu_common import gpu_layer

pytestmark = pytest.mark.gpu
SPLIT, MAXC = 256, 1024


def _wl():
    return synth.make_custom([130, 1, 700, 64, 1000, 333], seed=400, device="cuda", max_pages=16)


def test_page_permutation_is_bitwise_invisible(gpu_lib):
    wl = _wl()
    base = gpu_layer(wl, 0, split=SPLIT, max_ctx=MAXC)
    perm = torch.from_numpy(np.random.default_rng(5).permutation(wl.n_pages)).cuda()
    slab2 = torch.empty_like(wl.slab)
    slab2[perm] = wl.slab
    pn = perm.cpu().numpy()
    tbl2 = np.where(wl.block_table >= 0, pn[np.maximum(wl.block_table, 0)], -1).astype(np.int32)
    r = gpu_layer(wl, 0, split=SPLIT, max_ctx=MAXC, slab=slab2, table=torch.from_numpy(tbl2).cuda())
    assert np.array_equal(base["out"], r["out"]) and np.array_equal(base["argmax"], r["argmax"])


def _padded(wl, n_pad=1, n_empty=1):
    """The workload with padding rows interleaved: before each real slot n_pad rows with all -1
    tables (context drawn like the rest), after it n_empty rows with empty contexts."""
    B = wl.B
    order = []
    for b in range(B):
        order += [("pad", 500 + b + 37 * k) for k in range(n_pad)] + [("real", b)] + [("empty", 0)] * n_empty
    tbl = np.full((len(order), wl.block_table.shape[1]), -1, np.int32)
    ctx = np.zeros(len(order), np.int32)
    idx = []
    for i, (kind, v) in enumerate(order):
        if kind == "real":
            tbl[i] = wl.block_table[v]
            ctx[i] = wl.ctx_len[v]
            idx.append(v)
        else:
            ctx[i] = v
    q_big = torch.zeros((1, len(order), 96, 192), dtype=torch.bfloat16, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(9)
    q_big[0] = torch.randn(len(order), 96, 192, generator=g, device="cuda").to(torch.bfloat16)
    real_rows = [i for i, (k, _) in enumerate(order) if k == "real"]
    q_big[0, real_rows] = wl.q[0, idx]
    big = synth.Workload(name="padded", seed=0, n_layers=1, B=len(order), ctx_len=ctx, block_table=tbl,
                         n_pages=wl.n_pages, device="cuda", q=q_big, w_kv_b=wl.w_kv_b, slab=wl.slab,
                         new_c=wl.new_c, new_rope=wl.new_rope)
    empty_rows = [i for i, (k, _) in enumerate(order) if k == "empty"]
    pad_rows = [i for i, (k, _) in enumerate(order) if k == "pad"]
    return big, real_rows, idx, empty_rows, pad_rows


@pytest.mark.parametrize("split,n_pad,n_empty", [(SPLIT, 1, 1), (MAXC, 5, 6)])
def test_padding_slots_leave_real_slots_bitwise_unchanged(gpu_lib, split, n_pad, n_empty):
    # (MAXC, 5, 6): one split per slot and 72 rows, so the padded batch's absorption runs with 128
    # slots per CTA and its expansion over two 64-slot tiles, while the 6 slots fit one of each
    wl = _wl()
    base = gpu_layer(wl, 0, split=split, max_ctx=MAXC)
    big, real_rows, idx, empty_rows, pad_rows = _padded(wl, n_pad, n_empty)
    assert (big.B > 64) == (n_pad + n_empty + 1 > 10)
    r = gpu_layer(big, 0, split=split, max_ctx=MAXC)
    assert np.array_equal(r["out"][real_rows], base["out"][idx])
    assert np.array_equal(r["argmax"][real_rows], base["argmax"][idx])
    assert np.all(r["out"][empty_rows] == 0) and np.all(r["argmax"][empty_rows] == -1)
    assert np.all(r["out"][pad_rows] == 0) and np.all(r["argmax"][pad_rows] == 0)


def test_minus_one_equals_a_physical_zero_page(gpu_lib):
    wl = _wl()
    tbl_a = wl.block_table.copy()
    tbl_a[0, 1] = -1
    tbl_a[2, 4] = -1
    zero_page = int(np.setdiff1d(np.arange(wl.n_pages), wl.block_table[wl.block_table >= 0])[0])
    wl.slab[zero_page] = 0
    tbl_b = wl.block_table.copy()
    tbl_b[0, 1] = zero_page
    tbl_b[2, 4] = zero_page
    ra = gpu_layer(wl, 0, split=SPLIT, max_ctx=MAXC, table=torch.from_numpy(tbl_a).cuda())
    rb = gpu_layer(wl, 0, split=SPLIT, max_ctx=MAXC, table=torch.from_numpy(tbl_b).cuda())
    assert np.array_equal(ra["out"], rb["out"]) and np.array_equal(ra["argmax"], rb["argmax"])


def test_stale_nan_rows_past_the_context_do_not_leak(gpu_lib):
    wl = _wl()
    base = gpu_layer(wl, 0, split=SPLIT, max_ctx=MAXC)
    used = set()
    for b in range(wl.B):
        n = int(wl.ctx_len[b])
        last = int(wl.block_table[b, (n - 1) // 64])
        if n % 64:
            wl.slab[last, 0, n % 64:, :] = float("nan")
        used.update(int(x) for x in wl.block_table[b] if x >= 0)
    for p in range(wl.n_pages):
        if p not in used:
            wl.slab[p] = float("nan")
    r = gpu_layer(wl, 0, split=SPLIT, max_ctx=MAXC)
    assert np.array_equal(base["out"], r["out"]) and np.array_equal(base["argmax"], r["argmax"])


def test_bad_page_id_is_flagged_and_read_as_zero(gpu_lib):
    wl = _wl()
    tbl_bad = wl.block_table.copy()
    tbl_bad[2, 3] = wl.n_pages + 5
    tbl_neg = wl.block_table.copy()
    tbl_neg[2, 3] = -1
    rb = gpu_layer(wl, 0, split=SPLIT, max_ctx=MAXC, table=torch.from_numpy(tbl_bad).cuda())
    rn = gpu_layer(wl, 0, split=SPLIT, max_ctx=MAXC, table=torch.from_numpy(tbl_neg).cuda())
    assert rb["dev_err"] & k3mla.DEV_BAD_PAGE
    assert np.array_equal(rb["out"], rn["out"])


def test_context_past_the_table_is_clamped_and_flagged(gpu_lib):
    wl = synth.make_custom([256, 100], seed=401, device="cuda", max_pages=4)
    ok = gpu_layer(wl, 0, split=SPLIT, max_ctx=256)
    ctx = torch.tensor([300, 100], dtype=torch.int32, device="cuda")
    r = gpu_layer(wl, 0, split=SPLIT, max_ctx=256, ctx=ctx)
    assert r["dev_err"] & k3mla.DEV_CTX
    assert np.array_equal(r["out"], ok["out"])


def test_repeat_runs_and_graph_replay_are_bitwise_identical(gpu_lib):
    wl = _wl()
    B = wl.B
    table = torch.from_numpy(wl.block_table).cuda()
    ctx = torch.from_numpy(wl.ctx_len).cuda()
    q_abs = torch.empty(B, 96, 576, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(B, 96, 128, dtype=torch.bfloat16, device="cuda")
    am = torch.empty(B, 96, dtype=torch.int32, device="cuda")
    ws = torch.empty(k3mla.decode_workspace_bytes(B, MAXC, SPLIT), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()

    def step():
        k3mla.absorb_q(wl.q[0], wl.w_kv_b[0], q_abs)
        k3mla.paged_decode(q_abs, wl.slab, 0, table, ctx, wl.w_kv_b[0], wl.scale_bits, out, ws, MAXC, SPLIT,
                           argmax=am)

    with torch.cuda.stream(s):
        step()
    torch.cuda.synchronize()
    eager1 = (out.clone(), am.clone())
    with torch.cuda.stream(s):
        step()
    torch.cuda.synchronize()
    assert torch.equal(out, eager1[0]) and torch.equal(am, eager1[1])
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step()
    out.zero_()
    am.zero_()
    for _ in range(3):
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager1[0]) and torch.equal(am, eager1[1])
