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


def _graph_decode(q, slab, w, table, ctx, max_ctx, scale_bits, split=k3mla.SPLIT_AUTO):
    """Absorption + paged decode of one layer, run eagerly once and then captured in a CUDA graph and
    replayed twice into cleared (NaN) outputs; the replay must equal the eager run bit for bit.
    Returns the replayed out / argmax as numpy arrays and the device error word."""
    B = q.shape[0]
    q_abs = torch.empty(B, 96, 576, dtype=torch.bfloat16, device="cuda")
    out = torch.full((B, 96, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    am = torch.full((B, 96), -7, dtype=torch.int32, device="cuda")
    ws = torch.full((k3mla.decode_workspace_bytes(B, max_ctx, split),), 0xFF, dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()

    def step():
        k3mla.absorb_q(q, w, q_abs)
        k3mla.paged_decode(q_abs, slab, 0, table, ctx, w, scale_bits, out, ws, max_ctx, split, argmax=am,
                           dev_err=err)

    with torch.cuda.stream(s):
        step()
    torch.cuda.synchronize()
    eager = (synth.bf16_bits(out), am.cpu().numpy())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step()
    out.fill_(float("nan"))
    am.fill_(-7)
    ws.fill_(0xFF)
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    res = (synth.bf16_bits(out), am.cpu().numpy())
    assert np.array_equal(res[0], eager[0]) and np.array_equal(res[1], eager[1])
    return res[0], res[1], int(err.item())


def test_padding128_rows_are_bitwise_invariant_under_the_default_split(gpu_lib):
    """The 128-row padding workload (40 % all -1 padding rows, contexts <= 256, -1 holes, one empty
    slot) decoded with the library's default split (K3MLA_SPLIT_AUTO, nothing pinned by hand), every
    batch from a CUDA graph replay.  Its real rows must come out with the same bits when they are
    decoded (a) in the full 128-row batch; (b) reordered, on physically permuted pages, among added
    all -1 padding rows and long neighbours with several splits each, under a larger max_ctx (the
    launch then has f32 partials, the merge path and 16-slot expansion tiles instead of 64-slot
    ones); (c) five at a time in small batches."""
    wl = synth.make_workload("padding128", device="cuda")
    w, q0 = wl.w_kv_b[0], wl.q[0]
    pad = (wl.block_table < 0).all(axis=1) & (wl.ctx_len > 0)
    real = [b for b in range(wl.B) if not pad[b]]
    assert len(real) > 60 and pad.sum() > 30 and (wl.ctx_len[real] == 0).sum() == 1
    g = torch.Generator(device="cuda").manual_seed(44)

    # (a) the workload as drawn
    out_a, am_a, err_a = _graph_decode(q0, wl.slab, w, torch.from_numpy(wl.block_table).cuda(),
                                       torch.from_numpy(wl.ctx_len).cuda(), 256, wl.scale_bits)
    assert err_a == 0
    assert np.all(out_a[pad] == 0)
    empty = [b for b in real if wl.ctx_len[b] == 0][0]
    assert np.all(out_a[empty] == 0) and np.all(am_a[empty] == -1)

    # (b) reversed real rows, permuted pages, extra padding rows and multi-split neighbours
    perm = np.random.default_rng(6).permutation(wl.n_pages)
    slab2 = torch.empty_like(wl.slab)
    slab2[torch.from_numpy(perm).cuda()] = wl.slab
    long_ctx = [9000, 4097, 20000]
    max_ctx = 20000
    mp = -(-max_ctx // 64)
    rows = list(reversed(real))
    n_extra_pad = 10
    B2 = len(rows) + len(long_ctx) + n_extra_pad
    tbl = np.full((B2, mp), -1, np.int32)
    ctx = np.zeros(B2, np.int32)
    q2 = (torch.randn(B2, 96, 192, generator=g, device="cuda")).to(torch.bfloat16)
    order = []  # (kind, source row)
    rng = np.random.default_rng(7)
    slots = list(range(B2))
    rng.shuffle(slots)
    it = iter(slots)
    for b in rows:
        i = next(it)
        t = wl.block_table[b]
        tbl[i, :t.shape[0]] = np.where(t >= 0, perm[np.maximum(t, 0)], -1)
        ctx[i] = wl.ctx_len[b]
        q2[i] = q0[b]
        order.append((i, b))
    for n in long_ctx:
        i = next(it)
        tbl[i, :-(-n // 64)] = rng.integers(0, wl.n_pages, size=-(-n // 64))
        ctx[i] = n
    for _ in range(n_extra_pad):
        i = next(it)
        ctx[i] = int(rng.integers(1, 257))
    assert max(k3mla.slot_split_tokens(n) for n in long_ctx) < 20000  # the neighbours have several splits
    out_b, am_b, err_b = _graph_decode(q2, slab2, w, torch.from_numpy(tbl).cuda(), torch.from_numpy(ctx).cuda(),
                                       max_ctx, wl.scale_bits)
    assert err_b == 0
    for i, b in order:
        assert np.array_equal(out_b[i], out_a[b]), f"row {b} differs in the mixed batch"
        assert np.array_equal(am_b[i], am_a[b]), f"argmax of row {b} differs in the mixed batch"

    # (c) five real rows at a time (absorption and expansion tiles of a small batch)
    for k in range(0, 20, 5):
        sel = real[k:k + 5]
        t = torch.from_numpy(np.ascontiguousarray(wl.block_table[sel])).cuda()
        c = torch.from_numpy(np.ascontiguousarray(wl.ctx_len[sel])).cuda()
        out_c, am_c, err_c = _graph_decode(q0[sel].contiguous(), wl.slab, w, t, c, 300, wl.scale_bits)
        assert err_c == 0
        assert np.array_equal(out_c, out_a[sel]) and np.array_equal(am_c, am_a[sel])


@pytest.mark.parametrize("split", [k3mla.SPLIT_AUTO, 256])
def test_max_ctx_does_not_change_a_slots_bits(gpu_lib, split):
    """max_ctx sizes the grid only: the same slots under max_ctx 1024 and 8192 (4 and 32 launch splits
    at a 256-token split) give the same bits, for the default rule and a fixed split."""
    wl = _wl()
    a = gpu_layer(wl, 0, split=split, max_ctx=MAXC)
    b = gpu_layer(wl, 0, split=split, max_ctx=8192)
    assert a["dev_err"] == 0 and b["dev_err"] == 0
    assert np.array_equal(a["out"], b["out"]) and np.array_equal(a["argmax"], b["argmax"])
