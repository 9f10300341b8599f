"""Chunked prefill on the GPU against the oracle.

* k3mla_append_latent_rows: bitwise (a copy into the rows the size_t indices name),
  ragged chunks across page boundaries, an empty chunk and an unmapped page
  (skipped and flagged).
* k3mla_chunk_views: the per-token tables and context lengths, bitwise.
* The chunk's causal attention -- absorption, views, paged decode over one view per
  token -- against the oracle's chain on the same views, at the decode's bar (4 bf16
  ULP of each row's largest magnitude, argmax up to the 1-ULP coin flips): short
  chunks in full, and 300-token chunks after ~3,000-token prefixes on sampled views.  The
  oracle's views are pinned to the token-by-token loop in the oracle's own tests."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from paged_latent_attention_k3mla_gb300 import k3mla, synth
from tests.gpu_common import compare

pytestmark = pytest.mark.gpu

H, V, ROW, LORA = 96, 128, 576, 512


def _case(prefix, chunk, seed):
    ctx = [p + n for p, n in zip(prefix, chunk)]
    wl = synth.make_custom(ctx, n_layers=2, seed=seed, device="cuda")
    pos0 = np.asarray(prefix, np.int32)
    row_start = np.concatenate([[0], np.cumsum(chunk)]).astype(np.int32)
    R = int(row_start[-1])
    g = torch.Generator(device="cuda").manual_seed(seed + 1)
    c = torch.randn(R, LORA, generator=g, device="cuda").to(torch.bfloat16)
    r = torch.randn(R, ROW - LORA, generator=g, device="cuda").to(torch.bfloat16)
    q = torch.randn(R, H, 192, generator=g, device="cuda").to(torch.bfloat16)
    return wl, pos0, row_start, c, r, q, R


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def test_append_rows_matches_oracle(gpu_lib):
    wl, pos0, row_start, c, r, _, R = _case([0, 60, 1, 130, 7], [70, 5, 0, 64, 3], seed=600)
    tbl = wl.block_table.copy()
    tbl[4, 0] = -1                                       # slot 4's rows 7..9 land in an unmapped page
    want = synth.bf16_bits(wl.slab).copy()
    assert oracle.append_rows(want, 1, tbl, pos0, row_start, synth.bf16_bits(c), synth.bf16_bits(r)) == 3
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    k3mla.append_latent_rows(wl.slab, 1, _dev(tbl), _dev(pos0), _dev(row_start), c, r, max_rows=70, dev_err=err)
    torch.cuda.synchronize()
    assert np.array_equal(synth.bf16_bits(wl.slab), want)
    assert err.item() == k3mla.DEV_UNMAPPED


def test_chunked_prefill_attention_matches_oracle(gpu_lib):
    # a prompt prefilled from scratch, chunks after long and short prefixes, a one-token chunk
    wl, pos0, row_start, c, r, q, R = _case([0, 100, 1, 300], [16, 5, 64, 1], seed=601)
    B, M = wl.block_table.shape
    table = _dev(wl.block_table)
    oslab = synth.bf16_bits(wl.slab).copy()          # the oracle appends on its own copy
    oracle.append_rows(oslab, 1, wl.block_table, pos0, row_start, synth.bf16_bits(c), synth.bf16_bits(r))
    k3mla.append_latent_rows(wl.slab, 1, table, _dev(pos0), _dev(row_start), c, r, max_rows=64)
    vt = torch.full((R + 1, M), 7, dtype=torch.int32, device="cuda")   # one view past the chunk
    vc = torch.full((R + 1,), 7, dtype=torch.int32, device="cuda")
    k3mla.chunk_views(table, _dev(pos0), _dev(row_start), vt, vc)
    q_abs = torch.empty(R, H, ROW, dtype=torch.bfloat16, device="cuda")
    k3mla.absorb_q(q, wl.w_kv_b[1], q_abs)
    max_ctx = M * 64
    split = k3mla.SPLIT_AUTO
    ws = torch.empty(k3mla.decode_workspace_bytes(R, max_ctx, split), dtype=torch.uint8, device="cuda")
    out = torch.full((R, H, V), float("nan"), dtype=torch.bfloat16, device="cuda")
    am = torch.full((R, H), -7, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    k3mla.paged_decode(q_abs, wl.slab, 1, vt[:R], vc[:R], wl.w_kv_b[1], wl.scale_bits, out, ws, max_ctx, split,
                       argmax=am, dev_err=err)
    torch.cuda.synchronize()
    assert err.item() == 0

    ovt, ovc = oracle.chunk_views(wl.block_table, pos0, row_start, R + 1)
    assert np.array_equal(vt.cpu().numpy(), ovt) and np.array_equal(vc.cpu().numpy(), ovc)
    w = synth.bf16_bits(wl.w_kv_b[1])
    o = oracle.decode(oracle.absorb(synth.bf16_bits(q), w), oslab, 1, ovt[:R], ovc[:R], w, wl.scale_bits,
                      nthreads=8, probs_stride=int(ovc.max()))
    o["slots"] = list(range(R))
    gpu = dict(out=synth.bf16_bits(out), argmax=am.cpu().numpy())
    ok, stats = compare(gpu, o, ovc[:R], name="chunked_prefill")
    print("chunked prefill:", stats)
    assert ok, stats
    assert np.array_equal(synth.bf16_bits(wl.slab), oslab)   # and the GPU append left the same slab


def test_long_chunks_after_long_prefixes_sampled(gpu_lib):
    # two slots, each a 300-token chunk after a prefix of ~3,000 tokens: 600 views (ten absorption
    # tiles, a multi-wave split grid); the oracle checks sampled views -- each chunk's first token,
    # the tokens on either side of a page boundary inside it, and its last token
    prefix, chunk = [3000, 2881], [300, 300]
    wl, pos0, row_start, c, r, q, R = _case(prefix, chunk, seed=603)
    B, M = wl.block_table.shape
    table = _dev(wl.block_table)
    oslab = synth.bf16_bits(wl.slab).copy()
    oracle.append_rows(oslab, 1, wl.block_table, pos0, row_start, synth.bf16_bits(c), synth.bf16_bits(r))
    k3mla.append_latent_rows(wl.slab, 1, table, _dev(pos0), _dev(row_start), c, r, max_rows=300)
    vt = torch.empty(R, M, dtype=torch.int32, device="cuda")
    vc = torch.empty(R, dtype=torch.int32, device="cuda")
    k3mla.chunk_views(table, _dev(pos0), _dev(row_start), vt, vc)
    q_abs = torch.empty(R, H, ROW, dtype=torch.bfloat16, device="cuda")
    k3mla.absorb_q(q, wl.w_kv_b[1], q_abs)
    max_ctx = M * 64
    split = k3mla.SPLIT_AUTO
    ws = torch.empty(k3mla.decode_workspace_bytes(R, max_ctx, split), dtype=torch.uint8, device="cuda")
    out = torch.full((R, H, V), float("nan"), dtype=torch.bfloat16, device="cuda")
    am = torch.full((R, H), -7, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    k3mla.paged_decode(q_abs, wl.slab, 1, vt, vc, wl.w_kv_b[1], wl.scale_bits, out, ws, max_ctx, split,
                       argmax=am, dev_err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert np.array_equal(synth.bf16_bits(wl.slab), oslab)

    ovt, ovc = oracle.chunk_views(wl.block_table, pos0, row_start, R)
    assert np.array_equal(vt.cpu().numpy(), ovt) and np.array_equal(vc.cpu().numpy(), ovc)
    sel = []
    for b in range(B):
        j_edge = 64 - prefix[b] % 64           # the chunk's first token on a new page
        sel += [int(row_start[b]) + j for j in (0, j_edge - 1, j_edge, chunk[b] - 1)]
    w = synth.bf16_bits(wl.w_kv_b[1])
    stride = int(ovc[sel].max())
    o = oracle.decode(oracle.absorb(synth.bf16_bits(q)[sel], w), oslab, 1, ovt[sel], ovc[sel], w, wl.scale_bits,
                      nthreads=8, probs_stride=stride)
    o["slots"] = sel
    gpu = dict(out=synth.bf16_bits(out), argmax=am.cpu().numpy())
    ok, stats = compare(gpu, o, ovc, name="long_chunks")
    print("long chunks:", split, stats)
    assert ok, stats


def test_chunk_path_copy_and_exact_mode_replay_from_a_cuda_graph(gpu_lib):
    """The calls beyond the decode step are graph-capturable like the rest: a chunk step (row append,
    views, absorption, decode), a page copy and the exact-chain decode, captured once and replayed,
    give the eager results bit for bit."""
    wl, pos0, row_start, c, r, q, R = _case([40, 200], [8, 3], seed=602)
    B, M = wl.block_table.shape
    table, p0, rs = _dev(wl.block_table), _dev(pos0), _dev(row_start)
    vt = torch.empty(R, M, dtype=torch.int32, device="cuda")
    vc = torch.empty(R, dtype=torch.int32, device="cuda")
    q_abs = torch.empty(R, H, ROW, dtype=torch.bfloat16, device="cuda")
    max_ctx = M * 64
    split = k3mla.SPLIT_AUTO
    ws = torch.empty(k3mla.decode_workspace_bytes(R, max_ctx, split), dtype=torch.uint8, device="cuda")
    out = torch.empty(R, H, V, dtype=torch.bfloat16, device="cuda")
    ex_ws = torch.empty(k3mla.decode_exact_workspace_bytes(B, max_ctx), dtype=torch.uint8, device="cuda")
    ex_out = torch.empty(B, H, V, dtype=torch.bfloat16, device="cuda")
    ctx = torch.from_numpy(wl.ctx_len).cuda()
    spare = torch.zeros(2, 2, 64, ROW, dtype=torch.bfloat16, device="cuda")
    src_ids = torch.tensor([int(wl.block_table[1, 0]), int(wl.block_table[0, 0])], dtype=torch.int32, device="cuda")
    dst_ids = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()

    def step():
        k3mla.append_latent_rows(wl.slab, 1, table, p0, rs, c, r, max_rows=8)
        k3mla.chunk_views(table, p0, rs, vt, vc)
        k3mla.absorb_q(q, wl.w_kv_b[1], q_abs)
        k3mla.paged_decode(q_abs, wl.slab, 1, vt, vc, wl.w_kv_b[1], wl.scale_bits, out, ws, max_ctx, split)
        k3mla.copy_pages(spare, wl.slab, src_ids, dst_ids)
        k3mla.decode_exact(wl.q[1], wl.slab, 1, table, ctx, wl.w_kv_b[1], wl.scale_bits, ex_out, ex_ws, max_ctx)

    with torch.cuda.stream(s):
        step()
    torch.cuda.synchronize()
    eager = [t.clone() for t in (out, spare, ex_out, vc)]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step()
    for t in (out, spare, ex_out, vc):
        t.zero_()
    for _ in range(2):
        graph.replay()
        torch.cuda.synchronize()
        assert all(torch.equal(a, b) for a, b in zip((out, spare, ex_out, vc), eager))
