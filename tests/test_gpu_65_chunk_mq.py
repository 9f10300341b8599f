"""The multi-query form of chunked prefill (k3mla_chunk_decode) on the GPU.

Each token row of a chunk gets the causal attention of the token-by-token loop (PR #869
description, follow-ups: chunked prefill).  The multi-query kernel runs up to four consecutive
rows of one slot in one unit, a row per TMEM quarter; a row's arithmetic is the same as that of
its own view decoded by k3mla_paged_decode with one split, so the two are compared bit for bit
(output and argmax), and the multi-query path is also checked against the oracle's chain at the
decode's bar.  Cases: chunk sizes that are not multiples of four (1, 3, 5, 7), an empty chunk,
chunks from position 0 and across page boundaries, a hole (-1 page) in a prefix, rows outside
every slot's range, a context past max_ctx (clamped and flagged), and long chunks after long
prefixes."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from paged_latent_attention_k3mla_gb300 import k3mla, synth
from tests.gpu_common import compare

pytestmark = pytest.mark.gpu

H, V, ROW, LORA = 96, 128, 576, 512


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _setup(prefix, chunk, seed, hole=None, extra_rows=0):
    ctx = [p + n for p, n in zip(prefix, chunk)]
    wl = synth.make_custom([max(c, 1) for c in ctx], n_layers=2, seed=seed, device="cuda")
    pos0 = np.asarray(prefix, np.int32)
    row_start = np.concatenate([[0], np.cumsum(chunk)]).astype(np.int32)
    R = int(row_start[-1]) + extra_rows
    g = torch.Generator(device="cuda").manual_seed(seed + 1)
    c = torch.randn(R, LORA, generator=g, device="cuda").to(torch.bfloat16)
    r = torch.randn(R, ROW - LORA, generator=g, device="cuda").to(torch.bfloat16)
    q = torch.randn(R, H, 192, generator=g, device="cuda").to(torch.bfloat16)
    tbl = wl.block_table.copy()
    if hole is not None:
        tbl[hole] = -1
    table = _dev(tbl)
    k3mla.append_latent_rows(wl.slab, 1, table, _dev(pos0), _dev(row_start), c, r, max_rows=max(max(chunk), 1))
    q_abs = torch.empty(R, H, ROW, dtype=torch.bfloat16, device="cuda")
    k3mla.absorb_q(q, wl.w_kv_b[1], q_abs)
    return wl, tbl, table, pos0, row_start, q, q_abs, R


def _mq(wl, table, pos0, row_start, q_abs, R, max_ctx):
    ws = torch.empty(k3mla.chunk_decode_workspace_bytes(len(pos0), R, max_ctx), dtype=torch.uint8, device="cuda")
    ws.fill_(0xFF)  # stale workspace
    out = torch.full((R, H, V), float("nan"), dtype=torch.bfloat16, device="cuda")
    am = torch.full((R, H), -7, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    k3mla.chunk_decode(q_abs, wl.slab, 1, table, _dev(pos0), _dev(row_start), wl.w_kv_b[1], wl.scale_bits, out, ws,
                       max_ctx, argmax=am, dev_err=err)
    torch.cuda.synchronize()
    return synth.bf16_bits(out), am.cpu().numpy(), int(err.item())


def _views(wl, table, pos0, row_start, q_abs, R, max_ctx):
    M = table.shape[1]
    vt = torch.empty(R, M, dtype=torch.int32, device="cuda")
    vc = torch.empty(R, dtype=torch.int32, device="cuda")
    k3mla.chunk_views(table, _dev(pos0), _dev(row_start), vt, vc)
    whole = -(-min(max_ctx, M * 64) // 128) * 128     # one split holds every view's context
    ws = torch.empty(k3mla.decode_workspace_bytes(R, max_ctx, whole), dtype=torch.uint8, device="cuda")
    out = torch.full((R, H, V), float("nan"), dtype=torch.bfloat16, device="cuda")
    am = torch.full((R, H), -7, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    k3mla.paged_decode(q_abs, wl.slab, 1, vt, vc, wl.w_kv_b[1], wl.scale_bits, out, ws, max_ctx, whole,
                       argmax=am, dev_err=err)
    torch.cuda.synchronize()
    return synth.bf16_bits(out), am.cpu().numpy(), int(err.item()), vt.cpu().numpy(), vc.cpu().numpy()


@pytest.mark.parametrize("prefix,chunk,hole", [
    ([0, 100, 1, 300, 63], [16, 5, 7, 1, 3], None),        # from position 0, across page boundaries, tiny chunks
    ([5, 130, 0, 64], [64, 0, 9, 33], (3, 0)),              # an empty chunk; slot 3 has a hole in its prefix
])
def test_rows_equal_their_one_split_views_bitwise(gpu_lib, prefix, chunk, hole):
    wl, tbl, table, pos0, row_start, q, q_abs, R = _setup(prefix, chunk, seed=650 + len(chunk), hole=hole)
    max_ctx = table.shape[1] * 64
    out, am, err = _mq(wl, table, pos0, row_start, q_abs, R, max_ctx)
    vout, vam, verr, _, _ = _views(wl, table, pos0, row_start, q_abs, R, max_ctx)
    assert err == 0 and verr == 0
    assert np.array_equal(out, vout), int((out != vout).sum())
    assert np.array_equal(am, vam)


def test_matches_the_oracle_chain(gpu_lib):
    prefix, chunk = [0, 100, 1, 300], [16, 5, 7, 1]
    wl, tbl, table, pos0, row_start, q, q_abs, R = _setup(prefix, chunk, seed=660)
    max_ctx = table.shape[1] * 64
    out, am, err = _mq(wl, table, pos0, row_start, q_abs, R, max_ctx)
    assert err == 0
    ovt, ovc = oracle.chunk_views(tbl, pos0, row_start, R)
    w = synth.bf16_bits(wl.w_kv_b[1])
    o = oracle.decode(oracle.absorb(synth.bf16_bits(q), w), synth.bf16_bits(wl.slab), 1, ovt, ovc, w, wl.scale_bits,
                      nthreads=8, probs_stride=int(ovc.max()))
    o["slots"] = list(range(R))
    ok, stats = compare(dict(out=out, argmax=am), o, ovc, name="chunk_mq")
    print("multi-query chunk decode:", stats)
    assert ok, stats


def test_rows_outside_every_slot_and_a_clamped_context(gpu_lib):
    # rows past row_start[B] get zero output and argmax -1; a max_ctx below the last row's context
    # clamps it (flagged), exactly as k3mla_paged_decode clamps ctx_len
    prefix, chunk = [40, 0], [9, 6]
    wl, tbl, table, pos0, row_start, q, q_abs, R = _setup(prefix, chunk, seed=670, extra_rows=5)
    out, am, err = _mq(wl, table, pos0, row_start, q_abs, R, table.shape[1] * 64)
    assert err == 0
    n = int(row_start[-1])
    assert np.all(out[n:] == 0) and np.all(am[n:] == -1)
    vout, vam, _, _, vc = _views(wl, table, pos0, row_start, q_abs, R, table.shape[1] * 64)
    assert np.array_equal(out, vout) and np.array_equal(am, vam)
    max_ctx = 45                                        # slot 0's rows 5.. have contexts 46..49
    out2, am2, err2 = _mq(wl, table, pos0, row_start, q_abs, R, max_ctx)
    assert err2 == k3mla.DEV_CTX
    vout2, vam2, verr2, _, _ = _views(wl, table, pos0, row_start, q_abs, R, max_ctx)
    assert verr2 == k3mla.DEV_CTX
    assert np.array_equal(out2, vout2) and np.array_equal(am2, vam2)
    # packed rows that start after row 0: rows before row_start[0] belong to no slot either
    shifted = row_start + 3
    out3, am3, err3 = _mq(wl, table, pos0, shifted, q_abs, R, table.shape[1] * 64)
    assert err3 == 0
    assert np.all(out3[:3] == 0) and np.all(am3[:3] == -1)
    vout3, vam3, _, _, _ = _views(wl, table, pos0, shifted, q_abs, R, table.shape[1] * 64)
    assert np.array_equal(out3, vout3) and np.array_equal(am3, vam3)


def test_long_chunks_after_long_prefixes(gpu_lib):
    # 300-token chunks after ~3,000-token prefixes: 75 groups a slot, units over several waves; and a
    # chunk after a 9,000-token prefix, whose rows' contexts (one split each) span 142 pages
    prefix, chunk = [3000, 2881, 64, 9000], [300, 300, 130, 21]
    wl, tbl, table, pos0, row_start, q, q_abs, R = _setup(prefix, chunk, seed=680)
    max_ctx = table.shape[1] * 64
    out, am, err = _mq(wl, table, pos0, row_start, q_abs, R, max_ctx)
    vout, vam, verr, _, _ = _views(wl, table, pos0, row_start, q_abs, R, max_ctx)
    assert err == 0 and verr == 0
    assert np.array_equal(out, vout), int((out != vout).sum())
    assert np.array_equal(am, vam)


def test_argument_checks(gpu_lib):
    wl, tbl, table, pos0, row_start, q, q_abs, R = _setup([10], [4], seed=690)
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    out = torch.empty(R, H, V, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(k3mla.K3mlaError):   # workspace too small
        k3mla.chunk_decode(q_abs, wl.slab, 1, table, _dev(pos0), _dev(row_start), wl.w_kv_b[1], wl.scale_bits,
                           out, ws, 64)
    assert k3mla.chunk_decode_workspace_bytes(0, 4, 64) == 0


def test_replay_from_a_cuda_graph_is_bitwise_the_eager_call(gpu_lib):
    # the group builder, the multi-query split kernel and the merge capture like the rest of the library
    wl, tbl, table, pos0, row_start, q, q_abs, R = _setup([0, 70, 200], [13, 4, 64], seed=695)
    max_ctx = table.shape[1] * 64
    eager, eager_am, err = _mq(wl, table, pos0, row_start, q_abs, R, max_ctx)
    assert err == 0
    ws = torch.empty(k3mla.chunk_decode_workspace_bytes(len(pos0), R, max_ctx), dtype=torch.uint8, device="cuda")
    out = torch.full((R, H, V), float("nan"), dtype=torch.bfloat16, device="cuda")
    am = torch.full((R, H), -7, dtype=torch.int32, device="cuda")
    p0, rs = _dev(pos0), _dev(row_start)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):  # the first call sets the kernels' attributes outside the capture
        k3mla.chunk_decode(q_abs, wl.slab, 1, table, p0, rs, wl.w_kv_b[1], wl.scale_bits, out, ws, max_ctx,
                           argmax=am, stream=s)
    torch.cuda.synchronize()
    out.fill_(float("nan"))
    am.fill_(-7)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        k3mla.chunk_decode(q_abs, wl.slab, 1, table, p0, rs, wl.w_kv_b[1], wl.scale_bits, out, ws, max_ctx,
                           argmax=am, stream=s)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(synth.bf16_bits(out), eager)
    assert np.array_equal(am.cpu().numpy(), eager_am)
