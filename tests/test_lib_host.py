"""Host-side tests of libk3mla.so that need no GPU: the library builds and loads,
exports every symbol include/k3mla.h declares, the page pool behaves as the
free-list allocator of pegainfer PR #869 ("K3: paged latent MLA KV + absorbed
decode", M1 commit: claim on a 64-token boundary, release-all on reset, 0 =
full coverage; review comment: expose total / allocated pages), and argument
errors come back as status codes before anything is launched."""
from __future__ import annotations

import ctypes
import os
import re

import numpy as np
import pytest

from paged_latent_attention_k3mla_gb300 import k3mla

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_header_declarations_are_all_exported():
    hdr = open(os.path.join(ROOT, "include", "k3mla.h")).read()
    declared = set(re.findall(r"\b(k3mla_[a-z_]+)\s*\(", hdr))
    assert declared == set(k3mla.EXPORTS), declared ^ set(k3mla.EXPORTS)
    lib = k3mla.load()
    for name in declared:
        assert hasattr(lib, name), name
    nm = os.popen(f"nm -D --defined-only {k3mla._build.LIB}").read()
    for name in declared:
        assert re.search(rf"\bT {name}\b", nm), f"{name} not exported"


def test_pool_claims_on_page_boundaries_and_releases():
    pool = k3mla.Pool(n_slots=3, max_ctx=256)
    assert (pool.n_pages, pool.max_pages) == (12, 4)          # full coverage: 3 slots x 4 pages
    assert pool.stats() == (12, 0)
    assert pool.ensure(0, 1) == 0
    assert pool.stats() == (12, 1)
    assert pool.ensure(0, 64) == 0 and pool.stats()[1] == 1  # still inside page 0
    assert pool.ensure(0, 65) == 0 and pool.stats()[1] == 2  # crossed a 64-token boundary
    t = pool.table()
    assert list(t[0, :2]) == [0, 1] and list(t[0, 2:]) == [-1, -1]
    assert pool.ensure(1, 256) == 0
    assert pool.stats() == (12, 6)
    before = pool.table()[1].copy()
    assert pool.release(1) == 0
    assert pool.stats() == (12, 2)
    assert np.all(pool.table()[1] == -1)
    assert pool.ensure(1, 256) == 0                            # the same ids come back
    assert np.array_equal(pool.table()[1], before)
    pool.close()


def test_pool_ensure_all_is_ensure_slot_by_slot():
    a = k3mla.Pool(n_slots=4, max_ctx=512, n_pages=12, shuffle_seed=3)
    b = k3mla.Pool(n_slots=4, max_ctx=512, n_pages=12, shuffle_seed=3)
    lens = np.array([65, 1, 300, 0], np.int32)
    assert a.ensure_all(lens) == 0
    for s, n in enumerate(lens):
        assert b.ensure(s, int(n)) == 0
    assert np.array_equal(a.table(), b.table()) and a.stats() == b.stats() == (12, 8)
    # slot 2 takes 3 of the 4 free pages, then slot 3 needs 3 and finds 1: it fails alone, unchanged
    assert a.ensure_all(np.array([65, 1, 512, 129], np.int32)) == -2
    assert a.stats() == (12, 11) and (a.table()[3] == -1).all() and (a.table()[2] >= 0).all()
    assert a.ensure_all(np.array([1, 1, 1, 1, 1], np.int32)) == -1    # more lengths than slots
    a.close()
    b.close()


def test_pool_errors_are_all_or_nothing():
    pool = k3mla.Pool(n_slots=2, max_ctx=256, n_pages=5)
    assert pool.ensure(0, 256) == 0                            # 4 pages
    assert pool.ensure(1, 129) == -2                           # needs 3, 1 left: K3MLA_E_NO_PAGES
    assert pool.stats() == (5, 4) and np.all(pool.table()[1] == -1)
    assert pool.ensure(1, 64) == 0
    assert pool.ensure(1, 257) == -4                           # beyond max_ctx: K3MLA_E_CTX
    assert pool.ensure(2, 1) == -3                             # no such slot: K3MLA_E_SLOT
    assert pool.release(7) == -3
    pool.close()


def test_pool_shuffle_is_seeded_and_a_permutation():
    a = k3mla.Pool(n_slots=4, max_ctx=1024, shuffle_seed=99)
    b = k3mla.Pool(n_slots=4, max_ctx=1024, shuffle_seed=99)
    c = k3mla.Pool(n_slots=4, max_ctx=1024, shuffle_seed=100)
    for p in (a, b, c):
        for s in range(4):
            assert p.ensure(s, 1024) == 0
    ta, tb, tc = a.table(), b.table(), c.table()
    assert np.array_equal(ta, tb) and not np.array_equal(ta, tc)
    assert sorted(ta.ravel().tolist()) == list(range(64))      # every page exactly once
    assert not np.array_equal(ta.ravel(), np.arange(64))       # actually scattered


def test_prefix_sharing_counts_references_and_copies_on_write():
    pool = k3mla.Pool(n_slots=3, max_ctx=512, n_pages=10)
    assert pool.ensure(0, 200) == 0                                # 4 pages
    t0 = pool.table()[0, :4].copy()
    assert pool.share_prefix(1, 0, 130) == 0                       # 3 pages shared, no copy
    assert np.array_equal(pool.table()[1, :3], t0[:3]) and pool.table()[1, 3] == -1
    assert [pool.refs(int(p)) for p in t0] == [2, 2, 2, 1]
    assert pool.stats() == (10, 4)                                 # shared pages count once
    assert pool.cow(0, 199) is None                                # page 3 of slot 0 is its own
    cp = pool.cow(1, 129)                                          # slot 1 writes into shared page 2
    assert cp is not None and cp[0] == t0[2] and cp[1] not in t0
    assert pool.table()[1, 2] == cp[1] and pool.refs(int(t0[2])) == 1 and pool.refs(cp[1]) == 1
    assert pool.cow(1, 129) is None                                # now private
    assert pool.stats() == (10, 5)
    assert pool.ensure(1, 300) == 0                                # grows with private pages
    assert pool.release(0) == 0                                    # slot 1 still holds pages 0, 1
    assert pool.refs(int(t0[0])) == 1 and pool.refs(int(t0[3])) == 0
    assert pool.release(1) == 0 and pool.stats() == (10, 0)
    assert all(pool.refs(p) == 0 for p in range(10))
    # errors: non-empty destination, same slot, more pages than the source maps, bad slot / page
    assert pool.ensure(0, 64) == 0 and pool.ensure(1, 1) == 0
    assert pool.share_prefix(1, 0, 64) == -1 and pool.share_prefix(2, 2, 1) == -1
    assert pool.share_prefix(2, 0, 65) == -1 and pool.share_prefix(3, 0, 1) == -3
    assert pool.share_prefix(2, 0, 513) == -4
    assert pool.cow(2, 0) == -4                                    # position not mapped
    assert pool.refs(10) == -1
    pool.close()


def test_copy_on_write_is_all_or_nothing_when_the_pool_is_full():
    pool = k3mla.Pool(n_slots=2, max_ctx=128, n_pages=2)
    assert pool.ensure(0, 128) == 0 and pool.share_prefix(1, 0, 128) == 0
    before = pool.table().copy()
    assert pool.cow(1, 5) == -2                                    # K3MLA_E_NO_PAGES
    assert np.array_equal(pool.table(), before) and pool.refs(int(before[0, 0])) == 2
    pool.close()


def test_invalid_arguments_return_status_without_launching():
    lib = k3mla.load()
    null = None
    # negative batch, bad layer, split not a multiple of the 128-token tile
    assert lib.k3mla_absorb_q(null, null, null, -1, null) == -1
    assert lib.k3mla_append_latent(null, 4, 2, 2, null, 1, null, null, 512, null, 64, 1, null, null) == -1
    assert lib.k3mla_append_latent(null, 4, 2, 0, null, 1, null, null, 511, null, 64, 1, null, null) == -1
    args = [null, null, 4, 1, 0, null, 4, null, null, 0x3D94, null, null, null, 0, 1, 256, 100, null, null]
    assert lib.k3mla_paged_decode(*args) == -1
    args[16] = -128                                            # negative split length
    assert lib.k3mla_paged_decode(*args) == -1
    assert b"invalid sizes" in lib.k3mla_last_error()
    args[16] = 0                                               # the default rule: arguments pass, pointers fail
    assert lib.k3mla_paged_decode(*args) == -1
    assert b"null or misaligned" in lib.k3mla_last_error()
    args[16] = 128
    assert lib.k3mla_paged_decode(*args) == -1                 # null pointers
    assert b"null or misaligned" in lib.k3mla_last_error()
    assert lib.k3mla_absorb_q(null, null, null, 0, null) == 0   # B == 0: nothing to do
    # the fused absorption + append checks both halves' arguments
    fused = [null, null, null, null, 4, 2, 0, null, 1, null, null, 512, null, 64, 1, null, null]
    assert lib.k3mla_absorb_q_append(*fused) == -1              # null pointers
    assert b"k3mla_absorb_q_append: null or misaligned" in lib.k3mla_last_error()
    fused[14] = 0
    assert lib.k3mla_absorb_q_append(*fused) == 0               # B == 0: nothing to do
    fused[6] = 2                                                # layer == n_layers
    assert lib.k3mla_absorb_q_append(*fused) == -1
    assert b"invalid sizes or strides" in lib.k3mla_last_error()
    assert lib.k3mla_diag_umma(5, null, null, null, null) == -1
    assert lib.k3mla_copy_pages(null, 4, null, 4, 2, null, null, 0, null, null) == 0    # n == 0
    assert lib.k3mla_copy_pages(null, 4, null, 4, 2, null, null, 1, null, null) == -1
    assert b"null or misaligned" in lib.k3mla_last_error()
    assert lib.k3mla_copy_pages(null, 4, null, 4, 0, null, null, 1, null, null) == -1   # no layers
    assert lib.k3mla_copy_pages(null, 4, null, 4, 2, null, null, 65536, null, null) == -1


def test_exact_workspace_formula_and_arguments():
    # bf16 scores/probabilities [B][96][max_ctx rounded up to 8] + q_abs [B][96][576] + o_lat [96][B][512],
    # the first two regions rounded up to 256 bytes
    r256 = lambda x: (x + 255) // 256 * 256
    for B, max_ctx in ((1, 130), (64, 4096), (3, 1)):
        want = r256(B * 96 * (-(-max_ctx // 8) * 8) * 2) + r256(B * 96 * 576 * 2) + B * 96 * 512 * 2
        assert k3mla.decode_exact_workspace_bytes(B, max_ctx) == want
    assert k3mla.decode_exact_workspace_bytes(0, 10) == 0
    lib = k3mla.load()
    args = [None, None, 4, 1, 0, None, 4, None, None, 0x3D94, None, None, None, 0, 1, 256, None, None]
    assert lib.k3mla_decode_exact(*args) == -1
    assert b"null or misaligned" in lib.k3mla_last_error()
    args[14] = 0
    assert lib.k3mla_decode_exact(*args) == 0                   # B == 0: nothing to do
    args[4] = 1                                                 # layer == n_layers
    assert lib.k3mla_decode_exact(*args) == -1


def test_workspace_formula():
    # o_lat [96][B][512] bf16, then -- only when a slot can have several splits -- f32 partial O
    # [B][nsplit][96][512], each rounded up to 256 B, then the records [B][nsplit][96][4] f32; nsplit
    # = ceil(max_ctx / split) for a fixed split, ceil(max_ctx / 4096) for the default rule
    r256 = lambda x: (x + 255) // 256 * 256
    for B, max_ctx, split in ((1, 130, 128), (64, 4096, 4096), (8, 32768, 3712), (128, 256, 256),
                              (64, 4096, 0), (8, 32768, 0), (3, 4097, 0), (16, 4096, 512)):
        ns = -(-max_ctx // (split if split else 4096))
        want = r256(B * 96 * 512 * 2) + (r256(B * ns * 96 * 512 * 4) if ns > 1 else 0) + B * ns * 96 * 4 * 4
        assert k3mla.decode_workspace_bytes(B, max_ctx, split) == want, (B, max_ctx, split)
    assert k3mla.decode_workspace_bytes(0, 4096, 128) == 0
    assert k3mla.decode_workspace_bytes(4, 4096, -128) == 0


def test_default_split_rule_depends_on_the_slot_alone():
    """The default rule cuts a slot of n tokens into ceil(n / 4096) splits of equal length rounded up
    to the 128-token tile: at most 4096 tokens, every split non-empty, a function of n alone."""
    for n in list(range(0, 300)) + [4095, 4096, 4097, 5000, 8191, 8192, 8193, 20000, 32768, 51200, 131073]:
        s = k3mla.slot_split_tokens(n)
        assert s % 128 == 0 and 128 <= s <= 4096, (n, s)
        ns = -(-n // s)
        assert ns == -(-n // 4096), (n, s)              # as many splits as 4096-token pieces
        assert n == 0 or (ns - 1) * s < n, (n, s)       # the last split holds tokens
        if 0 < n <= 4096:
            assert s >= n                               # one split: the slot lands o_lat itself
    assert k3mla.slot_split_tokens(32768) == 4096 and k3mla.slot_split_tokens(5000) == 2560
    assert k3mla.slot_split_tokens(1000, 256) == 256    # a fixed split length is used as given
    lib = k3mla.load()
    assert lib.k3mla_slot_split_tokens(100, -1) == -1


def test_layer_call_sizes_and_arguments():
    # q_abs [B][96][576] bf16 (256-aligned), then the decode workspace of the default split
    r256 = lambda x: (x + 255) // 256 * 256
    for B, max_ctx in ((1, 130), (64, 4096), (8, 32768)):
        want = r256(B * 96 * 576 * 2) + k3mla.decode_workspace_bytes(B, max_ctx, 0)
        assert k3mla.decode_layer_workspace_bytes(B, max_ctx) == want
    lib = k3mla.load()
    args = [None, None, None, 4, 1, 0, None, 4, None, None, 512, None, 64, 0x3D94, None, None, None, 0, 1, 256,
            None, None]
    assert lib.k3mla_decode_layer(*args) == -1
    assert b"null or misaligned" in lib.k3mla_last_error()
    args[18] = 0
    assert lib.k3mla_decode_layer(*args) == 0                   # B == 0: nothing to do
    args[18], args[10] = 1, 511                                 # c_stride below a latent row
    assert lib.k3mla_decode_layer(*args) == -1


def test_expanded_baseline_sizes_and_arguments():
    # the expanded cache: [n_pages][64 tokens][96 heads][128 K nope | 64 K rope | 128 V] bf16
    assert k3mla.expanded_cache_bytes(0) == 0
    assert k3mla.expanded_cache_bytes(3) == 3 * 64 * 96 * 320 * 2
    lib = k3mla.load()
    assert lib.k3mla_expand_latent_cache(None, 4, 2, 2, None, None, None, None) == -1   # layer past the slab
    assert b"invalid sizes" in lib.k3mla_last_error()
    assert lib.k3mla_expand_latent_cache(None, 4, 2, 1, None, None, None, None) == -1
    assert b"null or misaligned" in lib.k3mla_last_error()
    args = [None, None, 4, None, 2, None, 0x3D94, None, 0, 128, None, None]
    assert lib.k3mla_expanded_decode(*args) == 0                # B == 0: nothing to do
    args[8] = 1
    assert lib.k3mla_expanded_decode(*args) == -1
    assert b"null or misaligned" in lib.k3mla_last_error()
    args[2] = 0                                                 # no pages
    assert lib.k3mla_expanded_decode(*args) == -1
    assert b"invalid sizes" in lib.k3mla_last_error()


def test_chunk_decode_sizes_and_arguments():
    # o_lat [96][R][512] bf16 and the rows' records (the decode workspace of one split), then the groups
    # of rows (int4, at most (R + 3 B) / 4 + 1 of them) and the rows' contexts (int32), 256-aligned
    r256 = lambda x: (x + 255) // 256 * 256
    for B, R, max_ctx in ((1, 1, 64), (16, 1024, 4160), (3, 7, 300)):
        g = (R + 3 * B) // 4 + 1
        got = k3mla.chunk_decode_workspace_bytes(B, R, max_ctx)
        one_split = r256(R * 96 * 512 * 2) + r256(R * 96 * 4 * 4)
        assert got == one_split + r256(g * 16) + r256(R * 4), (B, R, got)
    assert k3mla.chunk_decode_workspace_bytes(0, 4, 64) == 0
    assert k3mla.chunk_decode_workspace_bytes(2, 0, 64) == 0
    lib = k3mla.load()
    # (q_abs, slab, n_pages, n_layers, layer, table, max_pages, pos0, row_start, B, R, w_kv_b, scale, out,
    #  argmax, workspace, ws_bytes, max_ctx, dev_err, stream)
    args = [None, None, 4, 1, 0, None, 4, None, None, 2, 0, None, 0x3D94, None, None, None, 0, 256, None, None]
    assert lib.k3mla_chunk_decode(*args) == 0                   # R == 0: nothing to do
    args[10] = 5
    assert lib.k3mla_chunk_decode(*args) == -1
    assert b"null or misaligned" in lib.k3mla_last_error()
    args[9] = 0                                                 # no slots
    assert lib.k3mla_chunk_decode(*args) == -1
    assert b"invalid sizes" in lib.k3mla_last_error()
    args[9], args[4] = 2, 1                                     # layer past the slab
    assert lib.k3mla_chunk_decode(*args) == -1
    assert b"invalid sizes" in lib.k3mla_last_error()


def test_exact_exp_diagnostic_arguments():
    lib = k3mla.load()
    assert lib.k3mla_diag_exact_exp(None, None, None, 0, None) == 0     # nothing to do
    assert lib.k3mla_diag_exact_exp(None, None, None, -1, None) == -1
    assert lib.k3mla_diag_exact_exp(None, None, None, 5, None) == -1
    assert b"invalid arguments" in lib.k3mla_last_error()


def test_product_and_oracle_share_no_code():
    """The CUDA path and the oracle are independent: no product source imports, includes or names
    the oracle's modules, and no oracle source imports the product package or includes its
    headers; only the seeded input generator (synth.py, no method arithmetic) serves both."""
    import re
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    pkg = os.path.join(root, "paged_latent_attention_k3mla_gb300")
    product = [os.path.join(pkg, f) for f in os.listdir(pkg) if f.endswith(".py") and f != "synth.py"]
    product += [os.path.join(pkg, "csrc", f) for f in os.listdir(os.path.join(pkg, "csrc"))]
    product += [os.path.join(root, "include", f) for f in os.listdir(os.path.join(root, "include"))]
    for f in product:
        src = open(f).read()
        assert not re.search(r"^\s*(import|from)\s+oracle\b", src, re.M), f
        assert "k3mla_oracle" not in src and "k3o_" not in src, f
    for f in os.listdir(os.path.join(root, "oracle")):
        if not f.endswith((".py", ".c", ".h")):
            continue
        src = open(os.path.join(root, "oracle", f)).read()
        assert "paged_latent_attention_k3mla_gb300" not in src, f
        assert "k3mla.h" not in src and "csrc" not in src, f


def _pairs():
    import torch
    if torch.cuda.is_available():
        return torch.cuda.get_device_properties(0).multi_processor_count // 2
    return 148 // 2  # the library's figure when no device answers


def _live(ctx, split):
    return sum(-(-max(int(c), 0) // split) for c in ctx)


def test_batch_planned_split_on_ragged_batches():
    pairs, tile = _pairs(), 128
    rng = np.random.default_rng(5)
    for B, max_ctx in [(16, 4096), (5, 32768), (40, 8192), (2, 640)]:
        ctx = rng.integers(1, max_ctx + 1, size=B)
        s = k3mla.batch_planned_split_tokens(ctx, max_ctx)
        whole = -(-max_ctx // tile) * tile
        assert s % tile == 0 and tile <= s <= whole
        if s < whole:  # the shortest length whose live splits fit one wave of SM pairs
            assert _live(ctx, s) <= pairs
            assert s == tile or _live(ctx, s - tile) > pairs
            assert s < int(ctx.max())
        else:  # no shorter length both fits and splits the longest context
            shorter = [t for t in range(tile, min(whole, int(ctx.max())), tile) if _live(ctx, t) <= pairs]
            assert not shorter
    # one short context under a long max_ctx: a single whole-context split, not many empty ones
    assert k3mla.batch_planned_split_tokens([100], 32768) == 32768
    assert k3mla.batch_planned_split_tokens([0, 0, 0], 4096) == 4096
    # more slots with tokens than SM pairs: one split per slot
    assert k3mla.batch_planned_split_tokens([200] * (pairs + 1), 256) == 256
    # clamping: contexts past max_ctx count as max_ctx, negative ones as empty
    assert k3mla.batch_planned_split_tokens([10**6] * 8, 32768) == k3mla.batch_planned_split_tokens([32768] * 8, 32768)
    assert k3mla.batch_planned_split_tokens([-5, 100], 32768) == 32768


def test_batch_planned_split_arguments():
    lib = k3mla.load()
    assert lib.k3mla_batch_planned_split_tokens(None, 0, 4096) == 128
    assert lib.k3mla_batch_planned_split_tokens(None, 3, 0) == 128
    assert lib.k3mla_batch_planned_split_tokens(None, 3, 4096) == -1
    assert b"ctx_host is NULL" in lib.k3mla_last_error()
