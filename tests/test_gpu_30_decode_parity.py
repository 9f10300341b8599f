"""Paged absorbed decode on the GPU against the oracle, element by element.

Bar: every output element within 4 bf16 ULP of its (slot, head) row's largest
oracle magnitude, and the argmax of the attention probabilities identical up to
the <= 1-ULP coin flips (a differing token must have an oracle score within one
bf16 ULP of the oracle maximum, or a tied oracle probability).

Cases span several 128-token tiles, ragged tails, multi-split merges, -1 holes,
padding slots and empty contexts at sizes the oracle finishes in seconds; the
full-size workloads are checked on sampled slots in the launch configuration the
benchmark times."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from paged_latent_attention_k3mla_gb300 import k3mla, synth
from tests.gpu_common import compare, gpu_layer, oracle_layer

pytestmark = pytest.mark.gpu


def _parity(wl, layer, slots=None, split=None, max_ctx=None, name="case"):
    g = gpu_layer(wl, layer, split=split, max_ctx=max_ctx)
    o = oracle_layer(wl, layer, slots=slots, probs_stride=int(max(1, wl.ctx_len.max())))
    ok, stats = compare(g, o, wl.ctx_len, name=name)
    print(f"{name}: split={g['split']} {stats}")
    assert g["dev_err"] == 0, g["dev_err"]
    assert ok, stats
    return stats


def test_tiny(gpu_lib):
    wl = synth.make_workload("tiny", device="cuda")
    _parity(wl, 0, name="tiny")


@pytest.mark.parametrize("split", [k3mla.SPLIT_AUTO, 128, 256, 1024])
def test_ragged_tails_and_split_merges(gpu_lib, split):
    ctx = [1, 2, 63, 64, 65, 127, 128, 129, 255, 300, 640, 1000]
    wl = synth.make_custom(ctx, seed=300, device="cuda")
    _parity(wl, 0, split=split, max_ctx=1024, name=f"ragged_split{split}")


def test_default_split_with_single_and_multi_split_slots(gpu_lib):
    # the default rule (at most 4096 tokens a split) on contexts around its boundaries: slots with one
    # split land o_lat in the split kernel, slots with two to five are merged, in one launch
    ctx = [4096, 4097, 100, 8192, 8193, 0, 12000, 1, 20000, 3000]
    wl = synth.make_custom(ctx, seed=305, device="cuda")
    ns = [-(-n // k3mla.slot_split_tokens(n)) for n in ctx]
    assert set(ns) == {0, 1, 2, 3, 5}
    _parity(wl, 0, split=k3mla.SPLIT_AUTO, max_ctx=20000, name="auto_mixed")


def test_prefetched_pages_with_holes_and_bad_ids(gpu_lib):
    # the PV CTA prefetches into L2 the page eight past the latest page whose P has arrived: contexts
    # around that distance (one split a slot of 8, 9, 10 and 64 pages), with -1 holes and a bad page id
    # where the prefetches start and on a last page.  A prefetch never changes a result, and the bad id
    # is flagged with the bit its load raises anyway
    ctx = [8 * 64, 8 * 64 + 1, 9 * 64, 10 * 64 - 3, 4096, 4096]
    wl = synth.make_custom(ctx, seed=310, device="cuda", max_pages=64)
    wl.block_table[1, 8] = -1                       # the one page past a 9-page context's first eight
    wl.block_table[3, 9] = -1
    wl.block_table[4, 8] = wl.slab.shape[0] + 5     # out of range: read as zero and flagged
    wl.block_table[5, 63] = -1                      # the last page of a full-length slot
    g = gpu_layer(wl, 0, split=k3mla.SPLIT_AUTO, max_ctx=4096)
    assert g["dev_err"] == k3mla.DEV_BAD_PAGE, g["dev_err"]
    o = oracle_layer(wl, 0, probs_stride=4096)
    ok, stats = compare(g, o, wl.ctx_len, name="prefetch_edges")
    print("prefetch edges:", stats)
    assert ok, stats


def test_single_split_batch_over_one_slot_tile(gpu_lib):
    # one split per slot (split = max_ctx): the split kernel lands o_lat itself and the expansion
    # reads it in place; 67 slots cover two 64-slot tiles, two contexts are empty
    ctx = [(37 * i * i + 11 * i) % 512 + 1 for i in range(67)]
    ctx[5] = 0
    ctx[66] = 0
    wl = synth.make_custom(ctx, seed=302, device="cuda")
    _parity(wl, 0, split=512, max_ctx=512, name="single_split67")


RESCALE_TAU = 16.0  # the split kernel moves a head's reference max only past this growth (natural log)


def _max_jump(scores, ctx, split):
    """Largest growth of a page max over the running max of the earlier pages of its split."""
    best = -np.inf
    for i, n in enumerate(ctx):
        for s0 in range(0, int(n), split):
            for h in range(scores.shape[1]):
                run = -np.inf
                for p0 in range(s0, min(int(n), s0 + split), 64):
                    pm = scores[i, h, p0:min(int(n), p0 + 64, s0 + split)].max()
                    if run > -np.inf:
                        best = max(best, pm - run)
                    run = max(run, pm)
    return best


def test_heavy_tailed_rows_force_rescales(gpu_lib):
    # late tokens with much larger scores than the early ones move the reference max of their
    # split by more than the rescale threshold, so the PV CTA rescales O (shown on the oracle's
    # own scores below, not assumed)
    wl = synth.make_custom([700, 1500], seed=301, device="cuda", row_scale=(0.25, 4.0))
    wl.slab[wl.block_table[0, 9], 0, 5, :] *= 100
    wl.slab[wl.block_table[1, 20], 0, 17, :] *= 150
    o = oracle_layer(wl, 0, probs_stride=int(wl.ctx_len.max()))
    assert _max_jump(o["scores"], wl.ctx_len, 1024) > RESCALE_TAU
    g = gpu_layer(wl, 0, split=1024, max_ctx=1536)
    ok, stats = compare(g, o, wl.ctx_len, name="rescale")
    print(f"rescale: {stats}")
    assert g["dev_err"] == 0 and ok, stats


def test_many_slots_over_several_waves_and_tiles(gpu_lib):
    # 150 slots: 150 clusters (two waves of SM pairs), two 128-slot absorption tiles, and one or two
    # splits per slot (max_ctx 640, split 384) merged in 16-slot tiles
    ctx = [(53 * i * i + 17 * i) % 640 + 1 for i in range(150)]
    wl = synth.make_custom(ctx, seed=303, device="cuda")
    _parity(wl, 0, split=384, max_ctx=640, name="many_slots150")


def test_one_long_slot_many_splits(gpu_lib):
    # one slot of 20,000 tokens at a 384-token split: 53 splits, merged by four split groups of 13-14
    # splits each; the oracle checks the whole context
    wl = synth.make_custom([20000], seed=304, device="cuda")
    _parity(wl, 0, split=384, max_ctx=20000, name="long_one_slot")


def test_padding_bucket(gpu_lib):
    wl = synth.make_workload("padding128", device="cuda")
    assert (wl.ctx_len == 0).sum() == 1 and (wl.block_table < 0).all(axis=1).sum() > 30
    _parity(wl, 0, name="padding128")


def test_ragged16_two_layers(gpu_lib):
    wl = synth.make_workload("ragged16", device="cuda", n_layers=24)
    for layer in (0, 23):
        _parity(wl, layer, name=f"ragged16_l{layer}")
    # and at the opt-in split planned for the whole batch (several splits per slot)
    planned = k3mla.batch_planned_split_tokens(wl.ctx_len, 4096)
    assert planned < 4096
    _parity(wl, 11, split=planned, max_ctx=4096, name="ragged16_planned")
    del wl
    torch.cuda.empty_cache()


def test_steady64_sampled_full_size(gpu_lib):
    wl = synth.make_workload("steady64", device="cuda")
    _parity(wl, 7, slots=[0, 31, 63], split=k3mla.SPLIT_AUTO, max_ctx=4096, name="steady64")
    del wl
    torch.cuda.empty_cache()


def test_long8_sampled_full_size(gpu_lib):
    wl = synth.make_workload("long8", device="cuda")
    _parity(wl, 11, slots=[3], split=k3mla.SPLIT_AUTO, max_ctx=32768, name="long8")
    del wl
    torch.cuda.empty_cache()


def test_a_flipped_latent_bit_fails_parity(gpu_lib):
    """Negative control: the comparison must catch a one-bit change in one row."""
    wl = synth.make_workload("tiny", device="cuda")
    o = oracle_layer(wl, 0, probs_stride=130)
    g0 = gpu_layer(wl, 0)
    assert compare(g0, o, wl.ctx_len, name="negctl_clean")[0]
    row = wl.slab[wl.block_table[0, 1], 0, 10]
    bits = row.view(torch.int16)
    bits[3] ^= 0x4000                         # exponent bit of one latent value
    g1 = gpu_layer(wl, 0)
    assert not compare(g1, o, wl.ctx_len, name="negctl_flipped")[0]
