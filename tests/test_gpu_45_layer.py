"""k3mla_decode_layer, one decode step of one layer (pegainfer PR #869, M1 and M2 commits: the new
token's row into its mapped page, q absorbed, the absorbed attention over the slot's pages), against
the calls it stands for: k3mla_absorb_q_append at position ctx_len - 1 followed by
k3mla_paged_decode under the default split: the same bits (outputs, argmax and the appended rows),
in one call per layer."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from paged_latent_attention_k3mla_gb300 import k3mla, synth
from tests.gpu_common import compare, oracle_layer

pytestmark = pytest.mark.gpu
H, V, ROW = 96, 128, 576


def _ref_calls(wl, layer, table, ctx, max_ctx):
    """absorb_q_append (write position ctx - 1) + paged_decode (default split)."""
    B = wl.B
    pos = (ctx - 1).to(torch.int32)
    q_abs = torch.empty(B, H, ROW, dtype=torch.bfloat16, device="cuda")
    out = torch.full((B, H, V), float("nan"), dtype=torch.bfloat16, device="cuda")
    am = torch.full((B, H), -7, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.full((k3mla.decode_workspace_bytes(B, max_ctx),), 0xFF, dtype=torch.uint8, device="cuda")
    k3mla.absorb_q_append(wl.q[layer], wl.w_kv_b[layer], q_abs, wl.slab, layer, table, pos, wl.new_c[layer],
                          wl.new_rope[layer], dev_err=err)
    k3mla.paged_decode(q_abs, wl.slab, layer, table, ctx, wl.w_kv_b[layer], wl.scale_bits, out, ws, max_ctx,
                       argmax=am, dev_err=err)
    torch.cuda.synchronize()
    return synth.bf16_bits(out), am.cpu().numpy(), int(err.item())


class _Layer:
    """decode_layer with its own NaN-poisoned workspace."""

    def __init__(self, B, max_ctx):
        self.B, self.max_ctx = B, max_ctx
        self.ws = torch.full((k3mla.decode_layer_workspace_bytes(B, max_ctx),), 0xFF, dtype=torch.uint8,
                             device="cuda")
        self.out = torch.full((B, H, V), float("nan"), dtype=torch.bfloat16, device="cuda")
        self.am = torch.full((B, H), -7, dtype=torch.int32, device="cuda")
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")

    def run(self, wl, layer, table, ctx, q=None):
        k3mla.decode_layer(wl.q[layer] if q is None else q, wl.w_kv_b[layer], wl.slab, layer, table, ctx,
                           wl.new_c[layer], wl.new_rope[layer], wl.scale_bits, self.out, self.ws, self.max_ctx,
                           argmax=self.am, dev_err=self.err)

    def result(self):
        torch.cuda.synchronize()
        return synth.bf16_bits(self.out), self.am.cpu().numpy(), int(self.err.item())


def _same_as_the_calls(wl, layers, max_ctx, expect_err=0):
    table = torch.from_numpy(wl.block_table).cuda()
    ctx = torch.from_numpy(wl.ctx_len).cuda()
    lay = _Layer(wl.B, max_ctx)
    for layer in layers:
        before = synth.bf16_bits(wl.slab[:, layer]).copy()
        ref_out, ref_am, ref_err = _ref_calls(wl, layer, table, ctx, max_ctx)
        after_ref = synth.bf16_bits(wl.slab[:, layer]).copy()
        wl.slab[:, layer] = synth.from_bf16_bits(before, "cuda")   # the step's rows are written again
        lay.out.fill_(float("nan"))
        lay.am.fill_(-7)
        lay.run(wl, layer, table, ctx)
        out, am, err = lay.result()
        assert err == ref_err == expect_err, (err, ref_err)
        assert np.array_equal(out, ref_out), f"layer {layer}: outputs differ from the separate calls"
        assert np.array_equal(am, ref_am), f"layer {layer}: argmax differs from the separate calls"
        assert np.array_equal(synth.bf16_bits(wl.slab[:, layer]), after_ref), f"layer {layer}: appended rows differ"
    return lay


def test_one_slot_tiny(gpu_lib):
    wl = synth.make_workload("tiny", device="cuda")
    _same_as_the_calls(wl, [0], 256)


def test_ragged16_layers(gpu_lib):
    wl = synth.make_workload("ragged16", device="cuda", n_layers=3)
    _same_as_the_calls(wl, [0, 2], 4096)


def test_64_slots_with_holes_empty_slots_and_padding(gpu_lib):
    ctx = [(41 * i * i + 7 * i) % 4096 + 1 for i in range(64)]
    ctx[3] = 0
    ctx[40] = 0
    wl = synth.make_custom(ctx, seed=450, device="cuda", max_pages=64)
    wl.block_table[10, 5] = -1
    wl.block_table[11, :] = -1          # a padding row with a context: its append is flagged and skipped
    _same_as_the_calls(wl, [0], 4096, expect_err=k3mla.DEV_UNMAPPED)


def test_steady64_full_size(gpu_lib):
    wl = synth.make_workload("steady64", device="cuda", n_layers=2)
    _same_as_the_calls(wl, [1], 4096)
    del wl
    torch.cuda.empty_cache()


@pytest.mark.parametrize("case", ["many_slots", "long_context"])
def test_many_slots_and_several_splits(gpu_lib, case):
    # more than 64 slots (128-slot absorption tiles), or contexts past one split (f32 partials, merge)
    if case == "many_slots":
        wl = synth.make_workload("padding128", device="cuda")  # its padding rows' appends are flagged
        _same_as_the_calls(wl, [0], 256, expect_err=k3mla.DEV_UNMAPPED)
    else:
        wl = synth.make_custom([9000, 100, 4097], seed=451, device="cuda")
        _same_as_the_calls(wl, [0], 9000)


def test_splits_with_every_page_unmapped(gpu_lib):
    # the layer call gives a split whose pages are all -1 its known result without streaming zero rows;
    # the bits must be those of the full pass: a padding slot of one split, a padding slot of several
    # splits, a slot whose first split is unmapped and whose second is not, and an ordinary slot
    wl = synth.make_custom([300, 9000, 5000, 700], seed=452, device="cuda")
    wl.block_table[0, :] = -1                    # one split, all unmapped (its append is flagged)
    wl.block_table[1, :] = -1                    # three splits, all unmapped
    split = int(k3mla.slot_split_tokens(5000, k3mla.SPLIT_AUTO))
    wl.block_table[2, :split // 64] = -1         # slot 2: its first split unmapped
    _same_as_the_calls(wl, [0], 9000, expect_err=k3mla.DEV_UNMAPPED)


def test_matches_the_oracle(gpu_lib):
    wl = synth.make_workload("ragged16", device="cuda", n_layers=2)
    slab_before = synth.bf16_bits(wl.slab).copy()
    table = torch.from_numpy(wl.block_table).cuda()
    ctx = torch.from_numpy(wl.ctx_len).cuda()
    lay = _Layer(wl.B, 4096)
    lay.run(wl, 1, table, ctx)
    out, am, err = lay.result()
    assert err == 0
    slab = slab_before.copy()
    oracle.append(slab, 1, wl.block_table, wl.pos, synth.bf16_bits(wl.new_c[1]), synth.bf16_bits(wl.new_rope[1]))
    assert np.array_equal(slab, synth.bf16_bits(wl.slab)), "append differs from the oracle"
    o = oracle_layer(wl, 1, probs_stride=int(wl.ctx_len.max()))
    ok, stats = compare({"out": out, "argmax": am}, o, wl.ctx_len, name="decode_layer")
    print("decode_layer vs oracle:", stats)
    assert ok, stats


def test_back_to_back_layers_and_graph_replay(gpu_lib):
    # 24 calls back to back on one stream, then the same calls captured in a CUDA graph and replayed:
    # bitwise the same
    wl = synth.make_workload("ragged16", device="cuda", n_layers=24)
    table = torch.from_numpy(wl.block_table).cuda()
    ctx = torch.from_numpy(wl.ctx_len).cuda()
    lay = _Layer(wl.B, 4096)
    outs = torch.empty(24, wl.B, H, V, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()

    def step():
        for layer in range(24):
            lay.run(wl, layer, table, ctx)
            outs[layer].copy_(lay.out)

    with torch.cuda.stream(s):
        step()
    torch.cuda.synchronize()
    assert lay.err.item() == 0
    eager = outs.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    outs.fill_(float("nan"))
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(outs.view(torch.int16), eager.view(torch.int16))
    assert lay.err.item() == 0
