"""Decode through k3mla_paged_decode_noalloc, the entry point that takes no
workspace, against k3mla_paged_decode with a workspace the caller allocated.

Some callers cannot allocate device memory where they decode: a server that
reserves all device memory for its own pool at start-up and allows no allocation
while it serves, or a plugin that its host framework hands only the pointers of
its inputs and outputs.  For them the library carries a fixed 16 MiB scratch
array.  Both entry points run the same kernels with the same split, so the
outputs and the argmax must be the same bits.  Two calls in a row on different
inputs -- one whose slots have several splits (f32 partials and the merge), one
whose slots land o_lat directly and that includes an empty context -- show that
what one call leaves in the shared scratch does not reach the next, also when
the second call follows the first on the stream with nothing in between.

The file name sorts last, so a run that stops at the first failure has already
run every other test."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from paged_latent_attention_k3mla_gb300 import k3mla, synth
from tests.gpu_common import gpu_layer

pytestmark = pytest.mark.gpu

H, V, ROW = 96, 128, 576


class _Call:
    """One decode's inputs and NaN-cleared outputs for the built-in-scratch entry point."""

    def __init__(self, ctx_lens, seed, split, max_ctx):
        self.wl = synth.make_custom(ctx_lens, seed=seed, device="cuda")
        self.split, self.max_ctx = split, max_ctx
        B = self.wl.B
        assert k3mla.decode_workspace_bytes(B, max_ctx, split) <= k3mla.NOALLOC_SCRATCH_BYTES
        self.table = torch.from_numpy(self.wl.block_table).cuda()
        self.ctx = torch.from_numpy(self.wl.ctx_len).cuda()
        self.q_abs = torch.empty(B, H, ROW, dtype=torch.bfloat16, device="cuda")
        k3mla.absorb_q(self.wl.q[0], self.wl.w_kv_b[0], self.q_abs)
        self.out = torch.full((B, H, V), float("nan"), dtype=torch.bfloat16, device="cuda")
        self.am = torch.full((B, H), -7, dtype=torch.int32, device="cuda")
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")

    def decode_noalloc(self):
        wl = self.wl
        k3mla.paged_decode_noalloc(self.q_abs, wl.slab, 0, self.table, self.ctx, wl.w_kv_b[0], wl.scale_bits,
                                   self.out, self.max_ctx, self.split, argmax=self.am, dev_err=self.err)

    def check_against_the_workspace_entry_point(self):
        torch.cuda.synchronize()
        ref = gpu_layer(self.wl, 0, split=self.split, max_ctx=self.max_ctx)
        assert ref["dev_err"] == 0 and int(self.err.item()) == 0, (ref["dev_err"], int(self.err.item()))
        got_out, got_am = synth.bf16_bits(self.out), self.am.cpu().numpy()
        assert np.array_equal(got_out, ref["out"]), "outputs differ from k3mla_paged_decode"
        assert np.array_equal(got_am, ref["argmax"]), "argmax differs from k3mla_paged_decode"
        return got_out, got_am


def _multi_split_call():
    # 7 slots x up to 8 splits of 256 tokens: f32 partials, merged by the expansion kernel
    return _Call([1, 63, 64, 65, 300, 1000, 2048], seed=910, split=256, max_ctx=2048)


def _single_split_call():
    # the default rule: every slot one split (o_lat landed by the split kernel), slot 2 empty
    return _Call([5, 129, 0, 700, 4096], seed=911, split=k3mla.SPLIT_AUTO, max_ctx=4096)


def test_two_calls_in_a_row_match_the_workspace_entry_point(gpu_lib):
    first = _multi_split_call()
    first.decode_noalloc()
    first.check_against_the_workspace_entry_point()
    second = _single_split_call()
    second.decode_noalloc()
    out, am = second.check_against_the_workspace_entry_point()
    assert np.all(out[2] == 0) and np.all(am[2] == -1)


def test_back_to_back_calls_share_the_scratch_safely(gpu_lib):
    # the two decodes follow each other on one stream with no other kernel between them, the second
    # with one split per slot and an empty context (whose o_lat it zeroes in the shared scratch)
    first, second = _multi_split_call(), _single_split_call()
    torch.cuda.synchronize()
    first.decode_noalloc()
    second.decode_noalloc()
    first.check_against_the_workspace_entry_point()
    second.check_against_the_workspace_entry_point()


def test_requests_beyond_the_scratch_are_rejected_before_launch(gpu_lib):
    B, max_ctx, split = 169, 128, 128  # one split a slot: 168 slots fit in 16 MiB, 169 do not
    assert k3mla.decode_workspace_bytes(B - 1, max_ctx, split) <= k3mla.NOALLOC_SCRATCH_BYTES
    assert k3mla.decode_workspace_bytes(B, max_ctx, split) > k3mla.NOALLOC_SCRATCH_BYTES
    q_abs = torch.zeros(B, H, ROW, dtype=torch.bfloat16, device="cuda")
    slab = torch.zeros(2, 1, 64, ROW, dtype=torch.bfloat16, device="cuda")
    table = torch.zeros(B, 2, dtype=torch.int32, device="cuda")
    ctx = torch.full((B,), 100, dtype=torch.int32, device="cuda")
    w = torch.zeros(H * 256, 512, dtype=torch.bfloat16, device="cuda")
    out = torch.full((B, H, V), float("nan"), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(k3mla.K3mlaError, match="built-in scratch"):
        k3mla.paged_decode_noalloc(q_abs, slab, 0, table, ctx, w, 0x3D94, out, max_ctx, split)
    torch.cuda.synchronize()
    assert torch.isnan(out.float()).all()  # nothing ran
