"""Decode through k3mla_paged_decode_noalloc, the entry point that takes no
workspace, against k3mla_paged_decode with a workspace the caller allocated.

Some callers cannot allocate device memory where they decode: a server that
reserves all device memory for its own pool at start-up and allows no allocation
while it serves, or a plugin that its host framework hands only the pointers of
its inputs and outputs.  For them the library carries a fixed 16 MiB scratch
array.  Both entry points run the same kernels, so the outputs are held to the
bar of the other decode tests (4 bf16 ULP of the row's largest magnitude) and
the argmax must be the same token.  Two calls in a row on different inputs show
that what one call leaves in the shared scratch does not reach the next.

The file name sorts last, so a run that stops at the first failure has already
run every other test."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from paged_latent_attention_k3mla_gb300 import k3mla, synth
from tests.gpu_common import gpu_layer
from tests.helpers import ULP_TOL, bits_to_f32, row_ulp_error

pytestmark = pytest.mark.gpu

H, V, ROW = 96, 128, 576


def _noalloc_layer(wl, layer, split, max_ctx):
    B = wl.B
    table = torch.from_numpy(wl.block_table).cuda()
    ctx = torch.from_numpy(wl.ctx_len).cuda()
    q_abs = torch.empty(B, H, ROW, dtype=torch.bfloat16, device="cuda")
    k3mla.absorb_q(wl.q[layer], wl.w_kv_b[layer], q_abs)
    out = torch.full((B, H, V), float("nan"), dtype=torch.bfloat16, device="cuda")
    am = torch.full((B, H), -7, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    k3mla.paged_decode_noalloc(q_abs, wl.slab, layer, table, ctx, wl.w_kv_b[layer], wl.scale_bits, out,
                               max_ctx, split, argmax=am, dev_err=err)
    torch.cuda.synchronize()
    return dict(out=synth.bf16_bits(out), argmax=am.cpu().numpy(), dev_err=int(err.item()))


def _check_same(ctx_lens, seed, split, max_ctx):
    wl = synth.make_custom(ctx_lens, seed=seed, device="cuda")
    nsplit = -(-max_ctx // split)
    assert k3mla.decode_workspace_bytes(wl.B, max_ctx, split) <= k3mla.NOALLOC_SCRATCH_BYTES, (wl.B, nsplit)
    ref = gpu_layer(wl, 0, split=split, max_ctx=max_ctx)
    got = _noalloc_layer(wl, 0, split, max_ctx)
    assert ref["dev_err"] == 0 and got["dev_err"] == 0, (ref["dev_err"], got["dev_err"])
    g, r = bits_to_f32(got["out"]), bits_to_f32(ref["out"])
    assert np.all(np.isfinite(g))
    err = row_ulp_error(g, r)
    assert err.max() <= ULP_TOL, f"max error {err.max():.3f} row-max bf16 ULP"
    assert np.array_equal(got["argmax"], ref["argmax"])


def test_two_calls_in_a_row_match_the_workspace_entry_point(gpu_lib):
    # first call: 7 slots x 8 splits of 256 tokens (56 of the 84 slot-splits the scratch holds)
    _check_same([1, 63, 64, 65, 300, 1000, 2048], seed=910, split=256, max_ctx=2048)
    # second call, other inputs and shapes: 3 slots x 8 splits of 128 tokens
    _check_same([5, 129, 700], seed=911, split=128, max_ctx=1024)


def test_requests_beyond_the_scratch_are_rejected_before_launch(gpu_lib):
    B, max_ctx, split = 85, 128, 128  # 85 slot-splits: one more than 16 MiB holds
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
