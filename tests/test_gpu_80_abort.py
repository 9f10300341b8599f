"""The abort path of the bounded device waits, exercised without any GPU fault: a diagnostic entry
runs the paged decode with one page of every split never loaded and a short wait limit, so that the
waits on that page run out.  The call must return with K3MLA_DEV_TIMEOUT in the device error word
(no trap, no hang), and the context must stay usable: a normal decode right after it on the same
stream matches the oracle."""
from __future__ import annotations

import time

import numpy as np
import pytest
import torch

from paged_latent_attention_k3mla_gb300 import k3mla, synth
from tests.gpu_common import compare, gpu_layer, oracle_layer

pytestmark = pytest.mark.gpu
H, V, ROW = 96, 128, 576


@pytest.mark.parametrize("ctx,split,max_ctx", [([130], 0, 256), ([300, 130, 0, 64], 128, 512)])
def test_a_withheld_page_times_out_and_the_context_stays_usable(gpu_lib, ctx, split, max_ctx):
    wl = synth.make_custom(ctx, seed=800, device="cuda")
    B = wl.B
    table = torch.from_numpy(wl.block_table).cuda()
    ctx_d = torch.from_numpy(wl.ctx_len).cuda()
    q_abs = torch.empty(B, H, ROW, dtype=torch.bfloat16, device="cuda")
    k3mla.absorb_q(wl.q[0], wl.w_kv_b[0], q_abs)
    out = torch.empty(B, H, V, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(k3mla.decode_workspace_bytes(B, max_ctx, split), dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    k3mla.diag_decode_timeout(q_abs, wl.slab, 0, table, ctx_d, wl.w_kv_b[0], wl.scale_bits, out, ws, max_ctx, split,
                              withhold_page=1, wait_us=2000, dev_err=err)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert err.item() & k3mla.DEV_TIMEOUT, f"device error word {err.item()}"
    assert elapsed < 0.5, f"the aborted call took {elapsed:.3f} s"
    # the same decode without the withheld page, right after, on the same stream and workspace
    g = gpu_layer(wl, 0, split=split, max_ctx=max_ctx)
    assert g["dev_err"] == 0
    ok, stats = compare(g, oracle_layer(wl, 0, probs_stride=max(1, int(wl.ctx_len.max()))), wl.ctx_len,
                        name="after_abort")
    assert ok, stats


def test_diagnostic_arguments_are_checked(gpu_lib):
    wl = synth.make_workload("tiny", device="cuda")
    q_abs = torch.empty(1, H, ROW, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(1, H, V, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(k3mla.decode_workspace_bytes(1, 256), dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    table = torch.from_numpy(wl.block_table).cuda()
    ctx_d = torch.from_numpy(wl.ctx_len).cuda()
    for page, us in ((0, 2000), (1, 50), (1, 200000)):
        with pytest.raises(k3mla.K3mlaError, match="withhold_page"):
            k3mla.diag_decode_timeout(q_abs, wl.slab, 0, table, ctx_d, wl.w_kv_b[0], wl.scale_bits, out, ws, 256, 0,
                                      withhold_page=page, wait_us=us, dev_err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
