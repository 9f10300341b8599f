"""q absorption and the latent append on the GPU against the oracle.

Absorption: within 4 bf16 ULP of each output row's max (f32 accumulation on the
tensor cores adds the 128 products in its own order), the rope half bitwise.
Append: bitwise -- it is a copy into the row the size_t index names."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from paged_latent_attention_k3mla_gb300 import k3mla, synth
from tests.helpers import bits_to_f32, row_ulp_error, ULP_TOL

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B", [1, 16, 37, 64, 65, 128, 200])
def test_absorb_matches_oracle(gpu_lib, B):
    # up to 64 slots one CTA per head covers 64 slots; above, 128 (65 and 128: one ragged and one
    # full tile; 200: a full and a ragged tile)
    g = torch.Generator(device="cuda").manual_seed(100 + B)
    q = torch.randn(B, 96, 192, generator=g, device="cuda").to(torch.bfloat16)
    w = (torch.randn(24576, 512, generator=g, device="cuda") * (1 / 512) ** 0.5).to(torch.bfloat16)
    q_abs = torch.full((B, 96, 576), float("nan"), dtype=torch.bfloat16, device="cuda")
    k3mla.absorb_q(q, w, q_abs)
    torch.cuda.synchronize()
    got = synth.bf16_bits(q_abs)
    ref = oracle.absorb(synth.bf16_bits(q), synth.bf16_bits(w))
    err = row_ulp_error(bits_to_f32(got[:, :, :512]), bits_to_f32(ref[:, :, :512]))
    assert err.max() <= ULP_TOL
    assert (got[:, :, :512] == ref[:, :, :512]).mean() > 0.9
    assert np.array_equal(got[:, :, 512:], ref[:, :, 512:])


def test_append_matches_oracle(gpu_lib):
    wl = synth.make_custom([64, 65, 1, 130, 7], n_layers=3, seed=200, device="cuda")
    tbl = wl.block_table.copy()
    pos = (wl.ctx_len - 1).astype(np.int32)
    pos[2] = -1                     # no write for this slot
    tbl[4, 0] = -1                  # unmapped position: skipped, flagged
    slab_ref = synth.bf16_bits(wl.slab).copy()
    c, r = wl.new_c[1], wl.new_rope[1]
    skipped = oracle.append(slab_ref, 1, tbl, pos, synth.bf16_bits(c), synth.bf16_bits(r))
    assert skipped == 1
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    k3mla.append_latent(wl.slab, 1, torch.from_numpy(tbl).cuda(), torch.from_numpy(pos).cuda(), c, r,
                        dev_err=err)
    torch.cuda.synchronize()
    assert np.array_equal(synth.bf16_bits(wl.slab), slab_ref)
    assert err.item() == k3mla.DEV_UNMAPPED


def test_append_indexes_past_2_31_elements(gpu_lib):
    # 1024 pages x 64 layers x 64 x 576 = 2.4e9 elements (4.8 GB): rows at the top
    n_pages, L = 1024, 64
    slab = torch.zeros(n_pages, L, 64, 576, dtype=torch.bfloat16, device="cuda")
    assert slab.numel() > 2**31
    tbl = torch.tensor([[n_pages - 1], [n_pages - 2]], dtype=torch.int32, device="cuda")
    pos = torch.tensor([63, 5], dtype=torch.int32, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(3)
    c = torch.randn(2, 512, generator=g, device="cuda").to(torch.bfloat16)
    r = torch.randn(2, 64, generator=g, device="cuda").to(torch.bfloat16)
    k3mla.append_latent(slab, L - 1, tbl, pos, c, r)
    torch.cuda.synchronize()
    assert torch.equal(slab[n_pages - 1, L - 1, 63, :512], c[0])
    assert torch.equal(slab[n_pages - 1, L - 1, 63, 512:], r[0])
    assert torch.equal(slab[n_pages - 2, L - 1, 5, :512], c[1])
    assert int(torch.count_nonzero(slab)) == int(torch.count_nonzero(c) + torch.count_nonzero(r))
    del slab
    torch.cuda.empty_cache()


@pytest.mark.parametrize("B", [6, 67, 120, 150])
def test_absorb_q_append_is_both_calls_in_one(gpu_lib, B):
    """The fused launch: q_abs bitwise equal to k3mla_absorb_q's (same kernel) and within the
    absorption bar of the oracle; the slab bitwise equal to the oracle's append, with a slot that
    writes nothing (pos -1) and one whose page is unmapped (skipped and flagged).  At 120 slots the
    grid has 96 CTAs (one per head), so some CTAs append two rows."""
    ctx = [(7 * i * i + 3 * i) % 300 + 1 for i in range(B)]
    wl = synth.make_custom(ctx, n_layers=2, seed=300 + B, device="cuda")
    tbl = wl.block_table.copy()
    pos = (wl.ctx_len - 1).astype(np.int32)
    pos[1] = -1
    tbl[2, pos[2] // 64] = -1
    slab_ref = synth.bf16_bits(wl.slab).copy()
    c, r = wl.new_c[1], wl.new_rope[1]
    assert oracle.append(slab_ref, 1, tbl, pos, synth.bf16_bits(c), synth.bf16_bits(r)) == 1
    q, w = wl.q[1], wl.w_kv_b[1]
    q_abs = torch.full((B, 96, 576), float("nan"), dtype=torch.bfloat16, device="cuda")
    q_abs_sep = torch.full_like(q_abs, float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    k3mla.absorb_q_append(q, w, q_abs, wl.slab, 1, torch.from_numpy(tbl).cuda(), torch.from_numpy(pos).cuda(),
                          c, r, dev_err=err)
    k3mla.absorb_q(q, w, q_abs_sep)
    torch.cuda.synchronize()
    assert np.array_equal(synth.bf16_bits(wl.slab), slab_ref)
    assert err.item() == k3mla.DEV_UNMAPPED
    got = synth.bf16_bits(q_abs)
    assert np.array_equal(got, synth.bf16_bits(q_abs_sep))
    ref = oracle.absorb(synth.bf16_bits(q), synth.bf16_bits(w))
    err_ulp = row_ulp_error(bits_to_f32(got[:, :, :512]), bits_to_f32(ref[:, :, :512]))
    assert err_ulp.max() <= ULP_TOL
    assert np.array_equal(got[:, :, 512:], ref[:, :, 512:])
