"""The expanded-cache design as an A/B baseline (pegainfer PR #869, "K3: paged latent MLA KV + absorbed
decode", M2 commit): before the absorbed kernel, kv_b expanded every token's latent into per-head K
(128 nope + the 64-wide rope key) and V (128) rows, and decode ran ordinary attention over them.

The build is checked element by element against the oracle's float64 expansion: each K nope and V
value is bf16 of an f32 sum of 512 exact products, so it lies within half a bf16 ULP of itself plus the
f32 summation bound of the exact value; the rope key is copied bit for bit.  The decode is checked
against the oracle's float64 expanded attention with the same 4 row-max bf16 ULP gate as the absorbed
path, on ragged contexts with holes, an empty slot, and sampled slots of the 64-slot 4096-token
workload."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from paged_latent_attention_k3mla_gb300 import k3mla, synth
from tests.gpu_common import gpu_layer
from tests.helpers import bits_to_f32, row_ulp_error, ULP_TOL

pytestmark = pytest.mark.gpu
H, NOPE, ROPE, V, LORA, PAGE, XR = 96, 128, 64, 128, 512, 64, 320


def _scale(wl) -> float:
    return float(bits_to_f32(np.array([wl.scale_bits]))[0])


def _build(wl, layer):
    n_pages = wl.slab.shape[0]
    x = torch.full((n_pages, PAGE, H, XR), float("nan"), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    k3mla.expand_latent_cache(wl.slab, layer, wl.w_kv_b[layer], x, dev_err=err)
    torch.cuda.synchronize()
    return x, int(err.item())


def _decode(wl, x, table, ctx, max_ctx, layer=0):
    out = torch.full((wl.B, H, V), float("nan"), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    k3mla.expanded_decode(wl.q[layer], x, table, ctx, wl.scale_bits, out, max_ctx, dev_err=err)
    torch.cuda.synchronize()
    return synth.bf16_bits(out), int(err.item())


def test_build_is_the_float64_expansion_landed_once(gpu_lib):
    wl = synth.make_custom([130, 64, 300], n_layers=2, seed=750, device="cuda")
    x, err = _build(wl, 1)
    assert err == 0
    slab = synth.bf16_bits(wl.slab)
    w = synth.bf16_bits(wl.w_kv_b[1])
    pages = [int(wl.block_table[0, 0]), int(wl.block_table[0, 2]), int(wl.block_table[2, 4]),
             wl.slab.shape[0] - 1]
    ref = oracle.expand_pages_f64(slab, 1, w, pages)                       # [P, 64, 96, 320] float64
    got_bits = synth.bf16_bits(x[pages])
    got = bits_to_f32(got_bits).astype(np.float64)
    # the rope key: the latent row's last 64 values, bit for bit, for every head
    rope = slab[pages, 1][:, :, None, LORA:]
    assert np.array_equal(got_bits[..., NOPE:NOPE + ROPE], np.broadcast_to(rope, got_bits[..., NOPE:NOPE + ROPE].shape))
    # K nope and V: |bf16(f) - exact| <= ulp(.)/2 + eps, eps = 2 * 511 * 2^-24 * sum |w||c|
    wf = (w.astype(np.uint32) << 16).view(np.float32).astype(np.float64).reshape(H, NOPE + V, LORA)
    for part, (lo, hi), rows in ((0, (0, NOPE), slice(0, NOPE)), (1, (NOPE + ROPE, XR), slice(NOPE, NOPE + V))):
        c_abs = np.abs(bits_to_f32(slab[pages, 1][:, :, :LORA]).astype(np.float64))   # [P, 64, 512]
        w_abs = np.abs(wf[:, rows, :]).reshape(H * 128, LORA)
        abs_sum = (c_abs.reshape(-1, LORA) @ w_abs.T).reshape(len(pages), PAGE, H, 128)
        exact, g = ref[..., lo:hi], got[..., lo:hi]
        eps = 2.0 * (LORA - 1) * 2.0**-24 * abs_sum
        half_ulp = 0.5 * np.exp2(np.floor(np.log2(np.maximum(np.abs(exact) + eps, 1e-300))) - 7)
        bad = np.abs(g - exact) > half_ulp + eps
        assert not bad.any(), f"part {part}: {int(bad.sum())} values outside the f32-sum bound"
        landed = synth.bf16_bits(torch.from_numpy(exact).to(torch.bfloat16))
        assert (got_bits[..., lo:hi] == landed).mean() > 0.95        # mostly the correctly rounded value


@pytest.mark.parametrize("case", ["ragged", "holes_and_flags"])
def test_decode_matches_the_float64_expanded_attention(gpu_lib, case):
    ctx_lens = [1, 2, 63, 64, 65, 300, 1000, 0, 700]
    wl = synth.make_custom(ctx_lens, seed=751, device="cuda")
    max_ctx = wl.block_table.shape[1] * PAGE
    x, err = _build(wl, 0)
    assert err == 0
    tbl, ctx = wl.block_table.copy(), wl.ctx_len.copy()
    expect = 0
    if case == "holes_and_flags":
        tbl[5, 2] = -1                       # an unmapped page inside a context: zero K and V rows
        tbl[6, 0] = -1
        tbl[8, 3] = wl.slab.shape[0] + 5     # an id past the pool: read as a zero row and flagged
        ctx[3] = max_ctx + 40                # a context past the table: clamped and flagged
        expect = k3mla.DEV_BAD_PAGE | k3mla.DEV_CTX
    out, err = _decode(wl, x, torch.from_numpy(tbl).cuda(), torch.from_numpy(ctx).cuda(), max_ctx)
    assert err == expect, (err, expect)
    tbl_ref = np.where((tbl >= 0) & (tbl < wl.slab.shape[0]), tbl, -1).astype(np.int32)
    ctx_ref = np.minimum(ctx, max_ctx).astype(np.int32)
    ref, _ = oracle.decode_expanded_f64(synth.bf16_bits(wl.q[0]), synth.bf16_bits(wl.slab), 0, tbl_ref, ctx_ref,
                                        synth.bf16_bits(wl.w_kv_b[0]), _scale(wl))
    e = row_ulp_error(bits_to_f32(out), ref)
    print(f"expanded decode vs float64 expanded attention ({case}): max {e.max():.3f} row ULP")
    assert np.all(np.isfinite(bits_to_f32(out)))
    assert e.max() <= ULP_TOL, f"max {e.max():.3f} row ULP"
    assert np.all(out[7] == 0)               # the empty context gives zeros
    if case == "ragged":
        # the absorbed decode on the same inputs sits within the same gate of the same reference
        a = gpu_layer(wl, 0, max_ctx=max_ctx)
        ea = row_ulp_error(bits_to_f32(a["out"]), ref)
        d = row_ulp_error(bits_to_f32(out), bits_to_f32(a["out"]).astype(np.float64))
        print(f"absorbed vs float64: max {ea.max():.3f}; expanded vs absorbed: max {d.max():.3f} row ULP")
        assert ea.max() <= ULP_TOL


def test_full_size_sampled_slots(gpu_lib):
    # the 64-slot, 4096-token workload at one layer (a 16 GB expanded cache), two slots checked
    wl = synth.make_workload("steady64", device="cuda", n_layers=1)
    x, err = _build(wl, 0)
    assert err == 0
    table, ctx = torch.from_numpy(wl.block_table).cuda(), torch.from_numpy(wl.ctx_len).cuda()
    out, err = _decode(wl, x, table, ctx, 4096)
    del x
    torch.cuda.empty_cache()
    assert err == 0
    slots = [0, 37]
    ref, _ = oracle.decode_expanded_f64(synth.bf16_bits(wl.q[0]), synth.bf16_bits(wl.slab), 0, wl.block_table,
                                        wl.ctx_len, synth.bf16_bits(wl.w_kv_b[0]), _scale(wl), slots=slots)
    e = row_ulp_error(bits_to_f32(out[slots]), ref[slots])
    print(f"full size, slots {slots}: max {e.max():.3f} row ULP")
    assert e.max() <= ULP_TOL


def test_argument_checks(gpu_lib):
    wl = synth.make_custom([10], seed=752, device="cuda")
    x = torch.zeros(wl.slab.shape[0] - 1, PAGE, H, XR, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(k3mla.K3mlaError):
        k3mla.expand_latent_cache(wl.slab, 0, wl.w_kv_b[0], x)            # cache of the wrong page count
    with pytest.raises(k3mla.K3mlaError):
        k3mla.expand_latent_cache(wl.slab, 1, wl.w_kv_b[0],
                                  torch.zeros(wl.slab.shape[0], PAGE, H, XR, dtype=torch.bfloat16, device="cuda"))
