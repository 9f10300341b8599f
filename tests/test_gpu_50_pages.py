"""Whole-page copy and page sharing on the GPU.

* k3mla_copy_pages against the oracle's page copy, bitwise (it moves bytes), within
  one slab and from a second (prefill) slab, with a bad pair skipped and flagged,
  and past 2^31 slab elements.
* Prefill adoption and prefix sharing with copy on write, end to end through the
  decode: the outputs are bitwise equal to the decode of the same logical rows laid
  out in private pages (no physical page id enters the arithmetic), and within the
  usual 4-ULP bar of the oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from paged_latent_attention_k3mla_gb300 import k3mla, synth
from tests.gpu_common import compare, gpu_layer, oracle_layer

pytestmark = pytest.mark.gpu

PAGE, ROW = 64, 576


def _ids(x):
    return torch.tensor(x, dtype=torch.int32, device="cuda")


def test_copy_pages_matches_oracle(gpu_lib):
    g = torch.Generator(device="cuda").manual_seed(50)
    slab = torch.randn(12, 3, PAGE, ROW, generator=g, device="cuda").to(torch.bfloat16)
    prefill = torch.randn(5, 3, PAGE, ROW, generator=g, device="cuda").to(torch.bfloat16)
    want = synth.bf16_bits(slab).copy()
    src, dst = [4, 9, 0, 2], [1, 3, 11, 12]                        # the last pair names page 12 of 12
    assert oracle.copy_pages(want, want.copy(), src, dst) == 1
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    k3mla.copy_pages(slab, slab, _ids(src), _ids(dst), dev_err=err)
    torch.cuda.synchronize()
    assert np.array_equal(synth.bf16_bits(slab), want)
    assert err.item() == k3mla.DEV_BAD_PAGE
    # adoption from another pool
    assert oracle.copy_pages(want, synth.bf16_bits(prefill), [3, 0, 4], [5, 6, 7]) == 0
    err.zero_()
    k3mla.copy_pages(slab, prefill, _ids([3, 0, 4]), _ids([5, 6, 7]), dev_err=err)
    torch.cuda.synchronize()
    assert np.array_equal(synth.bf16_bits(slab), want) and err.item() == 0


def test_copy_pages_past_2_31_elements(gpu_lib):
    n_pages, L = 1024, 64                                          # 2.4e9 elements (4.8 GB)
    slab = torch.zeros(n_pages, L, PAGE, ROW, dtype=torch.bfloat16, device="cuda")
    assert slab.numel() > 2**31
    g = torch.Generator(device="cuda").manual_seed(51)
    slab[n_pages - 1] = torch.randn(L, PAGE, ROW, generator=g, device="cuda").to(torch.bfloat16)
    slab[3] = torch.randn(L, PAGE, ROW, generator=g, device="cuda").to(torch.bfloat16)
    k3mla.copy_pages(slab, slab, _ids([n_pages - 1, 3]), _ids([2, n_pages - 2]))
    torch.cuda.synchronize()
    assert torch.equal(slab[2], slab[n_pages - 1]) and torch.equal(slab[n_pages - 2], slab[3])
    assert int(torch.count_nonzero(slab[4:n_pages - 2])) == 0
    del slab
    torch.cuda.empty_cache()


def _decode(wl, table_np, ctx_np, slab=None):
    return gpu_layer(wl, 1, split=256, max_ctx=512, table=torch.from_numpy(table_np).cuda(),
                     ctx=torch.from_numpy(np.asarray(ctx_np, np.int32)).cuda(), slab=slab)


def test_shared_prefix_with_copy_on_write_decodes_like_private_pages(gpu_lib):
    # slot 0 holds 200 tokens; slot 1 shares its first 130 and appends token 130 of its own
    wl = synth.make_custom([200, 131], n_layers=2, seed=52, device="cuda", max_pages=8, n_pages=16)
    pool = k3mla.Pool(n_slots=2, max_ctx=512, n_pages=16, shuffle_seed=9)
    assert pool.ensure(0, 200) == 0 and pool.share_prefix(1, 0, 130) == 0
    assert pool.ensure(1, 131) == 0                                # page 2 is already (shared-)mapped
    shared = pool.table()[0, :4].copy()
    cp = pool.cow(1, 130)                                          # token 130 lands in shared page 2
    assert cp is not None and cp[0] == shared[2]
    page2_before = wl.slab[int(shared[2])].clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    k3mla.copy_pages(wl.slab, wl.slab, _ids([cp[0]]), _ids([cp[1]]), dev_err=err)
    table = pool.table()
    pos = torch.tensor([-1, 130], dtype=torch.int32, device="cuda")
    for layer in range(2):
        k3mla.append_latent(wl.slab, layer, torch.from_numpy(table).cuda(), pos, wl.new_c[layer],
                            wl.new_rope[layer], dev_err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    got = _decode(wl, table, [200, 131])

    # the same logical rows in private pages: slot 1's three pages copied to fresh ids
    ref_slab = wl.slab.clone()
    table_ref = table.copy()
    free = [p for p in range(16) if p not in set(table[table >= 0].tolist())]
    for lp in range(3):
        ref_slab[free[lp]] = wl.slab[int(table[1, lp])]
        table_ref[1, lp] = free[lp]
    ref = _decode(wl, table_ref, [200, 131], slab=ref_slab)
    assert got["dev_err"] == 0 and ref["dev_err"] == 0
    assert np.array_equal(got["out"], ref["out"]) and np.array_equal(got["argmax"], ref["argmax"])
    # slot 0's page 2 is untouched by slot 1's write, which went to the private copy
    assert torch.equal(wl.slab[int(shared[2])], page2_before)
    assert not torch.equal(wl.slab[int(cp[1]), :, 130 % PAGE], page2_before[:, 130 % PAGE])
    # and the pair decodes within the usual bar of the oracle (which reads the shared pages as they are)
    wl.block_table = table
    wl.ctx_len = np.asarray([200, 131], np.int32)
    ok, stats = compare(got, oracle_layer(wl, 1, probs_stride=200), wl.ctx_len, name="shared_prefix")
    assert ok, stats


def test_prefill_adoption_decodes_like_the_prefill_pool(gpu_lib):
    # a prefill pool holds a 300-token sequence; a decode slot adopts it by whole-page copies
    wl = synth.make_custom([300], n_layers=2, seed=53, device="cuda", max_pages=8, n_pages=8)
    pool = k3mla.Pool(n_slots=3, max_ctx=512, n_pages=20, shuffle_seed=4)
    assert pool.ensure(0, 64) == 0 and pool.ensure(2, 1) == 0     # other slots hold pages already
    assert pool.ensure(1, 300) == 0
    dst = pool.table()[1, :5].copy()
    src = wl.block_table[0, :5].copy()
    decode_slab = torch.zeros(20, 2, PAGE, ROW, dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    k3mla.copy_pages(decode_slab, wl.slab, _ids(src.tolist()), _ids(dst.tolist()), dev_err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    ref = _decode(wl, wl.block_table, [300])
    adopted = _decode(wl, pool.table()[1:2], [300], slab=decode_slab)
    assert np.array_equal(adopted["out"], ref["out"]) and np.array_equal(adopted["argmax"], ref["argmax"])
