"""Pins for the CPU oracle: what the pages and the mathematics fix, checked
against the oracle without trusting it.

Sources: pegainfer PR #869, "K3: paged latent MLA KV + absorbed decode" (M1
commit: slab layout, -1 entries, size_t row write; M2 commit: the per-head math,
the rounding chain, the byte figures and the page-permutation / padding
invariants).

Pins, and the mistakes each would catch:
  * bf16 rounding == torch's round-to-nearest-even conversion (a wrong rounding).
  * absorption vs an exact float64 product (transposed / mis-indexed W_UK).
  * whole chain vs the float64 expanded-K/V attention that never absorbs
    (dropped rope term, wrong sign, missing scale, wrong W_UV rows, wrong
    page/layer index, wrong normaliser) -- within 4 bf16 ULP of the row max.
  * closed forms: one token gives p = 1 and out = bf16(W_UV c_0) whatever q is;
    q = 0 with a zero rope key gives p = bf16(1/n); an all -1 table gives 0;
    an empty context gives 0 and argmax -1.
  * invariants: permuting physical pages and relabelling the table is bitwise
    invisible; a -1 entry equals a physical all-zero page bitwise; rows past the
    context are never read; slots are independent.
  * the byte figures the page prints (27.6 KB/token absorbed vs ~1.47 MB/token
    expanded over 24 layers) from the slab geometry.
Planted mistakes (the oracle's ``mutation`` argument) must each fail one pin.
"""
from __future__ import annotations

import os

import numpy as np
import pytest
import torch

import oracle
from oracle.expanded import bf16_bits_to_f64
from paged_latent_attention_k3mla_gb300 import synth
from tests.helpers import argmax_mismatch_ok, bits_to_f32, row_ulp_error, ULP_TOL
from tests.twin import twin_head

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
H, NOPE, ROPE, V, LORA, PAGE, ROW = 96, 128, 64, 128, 512, 64, 576


def np_inputs(wl: synth.Workload, layer=0):
    return dict(q=synth.bf16_bits(wl.q[layer]), w=synth.bf16_bits(wl.w_kv_b[layer]),
                slab=synth.bf16_bits(wl.slab), tbl=wl.block_table, ctx=wl.ctx_len)


def within_f32_sum_bound(got_bits, exact, abs_sum, n_terms):
    """bf16(f) with f a recursive f32 sum of n_terms exact products:
    |f - exact| <= (n_terms - 1) * 2**-24 * sum|terms| (first-order bound, with a
    factor 2 margin) and |bf16(f) - f| <= ulp_bf16(f) / 2."""
    got = bits_to_f32(got_bits).astype(np.float64)
    eps = 2.0 * max(n_terms - 1, 1) * 2.0**-24 * abs_sum
    half_ulp = 0.5 * np.exp2(np.floor(np.log2(np.maximum(np.abs(exact) + eps, 1e-300))) - 7)
    return np.all(np.abs(got - exact) <= half_ulp + eps)


def run_chain(d, layer=0, mutation=0, **kw):
    q_abs = oracle.absorb(d["q"], d["w"], mutation=mutation)
    r = oracle.decode(q_abs, d["slab"], layer, d["tbl"], d["ctx"], d["w"],
                      synth.scale_bf16_bits(), nthreads=4, mutation=mutation, **kw)
    r["q_abs"] = q_abs
    return r


# ---------------------------------------------------------------- rounding

def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(5000) * 1e30).astype(np.float32),
        (rng.standard_normal(5000) * 1e-39).astype(np.float32),   # subnormals
        np.array([0.0, -0.0, np.inf, -np.inf, 3.3895314e38, -3.3895314e38,
                  1.0 + 2**-8, 1.0 + 3 * 2**-8, 1.0 + 2**-8 + 2**-20], np.float32),
    ])
    # exact halfway points (ties) around random bf16 values
    base = (rng.integers(0, 2**16, 4000).astype(np.uint32) << 16) | 0x8000
    x = np.concatenate([x, base.view(np.float32)])
    x = x[np.isfinite(x) | np.isinf(x)]
    ours = oracle.f32_to_bf16(x)
    ref = synth.bf16_bits(torch.from_numpy(x).to(torch.bfloat16))
    nan = np.isnan(x)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_scale_constant_is_bf16_of_inverse_sqrt_192():
    bits = synth.scale_bf16_bits()
    assert bits == 0x3D94
    assert float(bits_to_f32(np.array([bits]))[0]) == 0.072265625


# ---------------------------------------------------------------- absorption

def test_absorb_against_exact_float64():
    wl = synth.make_workload("tiny")
    d = np_inputs(wl)
    q_abs = oracle.absorb(d["q"], d["w"])
    w = bf16_bits_to_f64(d["w"]).reshape(H, NOPE + V, LORA)
    q = bf16_bits_to_f64(d["q"])
    exact = np.einsum("bhd,hdj->bhj", q[:, :, :NOPE], w[:, :NOPE, :])
    abs_sum = np.einsum("bhd,hdj->bhj", np.abs(q[:, :, :NOPE]), np.abs(w[:, :NOPE, :]))
    landed = synth.bf16_bits(torch.from_numpy(exact).to(torch.bfloat16))
    got = q_abs[:, :, :LORA]
    assert within_f32_sum_bound(got, exact, abs_sum, NOPE)
    assert (got == landed).mean() > 0.95          # mostly the correctly rounded value
    assert np.array_equal(q_abs[:, :, LORA:], d["q"][:, :, NOPE:])


# ---------------------------------------------------------------- expanded reference

def _vs_expanded(wl, layer=0, mutation=0):
    d = np_inputs(wl, layer)
    r = run_chain(d, layer, mutation=mutation, probs_stride=int(max(1, wl.ctx_len.max())))
    ref, am = oracle.decode_expanded_f64(d["q"], d["slab"], layer, d["tbl"], d["ctx"], d["w"],
                                         float(bits_to_f32(np.array([synth.scale_bf16_bits()]))[0]))
    err = row_ulp_error(bits_to_f32(r["out"]), ref)
    return r, ref, am, err


@pytest.mark.parametrize("case", ["tiny", "small_ragged", "two_layers"])
def test_chain_matches_expanded_float64(case):
    if case == "tiny":
        wl, layer = synth.make_workload("tiny"), 0
    elif case == "small_ragged":
        wl, layer = synth.make_custom([1, 2, 7, 64, 65, 200], seed=11), 0
    else:
        wl, layer = synth.make_custom([70, 129], n_layers=2, seed=12), 1
    r, ref, am, err = _vs_expanded(wl, layer)
    assert err.max() <= ULP_TOL, f"max {err.max():.3f} ULP"
    # the absorbed chain and the expanded float64 attention pick the same token,
    # up to the <= 1-ULP coin flips
    for b in range(wl.B):
        n = int(wl.ctx_len[b])
        for h in range(H):
            assert argmax_mismatch_ok(r["scores"][b, h], r["probs"][b, h], n,
                                      int(r["argmax"][b, h]), int(am[b, h]))


def test_expanded_pages_select_the_latent_entries_a_permutation_weight_picks():
    # closed form: with W_UK[h][i, j] = [j == (i + h) mod 512] and W_UV[h][i, j] = 2 [j == (511 - i - h) mod 512]
    # the expansion is a gather, so a transposed weight, a head mixed up or K and V swapped all fail
    wl = synth.make_custom([130], seed=21)
    d = np_inputs(wl)
    w = np.zeros((H, NOPE + V, LORA), np.float32)
    for h in range(H):
        for i in range(NOPE):
            w[h, i, (i + h) % LORA] = 1.0
            w[h, NOPE + i, (LORA - 1 - i - h) % LORA] = 2.0
    wbits = synth.bf16_bits(torch.from_numpy(w.reshape(H * (NOPE + V), LORA)).to(torch.bfloat16))
    pages = [int(wl.block_table[0, 1]), int(wl.block_table[0, 0])]
    x = oracle.expand_pages_f64(d["slab"], 0, wbits, pages)
    for k, pid in enumerate(pages):
        rows = bf16_bits_to_f64(d["slab"][pid, 0])
        for h in (0, 1, 57, 95):
            i = np.arange(NOPE)
            assert np.array_equal(x[k, :, h, :NOPE], rows[:, (i + h) % LORA])
            assert np.array_equal(x[k, :, h, NOPE:NOPE + 64], rows[:, LORA:])
            assert np.array_equal(x[k, :, h, NOPE + 64:], 2.0 * rows[:, (LORA - 1 - i - h) % LORA])


def test_expanded_scores_equal_the_absorbed_association():
    # q . [W_UK c ; k_rope] against (W_UK^T q) . c + q_rope . k_rope, both in float64: the absorption identity
    wl = synth.make_custom([64], seed=22)
    d = np_inputs(wl)
    pid = int(wl.block_table[0, 0])
    x = oracle.expand_pages_f64(d["slab"], 0, d["w"], [pid])[0]              # [64, 96, 320]
    q = bf16_bits_to_f64(d["q"])[0]                                           # [96, 192]
    w = bf16_bits_to_f64(d["w"]).reshape(H, NOPE + V, LORA)
    rows = bf16_bits_to_f64(d["slab"][pid, 0])
    s_exp = np.einsum("thd,hd->th", x[:, :, :NOPE + 64], q)
    q_abs = np.einsum("hd,hdj->hj", q[:, :NOPE], w[:, :NOPE, :])
    s_abs = rows[:, :LORA] @ q_abs.T + rows[:, LORA:] @ q[:, NOPE:].T
    scale = np.abs(rows[:, :LORA]) @ np.abs(np.einsum("hd,hdj->hj", np.abs(q[:, :NOPE]), np.abs(w[:, :NOPE, :]))).T
    assert np.all(np.abs(s_exp - s_abs) <= 1e-12 * (scale + 1.0))


# ---------------------------------------------------------------- closed forms

def test_single_token_closed_form_and_q_independence():
    wl = synth.make_custom([1, 1], seed=21)
    d = np_inputs(wl)
    r1 = run_chain(d, want_olat=True, probs_stride=1)
    assert np.all(bits_to_f32(r1["probs"][:, :, 0]) == 1.0)
    d2 = dict(d)
    d2["q"] = synth.bf16_bits(torch.randn(d["q"].shape, generator=torch.Generator().manual_seed(5))
                              .to(torch.bfloat16))
    r2 = run_chain(d2)
    assert np.array_equal(r1["out"], r2["out"])                 # q cannot matter
    w = bf16_bits_to_f64(d["w"]).reshape(H, NOPE + V, LORA)
    for b in range(2):
        c0 = bf16_bits_to_f64(d["slab"][d["tbl"][b, 0], 0, 0, :LORA])
        assert np.array_equal(r1["o_lat"][b], np.broadcast_to(d["slab"][d["tbl"][b, 0], 0, 0, :LORA],
                                                              (H, LORA)))
        exact = np.einsum("hvj,j->hv", w[:, NOPE:, :], c0)
        abs_sum = np.einsum("hvj,j->hv", np.abs(w[:, NOPE:, :]), np.abs(c0))
        assert within_f32_sum_bound(r1["out"][b], exact, abs_sum, LORA)


@pytest.mark.parametrize("n", [1, 2, 4, 8, 64, 128])
def test_uniform_softmax_closed_form(n):
    wl = synth.make_custom([n], seed=30 + n)
    d = np_inputs(wl)
    d["q"][:, :, :NOPE] = 0                                    # q_abs = 0
    d["slab"][:, :, :, LORA:] = 0                              # k_rope = 0
    r = run_chain(d, want_olat=True, probs_stride=n)
    p = bits_to_f32(r["probs"][0, :, :n])
    assert np.all(p == np.float32(1.0 / n))                   # exact for powers of two
    assert np.all(r["argmax"][0] == 0)
    rows = np.stack([bf16_bits_to_f64(d["slab"][d["tbl"][0, t // PAGE], 0, t % PAGE, :LORA])
                     for t in range(n)])
    mean = rows.mean(axis=0)
    abs_sum = np.abs(rows).mean(axis=0)
    assert within_f32_sum_bound(r["o_lat"][0], mean[None, :], abs_sum[None, :], n)


def test_all_unmapped_gives_zero_and_empty_gives_minus_one():
    wl = synth.make_custom([130, 5, 0], seed=40)
    d = np_inputs(wl)
    d["tbl"] = d["tbl"].copy()
    d["tbl"][0, :] = -1
    r = run_chain(d)
    assert np.all(r["out"][0] == 0) and np.all(r["argmax"][0] == 0)
    assert np.all(r["out"][2] == 0) and np.all(r["argmax"][2] == -1)
    assert np.any(r["out"][1] != 0)


# ---------------------------------------------------------------- invariants

def test_page_permutation_is_bitwise_invisible():
    wl = synth.make_custom([130, 64, 300, 1], seed=50)
    d = np_inputs(wl)
    base = run_chain(d, want_olat=True)
    perm = np.random.default_rng(3).permutation(wl.n_pages)       # new id of page p = perm[p]
    slab2 = np.empty_like(d["slab"])
    slab2[perm] = d["slab"]
    tbl2 = np.where(d["tbl"] >= 0, perm[np.maximum(d["tbl"], 0)], -1).astype(np.int32)
    r = run_chain(dict(d, slab=slab2, tbl=tbl2), want_olat=True)
    for k in ("out", "argmax", "o_lat"):
        assert np.array_equal(base[k], r[k])


def test_minus_one_equals_physical_zero_page():
    wl = synth.make_custom([200, 150], seed=51)
    d = np_inputs(wl)
    tbl_a = d["tbl"].copy()
    tbl_a[0, 1] = -1
    tbl_a[1, 0] = -1
    slab_b = np.concatenate([d["slab"], np.zeros_like(d["slab"][:1])])
    zero_id = slab_b.shape[0] - 1
    tbl_b = d["tbl"].copy()
    tbl_b[0, 1] = zero_id
    tbl_b[1, 0] = zero_id
    ra = run_chain(dict(d, tbl=tbl_a), want_olat=True)
    rb = run_chain(dict(d, slab=slab_b, tbl=tbl_b), want_olat=True)
    for k in ("out", "argmax", "o_lat"):
        assert np.array_equal(ra[k], rb[k])


def test_rows_past_context_are_never_read():
    wl = synth.make_custom([130, 70], seed=52, max_pages=4)
    d = np_inputs(wl)
    base = run_chain(d)
    slab = d["slab"].copy()
    nan = np.uint16(0x7FC0)
    for b in range(wl.B):
        n = int(wl.ctx_len[b])
        last = d["tbl"][b, (n - 1) // PAGE]
        slab[last, 0, n % PAGE if n % PAGE else PAGE:, :] = nan
    used = set(int(x) for x in d["tbl"].ravel() if x >= 0)
    for p in range(wl.n_pages):
        if p not in used:
            slab[p] = nan
    r = run_chain(dict(d, slab=slab))
    assert np.array_equal(base["out"], r["out"])
    assert np.all(np.isfinite(bits_to_f32(r["out"])))


def test_slots_are_independent():
    wl = synth.make_custom([90, 33, 257], seed=53)
    d = np_inputs(wl)
    full = run_chain(d)
    for b in range(wl.B):
        sub = dict(q=d["q"][b:b + 1], w=d["w"], slab=d["slab"], tbl=d["tbl"][b:b + 1],
                   ctx=d["ctx"][b:b + 1])
        r = run_chain(sub)
        assert np.array_equal(r["out"][0], full["out"][b])


# ---------------------------------------------------------------- second emulation

@pytest.mark.parametrize("n", [1, 3, 8])
def test_scalar_twin_bitwise(n):
    wl = synth.make_custom([n], seed=60 + n)
    d = np_inputs(wl)
    if n == 8:
        d["tbl"] = d["tbl"].copy()
        d["tbl"][0, 0] = d["tbl"][0, 0]        # keep mapped
    r = run_chain(d, probs_stride=n)
    w = d["w"].reshape(H, NOPE + V, LORA)
    for h in (0, 41, 95):
        rows = [d["slab"][d["tbl"][0, t // PAGE], 0, t % PAGE] for t in range(n)]
        out, p, s = twin_head(r["q_abs"][0, h], rows, n, w[h, NOPE:, :], synth.scale_bf16_bits())
        assert np.array_equal(bits_to_f32(r["out"][0, h]), out)
        assert np.array_equal(bits_to_f32(r["probs"][0, h, :n]), p)
        assert np.array_equal(r["scores"][0, h, :n], s)


# ---------------------------------------------------------------- append + bytes

def test_append_lands_in_the_mapped_row():
    wl = synth.make_custom([64, 65, 1, 130], n_layers=3, seed=70)
    slab = synth.bf16_bits(wl.slab).copy()
    before = slab.copy()
    pos = (wl.ctx_len - 1).astype(np.int32)
    pos[2] = -1                                          # no append for this slot
    c = synth.bf16_bits(wl.new_c[1])
    rope = synth.bf16_bits(wl.new_rope[1])
    skipped = oracle.append(slab, 1, wl.block_table, pos, c, rope)
    assert skipped == 0
    touched = np.zeros(slab.shape[:3], bool)
    for b in (0, 1, 3):
        pid = wl.block_table[b, pos[b] // PAGE]
        assert np.array_equal(slab[pid, 1, pos[b] % PAGE, :LORA], c[b])
        assert np.array_equal(slab[pid, 1, pos[b] % PAGE, LORA:], rope[b])
        touched[pid, 1, pos[b] % PAGE] = True
    assert np.array_equal(slab[~touched], before[~touched])


def test_whole_page_copy_moves_every_layer_of_the_page():
    """Adoption copy: each page of a tiny slab is filled with its own id (all layers, rows and
    columns), so after the copy a page's contents name the page it came from."""
    n_pages, L = 9, 3
    ids = np.arange(n_pages, dtype=np.uint16)[:, None, None, None]
    slab = np.broadcast_to(ids, (n_pages, L, PAGE, ROW)).copy()
    other = np.broadcast_to(ids[:4] + 100, (4, L, PAGE, ROW)).copy()   # a second pool (prefill side)
    src, dst = [2, 5, 8, 1], [7, 0, 3, 99]                         # the last pair is out of range
    assert oracle.copy_pages(slab, slab, src, dst) == 1
    want = np.arange(n_pages)
    want[[7, 0, 3]] = [2, 5, 8]
    assert np.array_equal(slab[:, 0, 0, 0], want)
    assert all((slab[p] == want[p]).all() for p in range(n_pages))   # every layer, row and column
    assert oracle.copy_pages(slab, other, [3, 0], [4, 6]) == 0      # cross-pool adoption
    assert (slab[4] == 103).all() and (slab[6] == 100).all() and (slab[5] == 5).all()


def _chunk_case(seed):
    """Two slots with 70 and 10 tokens cached, then chunks of 5 and 3 new tokens (packed)."""
    wl = synth.make_custom([75, 13], n_layers=2, seed=seed)
    pos0 = np.array([70, 10], np.int32)
    row_start = np.array([0, 5, 8], np.int32)
    rng = np.random.default_rng(seed)
    c = synth.bf16_bits(torch.from_numpy(rng.standard_normal((8, LORA)).astype(np.float32)).to(torch.bfloat16))
    r = synth.bf16_bits(torch.from_numpy(rng.standard_normal((8, ROW - LORA)).astype(np.float32)).to(torch.bfloat16))
    q = synth.bf16_bits(torch.from_numpy(rng.standard_normal((8, H, NOPE + ROPE)).astype(np.float32)).to(torch.bfloat16))
    return wl, pos0, row_start, c, r, q


def test_chunk_append_is_the_indexed_write_once_per_token():
    wl, pos0, row_start, c, r, _ = _chunk_case(80)
    a = synth.bf16_bits(wl.slab).copy()
    b = a.copy()
    tbl = wl.block_table.copy()
    tbl[1, 0] = -1                                          # slot 1's page 0 unmapped: its 3 rows skip
    assert oracle.append_rows(a, 1, tbl, pos0, row_start, c, r) == 3
    for j in range(5):                                      # the C oracle's single-row append, row by row
        pos = np.array([pos0[0] + j, pos0[1] + j if j < 3 else -1], np.int32)
        rows = [row_start[0] + j, row_start[1] + min(j, 2)]
        assert oracle.append(b, 1, tbl, pos, c[rows], r[rows]) == (1 if j < 3 else 0)
    assert np.array_equal(a, b)


def test_chunked_views_reproduce_the_token_loop():
    """Decoding a chunk through per-token views is bitwise the token-by-token loop it replaces:
    append token j, decode token j with the context grown by one, repeat."""
    wl, pos0, row_start, c, r, q = _chunk_case(81)
    w = synth.bf16_bits(wl.w_kv_b[1])
    q_abs = oracle.absorb(q, w)
    slab = synth.bf16_bits(wl.slab).copy()
    loop_out = np.zeros((8, H, V), np.uint16)
    for j in range(5):
        for b in range(2):
            if row_start[b] + j >= row_start[b + 1]:
                continue
            row = row_start[b] + j
            pos = np.full(2, -1, np.int32)
            pos[b] = pos0[b] + j
            cc = np.zeros((2, LORA), np.uint16)
            rr = np.zeros((2, ROW - LORA), np.uint16)
            cc[b], rr[b] = c[row], r[row]
            oracle.append(slab, 1, wl.block_table, pos, cc, rr)
            ctx = np.array([pos0[b] + j + 1], np.int32)
            o = oracle.decode(q_abs[row:row + 1], slab, 1, wl.block_table[b:b + 1], ctx, w, wl.scale_bits)
            loop_out[row] = o["out"][0]
    slab2 = synth.bf16_bits(wl.slab).copy()
    oracle.append_rows(slab2, 1, wl.block_table, pos0, row_start, c, r)
    assert np.array_equal(slab, slab2)
    vt, vc = oracle.chunk_views(wl.block_table, pos0, row_start, 9)   # one row past the chunk
    assert list(vc) == [71, 72, 73, 74, 75, 11, 12, 13, 0] and (vt[8] == -1).all()
    assert np.array_equal(vt[3], wl.block_table[0]) and np.array_equal(vt[6], wl.block_table[1])
    chunked = oracle.decode(q_abs, slab2, 1, vt[:8], vc[:8], w, wl.scale_bits)
    assert np.array_equal(chunked["out"], loop_out)


def test_byte_figures_from_the_page():
    """27.6 KB/token absorbed vs ~1.47 MB/token expanded over the 24 MLA layers."""
    rows = dict(line.split("=", 1) for line in open(os.path.join(GOLDEN, "bytes_per_token.txt"))
                .read().splitlines() if line and not line.startswith("#"))
    L = int(rows["mla_layers"])
    absorbed = L * ROW * 2                                       # one slab row per layer
    expanded = L * H * ((NOPE + ROPE) + V) * 2                   # per-head K (192) + V (128)
    assert absorbed == int(rows["absorbed_bytes_per_token"])
    assert expanded == int(rows["expanded_bytes_per_token"])
    assert round(absorbed / 1000, 1) == float(rows["absorbed_kb_printed"])
    assert round(expanded / 1e6, 2) == float(rows["expanded_mb_printed"])
    wl = synth.make_custom([1], n_layers=L, seed=1)
    per_token = wl.slab[0, :, 0, :].numel() * wl.slab.element_size()
    assert per_token == absorbed


# ---------------------------------------------------------------- negative controls

def _pins_failed(mutation: int) -> list[str]:
    failed = []
    for name, wl, layer in (("expanded_tiny", synth.make_workload("tiny"), 0),
                            ("expanded_small", synth.make_custom([3, 65], seed=81), 0),
                            ("expanded_layers", synth.make_custom([70], n_layers=2, seed=82), 1)):
        _, _, _, err = _vs_expanded(wl, layer, mutation=mutation)
        if not (err.max() <= ULP_TOL):
            failed.append(name)
    wl = synth.make_custom([4], seed=83)
    d = np_inputs(wl)
    d["q"][:, :, :NOPE] = 0
    d["slab"][:, :, :, LORA:] = 0
    r = run_chain(d, probs_stride=4, mutation=mutation)
    if not np.all(bits_to_f32(r["probs"][0, :, :4]) == np.float32(0.25)):
        failed.append("uniform")
    return failed


@pytest.mark.parametrize("name", [k for k in oracle.MUTATIONS if k != "none"])
def test_planted_mistake_is_caught(name):
    assert _pins_failed(oracle.MUTATIONS[name]), f"mutation {name} slipped through every pin"


def test_faithful_oracle_passes_the_same_pins():
    assert _pins_failed(0) == []
