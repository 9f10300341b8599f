"""Helpers for the GPU tests: run the CUDA path through the C-ABI binding, run the
oracle on the same seeded inputs, and compare with the stated tolerance."""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle
from paged_latent_attention_k3mla_gb300 import k3mla, synth
from tests.helpers import argmax_mismatch_ok, bits_to_f32, row_ulp_error, ULP_TOL

H, NOPE, ROPE, V, LORA, PAGE, ROW = 96, 128, 64, 128, 512, 64, 576
NTHREADS = max(1, min(32, os.cpu_count() or 1))


def dump(name: str, **arrays):
    """Keep arrays of a failing comparison for offline study, in the directory that the
    K3MLA_DUMP_DIR environment variable names (nothing is written when it is unset)."""
    d = os.environ.get("K3MLA_DUMP_DIR")
    if d and os.path.isdir(d):
        np.savez_compressed(os.path.join(d, f"{name}.npz"), **arrays)


def to_dev(wl: synth.Workload):
    return dict(table=torch.from_numpy(wl.block_table).cuda(), ctx=torch.from_numpy(wl.ctx_len).cuda())


def gpu_layer(wl, layer, split=None, max_ctx=None, table=None, ctx=None, slab=None, want_qabs=False,
              dev_err=None):
    """absorb + paged decode of one layer through the C ABI.  Returns numpy bits."""
    B = wl.B
    max_ctx = max_ctx or max(PAGE, int(wl.block_table.shape[1]) * PAGE)
    split = k3mla.SPLIT_AUTO if split is None else split
    table = torch.from_numpy(wl.block_table).cuda() if table is None else table
    ctx = torch.from_numpy(wl.ctx_len).cuda() if ctx is None else ctx
    slab = wl.slab if slab is None else slab
    q_abs = torch.empty(B, H, ROW, dtype=torch.bfloat16, device="cuda")
    k3mla.absorb_q(wl.q[layer], wl.w_kv_b[layer], q_abs)
    out = torch.full((B, H, V), float("nan"), dtype=torch.bfloat16, device="cuda")
    am = torch.full((B, H), -7, dtype=torch.int32, device="cuda")
    ws = torch.empty(k3mla.decode_workspace_bytes(B, max_ctx, split), dtype=torch.uint8, device="cuda")
    ws.fill_(0xFF)   # NaN-poisoned scratch: every read value must have been written
    err = torch.zeros(1, dtype=torch.int32, device="cuda") if dev_err is None else dev_err
    k3mla.paged_decode(q_abs, slab, layer, table, ctx, wl.w_kv_b[layer], wl.scale_bits, out, ws, max_ctx,
                       split, argmax=am, dev_err=err)
    torch.cuda.synchronize()
    res = dict(out=synth.bf16_bits(out), argmax=am.cpu().numpy(), dev_err=int(err.item()), split=split)
    if want_qabs:
        res["q_abs"] = synth.bf16_bits(q_abs)
    return res


def compact(wl, layer, slots):
    """The pages the listed slots use at `layer`, as a 1-layer slab with a remapped
    table (page ids never enter the arithmetic, so the oracle may see any ids)."""
    slots = list(slots)
    tbl = wl.block_table[slots]
    # ids outside [0, n_pages) read as zero rows, like -1: they never reach the page gather below
    used = sorted(set(int(x) for x in tbl.ravel() if 0 <= x < wl.slab.shape[0]))
    remap = {p: i for i, p in enumerate(used)}
    idx = torch.tensor(used if used else [0], dtype=torch.long, device=wl.slab.device)
    pages = wl.slab.index_select(0, idx)[:, layer:layer + 1]
    slab = synth.bf16_bits(pages)
    t2 = np.vectorize(lambda x: remap.get(int(x), -1))(tbl).astype(np.int32) if tbl.size else tbl
    return slab, t2


def oracle_layer(wl, layer, slots=None, probs_stride=0):
    """The oracle's chain for the listed slots (all if None) of one layer."""
    slots = list(range(wl.B)) if slots is None else list(slots)
    slab, tbl = compact(wl, layer, slots)
    q = synth.bf16_bits(wl.q[layer][slots])
    w = synth.bf16_bits(wl.w_kv_b[layer])
    q_abs = oracle.absorb(q, w)
    ctx = wl.ctx_len[slots].astype(np.int32)
    r = oracle.decode(q_abs, slab, 0, tbl, ctx, w, wl.scale_bits, nthreads=NTHREADS,
                      probs_stride=probs_stride)
    r["slots"] = slots
    return r


def compare(gpu, orc, ctx, name="decode", check_argmax=True):
    """Element-wise parity of the sampled slots; returns the error statistics."""
    slots = orc["slots"]
    g = bits_to_f32(gpu["out"][slots])
    o = bits_to_f32(orc["out"])
    err = row_ulp_error(g, o)
    stats = dict(max_ulp=float(err.max()), mean_ulp=float(err.mean()),
                 exact=float((gpu["out"][slots] == orc["out"]).mean()))
    ok = np.all(np.isfinite(g)) and err.max() <= ULP_TOL
    flips = 0
    if check_argmax and "scores" in orc:
        for i, b in enumerate(slots):
            n = int(ctx[b])
            for h in range(H):
                a_ref, a_gpu = int(orc["argmax"][i, h]), int(gpu["argmax"][b, h])
                if n == 0:
                    ok = ok and a_gpu == -1 and a_ref == -1
                    continue
                if a_ref != a_gpu:
                    flips += 1
                    if not argmax_mismatch_ok(orc["scores"][i, h], orc["probs"][i, h], n, a_ref, a_gpu):
                        ok = False
    stats["argmax_coin_flips"] = flips
    if not ok:
        dump(f"fail_{name}", gpu=gpu["out"][slots], oracle=orc["out"], gpu_argmax=gpu["argmax"][slots],
             oracle_argmax=orc["argmax"], ctx=np.asarray(ctx)[slots])
    return ok, stats
