"""ctypes wrapper around ``k3mla_oracle.c`` (the rounding-chain oracle).

TEST INFRASTRUCTURE ONLY -- see ``oracle/__init__.py``.

All bf16 arrays are numpy ``uint16`` arrays holding bf16 bit patterns.
Geometry (pegainfer PR #869, "K3: paged latent MLA KV + absorbed decode", M1
and M2 commits): 96 heads, q_nope 128, q_rope 64, v_head 128, kv_lora 512,
page 64 tokens, cache row 576 = 512 latent + 64 rope.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

H, NOPE, ROPE, V, LORA, PAGE = 96, 128, 64, 128, 512, 64
ROW = LORA + ROPE

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "k3mla_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libk3mla_oracle.so")

# Planted mistakes for negative-control tests (0 is the faithful oracle).
MUTATIONS = {
    "none": 0,
    "drop_rope": 1,
    "swap_wuk_wuv": 2,
    "no_scale": 3,
    "page_off_by_one": 4,
    "drop_last_in_sum": 5,
    "transpose_wuk": 6,
    "layer_ignored": 7,
    "rope_sign": 8,
}

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (plain -O2, no contraction, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
             "-shared", "-pthread", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            lib.k3o_f32_to_bf16.argtypes = [P, P, ctypes.c_size_t]
            lib.k3o_f32_to_bf16.restype = None
            lib.k3o_absorb.argtypes = [P, P, I, P, I]
            lib.k3o_absorb.restype = None
            lib.k3o_decode.argtypes = [P, P, I, I, I, P, I, P, P, ctypes.c_uint16, P, I,
                                       P, P, P, P, P, I, I, I]
            lib.k3o_decode.restype = I
            lib.k3o_append.argtypes = [P, I, I, I, P, I, P, P, ctypes.c_longlong, P,
                                       ctypes.c_longlong, I]
            lib.k3o_append.restype = I
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    a = np.ascontiguousarray(a)
    assert a.dtype == dtype, (a.dtype, dtype)
    return a


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """The oracle's own f32 -> bf16 round-to-nearest-even (bit patterns)."""
    x = _c(np.asarray(x, dtype=np.float32), np.float32)
    y = np.empty(x.shape, np.uint16)
    _load().k3o_f32_to_bf16(_ptr(x), _ptr(y), x.size)
    return y


def absorb(q: np.ndarray, w_kv_b: np.ndarray, mutation: int = 0) -> np.ndarray:
    """Step 1 of the chain.  q [B,96,192] bf16, w_kv_b [24576,512] bf16 -> q_abs [B,96,576]."""
    q = _c(q, np.uint16)
    w = _c(w_kv_b, np.uint16)
    B = q.shape[0]
    assert q.shape == (B, H, NOPE + ROPE) and w.shape == (H * (NOPE + V), LORA)
    out = np.empty((B, H, ROW), np.uint16)
    _load().k3o_absorb(_ptr(q), _ptr(w), B, _ptr(out), mutation)
    return out


def decode(q_abs, slab, layer, block_table, ctx_len, w_kv_b, scale_bf16, slots=None,
           nthreads: int = 1, want_olat: bool = False, probs_stride: int = 0,
           mutation: int = 0):
    """Steps 2-7 of the chain for the listed slots.

    q_abs [B,96,576] bf16; slab [n_pages, L, 64, 576] bf16; block_table
    [B, max_pages] int32; ctx_len [B] int32; w_kv_b [24576, 512] bf16.
    Returns a dict with ``out`` [B,96,128] bf16, ``argmax`` [B,96] int32,
    optionally ``o_lat`` [B,96,512] bf16 and, when ``probs_stride`` > 0,
    ``probs`` (bf16 p_t) and ``scores`` (bf16-valued s_t as f32) padded to that
    many tokens, plus ``bad_table``.  Rows of slots not listed stay zero.
    """
    q_abs = _c(q_abs, np.uint16)
    slab = _c(slab, np.uint16)
    tbl = _c(block_table, np.int32)
    ctx = _c(ctx_len, np.int32)
    w = _c(w_kv_b, np.uint16)
    B = q_abs.shape[0]
    n_pages, L = slab.shape[0], slab.shape[1]
    assert slab.shape[2:] == (PAGE, ROW)
    max_pages = tbl.shape[1]
    assert tbl.shape[0] == B and ctx.shape == (B,)
    if slots is None:
        slots = np.arange(B, dtype=np.int32)
    slots = _c(np.asarray(slots, dtype=np.int32), np.int32)
    out = np.zeros((B, H, V), np.uint16)
    am = np.full((B, H), -7, np.int32)
    ol = np.zeros((B, H, LORA), np.uint16) if want_olat else None
    probs = np.zeros((B, H, probs_stride), np.uint16) if probs_stride > 0 else None
    scores = np.zeros((B, H, probs_stride), np.float32) if probs_stride > 0 else None
    bad = _load().k3o_decode(
        _ptr(q_abs), _ptr(slab), n_pages, L, layer, _ptr(tbl), max_pages, _ptr(ctx), _ptr(w),
        int(scale_bf16), _ptr(slots), len(slots), _ptr(out), _ptr(am),
        _ptr(ol) if ol is not None else None,
        _ptr(probs) if probs is not None else None,
        _ptr(scores) if scores is not None else None,
        probs_stride, nthreads, mutation)
    res = {"out": out, "argmax": am, "bad_table": bool(bad)}
    if ol is not None:
        res["o_lat"] = ol
    if probs is not None:
        res["probs"] = probs
        res["scores"] = scores
    return res


def append(slab, layer, block_table, pos, c_kv, k_rope) -> int:
    """In-place append of one row per slot (the indexed write).  Returns rows skipped."""
    assert slab.flags["C_CONTIGUOUS"] and slab.dtype == np.uint16
    tbl = _c(block_table, np.int32)
    pos = _c(pos, np.int32)
    c_kv = _c(c_kv, np.uint16)
    k_rope = _c(k_rope, np.uint16)
    B = pos.shape[0]
    return _load().k3o_append(_ptr(slab), slab.shape[0], slab.shape[1], layer, _ptr(tbl),
                              tbl.shape[1], _ptr(pos), _ptr(c_kv), c_kv.shape[1], _ptr(k_rope),
                              k_rope.shape[1], B)
