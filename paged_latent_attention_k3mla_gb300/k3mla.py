"""Thin ctypes binding of libk3mla.so (declared in include/k3mla.h).

Argument marshalling only: every function checks shapes / dtypes / devices,
passes raw pointers and the current CUDA stream to the C ABI, and raises on a
non-zero status.  All arithmetic runs in the library's CUDA kernels; if the
library cannot be built or loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import threading

import numpy as np
import torch

from . import build as _build

H, NOPE, ROPE, V, LORA, PAGE, ROW, TILE = 96, 128, 64, 128, 512, 64, 576, 128
SPLIT_AUTO, SPLIT_MAX = 0, 4096   # K3MLA_SPLIT_AUTO (the default per-slot rule), K3MLA_SPLIT_MAX

DEV_BAD_PAGE, DEV_UNMAPPED, DEV_CTX, DEV_TIMEOUT = 1, 2, 4, 8

# Every symbol include/k3mla.h declares.
EXPORTS = (
    "k3mla_last_error", "k3mla_absorb_q", "k3mla_append_latent", "k3mla_decode_workspace_bytes",
    "k3mla_paged_decode", "k3mla_slot_split_tokens", "k3mla_pool_create", "k3mla_pool_ensure",
    "k3mla_pool_release_slot", "k3mla_pool_host_table", "k3mla_pool_max_pages", "k3mla_pool_n_pages",
    "k3mla_pool_stats", "k3mla_pool_destroy", "k3mla_diag_umma", "k3mla_paged_decode_noalloc",
    "k3mla_absorb_q_append", "k3mla_pool_share_prefix", "k3mla_pool_cow", "k3mla_pool_page_refs",
    "k3mla_copy_pages", "k3mla_append_latent_rows", "k3mla_chunk_views", "k3mla_decode_exact",
    "k3mla_decode_exact_workspace_bytes", "k3mla_pool_ensure_all", "k3mla_batch_planned_split_tokens",
    "k3mla_decode_layer_workspace_bytes", "k3mla_decode_layer", "k3mla_diag_decode_timeout",
    "k3mla_expanded_cache_bytes", "k3mla_expand_latent_cache", "k3mla_expanded_decode", "k3mla_diag_exact_exp",
    "k3mla_chunk_decode_workspace_bytes", "k3mla_chunk_decode",
)

# Size of the library's built-in decode scratch (K3MLA_NOALLOC_SCRATCH_BYTES).
NOALLOC_SCRATCH_BYTES = 16 << 20

_lib = None
_lock = threading.Lock()


class K3mlaError(RuntimeError):
    pass


def load(build_if_needed: bool = True):
    """Load libk3mla.so (building it first when it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.build() if build_if_needed else _build.LIB
        lib = ctypes.CDLL(path)
        P, I, I64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
        sig = {
            "k3mla_last_error": ([], ctypes.c_char_p),
            "k3mla_absorb_q": ([P, P, P, I, P], I),
            "k3mla_append_latent": ([P, I, I, I, P, I, P, P, I64, P, I64, I, P, P], I),
            "k3mla_decode_workspace_bytes": ([I, I, I], SZ),
            "k3mla_paged_decode": ([P, P, I, I, I, P, I, P, P, ctypes.c_uint16, P, P, P, SZ, I, I, I, P, P],
                                   I),
            "k3mla_slot_split_tokens": ([I, I], I),
            "k3mla_batch_planned_split_tokens": ([P, I, I], I),
            "k3mla_pool_create": ([I, I, I, ctypes.c_uint64, ctypes.POINTER(P)], I),
            "k3mla_pool_ensure": ([P, I, I], I),
            "k3mla_pool_ensure_all": ([P, P, I], I),
            "k3mla_pool_release_slot": ([P, I], I),
            "k3mla_pool_host_table": ([P], ctypes.POINTER(ctypes.c_int32)),
            "k3mla_pool_max_pages": ([P], I),
            "k3mla_pool_n_pages": ([P], I),
            "k3mla_pool_stats": ([P, ctypes.POINTER(I), ctypes.POINTER(I)], I),
            "k3mla_pool_destroy": ([P], None),
            "k3mla_diag_umma": ([I, P, P, P, P], I),
            "k3mla_expanded_cache_bytes": ([I], SZ),
            "k3mla_expand_latent_cache": ([P, I, I, I, P, P, P, P], I),
            "k3mla_expanded_decode": ([P, P, I, P, I, P, ctypes.c_uint16, P, I, I, P, P], I),
            "k3mla_diag_exact_exp": ([P, P, P, I, P], I),
            "k3mla_diag_decode_timeout": ([P, P, I, I, I, P, I, P, P, ctypes.c_uint16, P, P, P, SZ, I, I, I, I,
                                           ctypes.c_uint32, P, P], I),
            "k3mla_paged_decode_noalloc": ([P, P, I, I, I, P, I, P, P, ctypes.c_uint16, P, P, I, I, I, P, P], I),
            "k3mla_absorb_q_append": ([P, P, P, P, I, I, I, P, I, P, P, I64, P, I64, I, P, P], I),
            "k3mla_pool_share_prefix": ([P, I, I, I], I),
            "k3mla_pool_cow": ([P, I, I, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)], I),
            "k3mla_pool_page_refs": ([P, I], I),
            "k3mla_copy_pages": ([P, I, P, I, I, P, P, I, P, P], I),
            "k3mla_append_latent_rows": ([P, I, I, I, P, I, P, P, P, I64, P, I64, I, I, P, P], I),
            "k3mla_chunk_views": ([P, I, I, P, P, I, P, P, P], I),
            "k3mla_chunk_decode_workspace_bytes": ([I, I, I], SZ),
            "k3mla_chunk_decode": ([P, P, I, I, I, P, I, P, P, I, I, P, ctypes.c_uint16, P, P, P, SZ, I, P, P], I),
            "k3mla_decode_exact_workspace_bytes": ([I, I], SZ),
            "k3mla_decode_layer_workspace_bytes": ([I, I], SZ),
            "k3mla_decode_layer": ([P, P, P, I, I, I, P, I, P, P, I64, P, I64, ctypes.c_uint16, P, P, P, SZ, I, I, P, P],
                                   I),
            "k3mla_decode_exact": ([P, P, I, I, I, P, I, P, P, ctypes.c_uint16, P, P, P, SZ, I, I, P, P], I),
        }
        for name, (args, res) in sig.items():
            f = getattr(lib, name)
            f.argtypes = args
            f.restype = res
        _lib = lib
        return lib


def _check(rc: int, what: str):
    if rc != 0:
        msg = load().k3mla_last_error().decode(errors="replace")
        raise K3mlaError(f"{what} failed with status {rc}: {msg}")


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dev(t: torch.Tensor, dtype, shape=None, name="tensor"):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise K3mlaError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise K3mlaError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise K3mlaError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise K3mlaError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return ctypes.c_void_p(t.data_ptr())


def _opt(t, dtype, shape, name):
    return None if t is None else _dev(t, dtype, shape, name)


def absorb_q(q: torch.Tensor, w_kv_b: torch.Tensor, q_abs: torch.Tensor, stream=None) -> None:
    """q [B,96,192] bf16, w_kv_b [24576,512] bf16 -> q_abs [B,96,576] bf16 (written)."""
    B = q.shape[0]
    lib = load()
    _check(lib.k3mla_absorb_q(_dev(q, torch.bfloat16, (B, H, NOPE + ROPE), "q"),
                              _dev(w_kv_b, torch.bfloat16, (H * (NOPE + V), LORA), "w_kv_b"),
                              _dev(q_abs, torch.bfloat16, (B, H, ROW), "q_abs"), B, _stream(stream)),
           "k3mla_absorb_q")


def append_latent(slab: torch.Tensor, layer: int, block_table: torch.Tensor, pos: torch.Tensor,
                  c_kv: torch.Tensor, k_rope: torch.Tensor, dev_err: torch.Tensor | None = None,
                  stream=None) -> None:
    """slab [n_pages,L,64,576] bf16 (in place); block_table [B,max_pages] int32; pos [B]
    int32; c_kv [B,>=512] bf16 and k_rope [B,>=64] bf16 with unit inner stride."""
    n_pages, L = slab.shape[0], slab.shape[1]
    B = pos.shape[0]
    for t, name in ((c_kv, "c_kv"), (k_rope, "k_rope")):
        if not t.is_cuda or t.dtype != torch.bfloat16 or t.dim() != 2 or t.stride(1) != 1 or t.shape[0] != B:
            raise K3mlaError(f"{name} must be a CUDA bf16 [B, n] tensor with unit inner stride")
    lib = load()
    _check(lib.k3mla_append_latent(
        _dev(slab, torch.bfloat16, (n_pages, L, PAGE, ROW), "slab"), n_pages, L, int(layer),
        _dev(block_table, torch.int32, None, "block_table"), block_table.shape[1],
        _dev(pos, torch.int32, (B,), "pos"), ctypes.c_void_p(c_kv.data_ptr()), c_kv.stride(0),
        ctypes.c_void_p(k_rope.data_ptr()), k_rope.stride(0), B,
        _opt(dev_err, torch.int32, (1,), "dev_err"), _stream(stream)), "k3mla_append_latent")


def _rows(t: torch.Tensor, B: int, name: str):
    if not t.is_cuda or t.dtype != torch.bfloat16 or t.dim() != 2 or t.stride(1) != 1 or t.shape[0] != B:
        raise K3mlaError(f"{name} must be a CUDA bf16 [B, n] tensor with unit inner stride")
    return ctypes.c_void_p(t.data_ptr())


def absorb_q_append(q: torch.Tensor, w_kv_b: torch.Tensor, q_abs: torch.Tensor, slab: torch.Tensor, layer: int,
                    block_table: torch.Tensor, pos: torch.Tensor, c_kv: torch.Tensor, k_rope: torch.Tensor,
                    dev_err: torch.Tensor | None = None, stream=None) -> None:
    """absorb_q(q, w_kv_b, q_abs) and append_latent(slab, layer, block_table, pos, c_kv, k_rope)
    in one launch (same arguments, same results)."""
    B = q.shape[0]
    n_pages, L = slab.shape[0], slab.shape[1]
    lib = load()
    _check(lib.k3mla_absorb_q_append(
        _dev(q, torch.bfloat16, (B, H, NOPE + ROPE), "q"),
        _dev(w_kv_b, torch.bfloat16, (H * (NOPE + V), LORA), "w_kv_b"),
        _dev(q_abs, torch.bfloat16, (B, H, ROW), "q_abs"),
        _dev(slab, torch.bfloat16, (n_pages, L, PAGE, ROW), "slab"), n_pages, L, int(layer),
        _dev(block_table, torch.int32, None, "block_table"), block_table.shape[1],
        _dev(pos, torch.int32, (B,), "pos"), _rows(c_kv, B, "c_kv"), c_kv.stride(0),
        _rows(k_rope, B, "k_rope"), k_rope.stride(0), B,
        _opt(dev_err, torch.int32, (1,), "dev_err"), _stream(stream)), "k3mla_absorb_q_append")


def copy_pages(dst_slab: torch.Tensor, src_slab: torch.Tensor, src_ids: torch.Tensor, dst_ids: torch.Tensor,
               dev_err: torch.Tensor | None = None, stream=None) -> None:
    """Whole-page copies page src_ids[i] of src_slab -> page dst_ids[i] of dst_slab (all layers);
    slabs [n_pages, L, 64, 576] bf16 with the same L (may be the same tensor)."""
    n = src_ids.shape[0]
    L = dst_slab.shape[1]
    if src_slab.dim() != 4 or src_slab.shape[1] != L:
        raise K3mlaError("src_slab must be [n_pages, L, 64, 576] with the layer count of dst_slab")
    lib = load()
    _check(lib.k3mla_copy_pages(
        _dev(dst_slab, torch.bfloat16, (dst_slab.shape[0], L, PAGE, ROW), "dst_slab"), dst_slab.shape[0],
        _dev(src_slab, torch.bfloat16, (src_slab.shape[0], L, PAGE, ROW), "src_slab"), src_slab.shape[0], L,
        _dev(src_ids, torch.int32, (n,), "src_ids"), _dev(dst_ids, torch.int32, (n,), "dst_ids"), n,
        _opt(dev_err, torch.int32, (1,), "dev_err"), _stream(stream)), "k3mla_copy_pages")


def append_latent_rows(slab: torch.Tensor, layer: int, block_table: torch.Tensor, pos0: torch.Tensor,
                       row_start: torch.Tensor, c_kv: torch.Tensor, k_rope: torch.Tensor, max_rows: int,
                       dev_err: torch.Tensor | None = None, stream=None) -> None:
    """Chunk append: row r of c_kv [R, >=512] / k_rope [R, >=64] (slot b's rows row_start[b] ..
    row_start[b+1]-1) lands at position pos0[b] + (r - row_start[b]) of slot b."""
    n_pages, L = slab.shape[0], slab.shape[1]
    B = pos0.shape[0]
    R = c_kv.shape[0]
    lib = load()
    _check(lib.k3mla_append_latent_rows(
        _dev(slab, torch.bfloat16, (n_pages, L, PAGE, ROW), "slab"), n_pages, L, int(layer),
        _dev(block_table, torch.int32, None, "block_table"), block_table.shape[1],
        _dev(pos0, torch.int32, (B,), "pos0"), _dev(row_start, torch.int32, (B + 1,), "row_start"),
        _rows(c_kv, R, "c_kv"), c_kv.stride(0), _rows(k_rope, R, "k_rope"), k_rope.stride(0), B, int(max_rows),
        _opt(dev_err, torch.int32, (1,), "dev_err"), _stream(stream)), "k3mla_append_latent_rows")


def chunk_views(block_table: torch.Tensor, pos0: torch.Tensor, row_start: torch.Tensor,
                view_table: torch.Tensor, view_ctx: torch.Tensor, stream=None) -> None:
    """Per-token views of the chunks: view_table [R, max_pages] and view_ctx [R] (written)."""
    B, M = block_table.shape
    R = view_ctx.shape[0]
    lib = load()
    _check(lib.k3mla_chunk_views(
        _dev(block_table, torch.int32, (B, M), "block_table"), B, M, _dev(pos0, torch.int32, (B,), "pos0"),
        _dev(row_start, torch.int32, (B + 1,), "row_start"), R, _dev(view_table, torch.int32, (R, M), "view_table"),
        _dev(view_ctx, torch.int32, (R,), "view_ctx"), _stream(stream)), "k3mla_chunk_views")


def chunk_decode_workspace_bytes(B: int, R: int, max_ctx: int) -> int:
    return int(load().k3mla_chunk_decode_workspace_bytes(B, R, max_ctx))


def chunk_decode(q_abs: torch.Tensor, slab: torch.Tensor, layer: int, block_table: torch.Tensor,
                 pos0: torch.Tensor, row_start: torch.Tensor, w_kv_b: torch.Tensor, scale_bf16: int,
                 out: torch.Tensor, workspace: torch.Tensor, max_ctx: int, argmax: torch.Tensor | None = None,
                 dev_err: torch.Tensor | None = None, stream=None) -> None:
    """Multi-query decode of prefill chunks (k3mla_chunk_decode): q_abs [R, 96, 576] of the chunks'
    token rows (slot b's rows row_start[b] .. row_start[b+1]-1, row j at position pos0[b] + j) ->
    out [R, 96, 128], each row attending causally over its slot's cache."""
    R = q_abs.shape[0]
    B = pos0.shape[0]
    n_pages, L = slab.shape[0], slab.shape[1]
    if workspace.dtype != torch.uint8 or not workspace.is_cuda:
        raise K3mlaError("workspace must be a CUDA uint8 tensor")
    lib = load()
    _check(lib.k3mla_chunk_decode(
        _dev(q_abs, torch.bfloat16, (R, H, ROW), "q_abs"), _dev(slab, torch.bfloat16, (n_pages, L, PAGE, ROW), "slab"),
        n_pages, L, int(layer), _dev(block_table, torch.int32, None, "block_table"), block_table.shape[1],
        _dev(pos0, torch.int32, (B,), "pos0"), _dev(row_start, torch.int32, (B + 1,), "row_start"), B, R,
        _dev(w_kv_b, torch.bfloat16, (H * (NOPE + V), LORA), "w_kv_b"), ctypes.c_uint16(scale_bf16),
        _dev(out, torch.bfloat16, (R, H, V), "out"), _opt(argmax, torch.int32, (R, H), "argmax"),
        ctypes.c_void_p(workspace.data_ptr()), workspace.numel(), int(max_ctx),
        _opt(dev_err, torch.int32, (1,), "dev_err"), _stream(stream)), "k3mla_chunk_decode")


def decode_exact_workspace_bytes(B: int, max_ctx: int) -> int:
    return int(load().k3mla_decode_exact_workspace_bytes(B, max_ctx))


def decode_exact(q: torch.Tensor, slab: torch.Tensor, layer: int, block_table: torch.Tensor, ctx_len: torch.Tensor,
                 w_kv_b: torch.Tensor, scale_bf16: int, out: torch.Tensor, workspace: torch.Tensor, max_ctx: int,
                 argmax: torch.Tensor | None = None, dev_err: torch.Tensor | None = None, stream=None) -> None:
    """The exact-chain decode (absorption included): q [B,96,192] bf16 -> out [B,96,128] bf16."""
    B = q.shape[0]
    n_pages, L = slab.shape[0], slab.shape[1]
    lib = load()
    _check(lib.k3mla_decode_exact(
        _dev(q, torch.bfloat16, (B, H, NOPE + ROPE), "q"), _dev(slab, torch.bfloat16, (n_pages, L, PAGE, ROW), "slab"),
        n_pages, L, int(layer), _dev(block_table, torch.int32, None, "block_table"), block_table.shape[1],
        _dev(ctx_len, torch.int32, (B,), "ctx_len"), _dev(w_kv_b, torch.bfloat16, (H * (NOPE + V), LORA), "w_kv_b"),
        ctypes.c_uint16(scale_bf16), _dev(out, torch.bfloat16, (B, H, V), "out"),
        _opt(argmax, torch.int32, (B, H), "argmax"), _dev(workspace, torch.uint8, None, "workspace"),
        workspace.numel(), B, int(max_ctx), _opt(dev_err, torch.int32, (1,), "dev_err"), _stream(stream)),
        "k3mla_decode_exact")


def decode_layer_workspace_bytes(B: int, max_ctx: int) -> int:
    return int(load().k3mla_decode_layer_workspace_bytes(B, max_ctx))



def decode_layer(q: torch.Tensor, w_kv_b: torch.Tensor, slab: torch.Tensor, layer: int, block_table: torch.Tensor,
                 ctx_len: torch.Tensor, c_kv: torch.Tensor, k_rope: torch.Tensor, scale_bf16: int, out: torch.Tensor,
                 workspace: torch.Tensor, max_ctx: int, argmax: torch.Tensor | None = None,
                 dev_err: torch.Tensor | None = None, stream=None) -> None:
    """One decode step of one layer (append at ctx_len - 1, absorption, paged decode under the
    default split); see k3mla_decode_layer.  `workspace`: uint8, >= decode_layer_workspace_bytes."""
    B = q.shape[0]
    n_pages, L = slab.shape[0], slab.shape[1]
    if workspace.dtype != torch.uint8 or not workspace.is_cuda:
        raise K3mlaError("workspace must be a CUDA uint8 tensor")
    lib = load()
    _check(lib.k3mla_decode_layer(
        _dev(q, torch.bfloat16, (B, H, NOPE + ROPE), "q"), _dev(w_kv_b, torch.bfloat16, (H * (NOPE + V), LORA), "w_kv_b"),
        _dev(slab, torch.bfloat16, (n_pages, L, PAGE, ROW), "slab"), n_pages, L, int(layer),
        _dev(block_table, torch.int32, None, "block_table"), block_table.shape[1],
        _dev(ctx_len, torch.int32, (B,), "ctx_len"), _rows(c_kv, B, "c_kv"), c_kv.stride(0),
        _rows(k_rope, B, "k_rope"), k_rope.stride(0), ctypes.c_uint16(scale_bf16),
        _dev(out, torch.bfloat16, (B, H, V), "out"), _opt(argmax, torch.int32, (B, H), "argmax"),
        ctypes.c_void_p(workspace.data_ptr()), workspace.numel(), B, int(max_ctx),
        _opt(dev_err, torch.int32, (1,), "dev_err"), _stream(stream)), "k3mla_decode_layer")


def decode_workspace_bytes(B: int, max_ctx: int, split_tokens: int = SPLIT_AUTO) -> int:
    return int(load().k3mla_decode_workspace_bytes(B, max_ctx, split_tokens))


def slot_split_tokens(ctx: int, split_tokens: int = SPLIT_AUTO) -> int:
    """The split length a slot of context ctx gets (k3mla_slot_split_tokens)."""
    rc = int(load().k3mla_slot_split_tokens(int(ctx), int(split_tokens)))
    if rc < 0:
        _check(rc, "k3mla_slot_split_tokens")
    return rc


def batch_planned_split_tokens(ctx_len, max_ctx: int) -> int:
    """OPT-IN, batch-dependent numerics: one split length planned for a batch whose context
    lengths are known on the host (a sequence or array of ints, one per slot); see
    k3mla_batch_planned_split_tokens.  Passing it as split_tokens makes a slot's output bits
    depend on the rest of the batch and on the GPU."""
    ctx = np.ascontiguousarray(np.asarray(ctx_len, dtype=np.int32).reshape(-1))
    rc = int(load().k3mla_batch_planned_split_tokens(ctx.ctypes.data_as(ctypes.c_void_p), int(ctx.size), max_ctx))
    if rc < 0:
        _check(rc, "k3mla_batch_planned_split_tokens")
    return rc


def paged_decode(q_abs: torch.Tensor, slab: torch.Tensor, layer: int, block_table: torch.Tensor,
                 ctx_len: torch.Tensor, w_kv_b: torch.Tensor, scale_bf16: int, out: torch.Tensor,
                 workspace: torch.Tensor, max_ctx: int, split_tokens: int = SPLIT_AUTO,
                 argmax: torch.Tensor | None = None, dev_err: torch.Tensor | None = None,
                 stream=None) -> None:
    """Paged absorbed decode of one layer for B slots; see include/k3mla.h.  split_tokens
    SPLIT_AUTO (0) cuts each slot by its own context (batch-invariant); a positive multiple of
    128 cuts every slot at that length."""
    B = q_abs.shape[0]
    n_pages, L = slab.shape[0], slab.shape[1]
    if workspace.dtype != torch.uint8 or not workspace.is_cuda:
        raise K3mlaError("workspace must be a CUDA uint8 tensor")
    lib = load()
    _check(lib.k3mla_paged_decode(
        _dev(q_abs, torch.bfloat16, (B, H, ROW), "q_abs"),
        _dev(slab, torch.bfloat16, (n_pages, L, PAGE, ROW), "slab"), n_pages, L, int(layer),
        _dev(block_table, torch.int32, None, "block_table"), block_table.shape[1],
        _dev(ctx_len, torch.int32, (B,), "ctx_len"),
        _dev(w_kv_b, torch.bfloat16, (H * (NOPE + V), LORA), "w_kv_b"), int(scale_bf16),
        _dev(out, torch.bfloat16, (B, H, V), "out"), _opt(argmax, torch.int32, (B, H), "argmax"),
        ctypes.c_void_p(workspace.data_ptr()), workspace.numel(), B, int(max_ctx), int(split_tokens),
        _opt(dev_err, torch.int32, (1,), "dev_err"), _stream(stream)), "k3mla_paged_decode")


def paged_decode_noalloc(q_abs: torch.Tensor, slab: torch.Tensor, layer: int, block_table: torch.Tensor,
                         ctx_len: torch.Tensor, w_kv_b: torch.Tensor, scale_bf16: int, out: torch.Tensor,
                         max_ctx: int, split_tokens: int = SPLIT_AUTO, argmax: torch.Tensor | None = None,
                         dev_err: torch.Tensor | None = None, stream=None) -> None:
    """paged_decode without a workspace argument, for callers that cannot allocate
    device memory where they decode: the split results go to the library's built-in
    16 MiB scratch (decode_workspace_bytes(B, max_ctx, split_tokens) must fit in it).
    Calls that overlap on the GPU share that scratch and race; see include/k3mla.h."""
    B = q_abs.shape[0]
    n_pages, L = slab.shape[0], slab.shape[1]
    lib = load()
    _check(lib.k3mla_paged_decode_noalloc(
        _dev(q_abs, torch.bfloat16, (B, H, ROW), "q_abs"),
        _dev(slab, torch.bfloat16, (n_pages, L, PAGE, ROW), "slab"), n_pages, L, int(layer),
        _dev(block_table, torch.int32, None, "block_table"), block_table.shape[1],
        _dev(ctx_len, torch.int32, (B,), "ctx_len"),
        _dev(w_kv_b, torch.bfloat16, (H * (NOPE + V), LORA), "w_kv_b"), int(scale_bf16),
        _dev(out, torch.bfloat16, (B, H, V), "out"), _opt(argmax, torch.int32, (B, H), "argmax"),
        B, int(max_ctx), int(split_tokens), _opt(dev_err, torch.int32, (1,), "dev_err"), _stream(stream)),
        "k3mla_paged_decode_noalloc")


def expanded_cache_bytes(n_pages: int) -> int:
    return int(load().k3mla_expanded_cache_bytes(int(n_pages)))


def expand_latent_cache(slab: torch.Tensor, layer: int, w_kv_b: torch.Tensor, xcache: torch.Tensor,
                        dev_err: torch.Tensor | None = None, stream=None) -> None:
    """The expanded-cache baseline's cache for one layer: xcache [n_pages, 64, 96, 320] bf16 (K nope |
    K rope | V per head) from the latent slab; see k3mla_expand_latent_cache."""
    n_pages, L = slab.shape[0], slab.shape[1]
    lib = load()
    _check(lib.k3mla_expand_latent_cache(
        _dev(slab, torch.bfloat16, (n_pages, L, PAGE, ROW), "slab"), n_pages, L, int(layer),
        _dev(w_kv_b, torch.bfloat16, (H * (NOPE + V), LORA), "w_kv_b"),
        _dev(xcache, torch.bfloat16, (n_pages, PAGE, H, NOPE + ROPE + V), "xcache"),
        _opt(dev_err, torch.int32, (1,), "dev_err"), _stream(stream)), "k3mla_expand_latent_cache")


def expanded_decode(q: torch.Tensor, xcache: torch.Tensor, block_table: torch.Tensor, ctx_len: torch.Tensor,
                    scale_bf16: int, out: torch.Tensor, max_ctx: int, dev_err: torch.Tensor | None = None,
                    stream=None) -> None:
    """Ordinary attention over the expanded cache: q [B,96,192] bf16 -> out [B,96,128] bf16."""
    B = q.shape[0]
    n_pages = xcache.shape[0]
    lib = load()
    _check(lib.k3mla_expanded_decode(
        _dev(q, torch.bfloat16, (B, H, NOPE + ROPE), "q"),
        _dev(xcache, torch.bfloat16, (n_pages, PAGE, H, NOPE + ROPE + V), "xcache"), n_pages,
        _dev(block_table, torch.int32, None, "block_table"), block_table.shape[1],
        _dev(ctx_len, torch.int32, (B,), "ctx_len"), ctypes.c_uint16(scale_bf16),
        _dev(out, torch.bfloat16, (B, H, V), "out"), B, int(max_ctx), _opt(dev_err, torch.int32, (1,), "dev_err"),
        _stream(stream)), "k3mla_expanded_decode")


def diag_decode_timeout(q_abs: torch.Tensor, slab: torch.Tensor, layer: int, block_table: torch.Tensor,
                        ctx_len: torch.Tensor, w_kv_b: torch.Tensor, scale_bf16: int, out: torch.Tensor,
                        workspace: torch.Tensor, max_ctx: int, split_tokens: int, withhold_page: int, wait_us: int,
                        dev_err: torch.Tensor, stream=None) -> None:
    """Diagnostic: paged_decode with page `withhold_page` of every split never loaded and every
    bounded wait limited to wait_us; see k3mla_diag_decode_timeout."""
    B = q_abs.shape[0]
    n_pages, L = slab.shape[0], slab.shape[1]
    lib = load()
    _check(lib.k3mla_diag_decode_timeout(
        _dev(q_abs, torch.bfloat16, (B, H, ROW), "q_abs"),
        _dev(slab, torch.bfloat16, (n_pages, L, PAGE, ROW), "slab"), n_pages, L, int(layer),
        _dev(block_table, torch.int32, None, "block_table"), block_table.shape[1],
        _dev(ctx_len, torch.int32, (B,), "ctx_len"),
        _dev(w_kv_b, torch.bfloat16, (H * (NOPE + V), LORA), "w_kv_b"), int(scale_bf16),
        _dev(out, torch.bfloat16, (B, H, V), "out"), None, ctypes.c_void_p(workspace.data_ptr()), workspace.numel(),
        B, int(max_ctx), int(split_tokens), int(withhold_page), ctypes.c_uint32(wait_us),
        _dev(dev_err, torch.int32, (1,), "dev_err"), _stream(stream)), "k3mla_diag_decode_timeout")


def diag_exact_exp(x: torch.Tensor, y: torch.Tensor, fast: torch.Tensor | None = None, stream=None) -> None:
    """Diagnostic: the exact-chain mode's exponential of every element of x (f32) into y; fast[i] = 1
    where the f32 evaluation decided; see k3mla_diag_exact_exp."""
    n = x.numel()
    lib = load()
    _check(lib.k3mla_diag_exact_exp(_dev(x, torch.float32, (n,), "x"), _dev(y, torch.float32, (n,), "y"),
                                    _opt(fast, torch.int32, (n,), "fast"), n, _stream(stream)),
           "k3mla_diag_exact_exp")


def diag_umma(mode: int, a: torch.Tensor, b: torch.Tensor, d: torch.Tensor, stream=None) -> None:
    lib = load()
    _check(lib.k3mla_diag_umma(int(mode), _dev(a, torch.bfloat16, None, "a"),
                               _dev(b, torch.bfloat16, (PAGE, ROW), "b"),
                               _dev(d, torch.float32, None, "d"), _stream(stream)), "k3mla_diag_umma")


class Pool:
    """Host free-list page allocator (k3mla_pool_*)."""

    def __init__(self, n_slots: int, max_ctx: int, n_pages: int = 0, shuffle_seed: int = 0):
        lib = load(build_if_needed=True)
        h = ctypes.c_void_p()
        _check(lib.k3mla_pool_create(n_pages, n_slots, max_ctx, shuffle_seed, ctypes.byref(h)),
               "k3mla_pool_create")
        self._h = h
        self.n_slots = n_slots
        self.max_ctx = max_ctx
        self.max_pages = lib.k3mla_pool_max_pages(h)
        self.n_pages = lib.k3mla_pool_n_pages(h)

    def ensure(self, slot: int, new_len: int) -> int:
        """Returns the status code (0 ok, negative K3MLA_E_*)."""
        return int(load().k3mla_pool_ensure(self._h, slot, new_len))

    def ensure_all(self, new_len) -> int:
        """ensure(b, new_len[b]) for b = 0 .. len-1 in one call (status of the first failure, or 0)."""
        a = np.ascontiguousarray(new_len, dtype=np.int32)
        return int(load().k3mla_pool_ensure_all(self._h, a.ctypes.data_as(ctypes.c_void_p), a.shape[0]))

    def release(self, slot: int) -> int:
        return int(load().k3mla_pool_release_slot(self._h, slot))

    def table(self) -> np.ndarray:
        ptr = load().k3mla_pool_host_table(self._h)
        return np.ctypeslib.as_array(ptr, shape=(self.n_slots, self.max_pages)).copy()

    def stats(self) -> tuple[int, int]:
        t, u = ctypes.c_int(), ctypes.c_int()
        _check(load().k3mla_pool_stats(self._h, ctypes.byref(t), ctypes.byref(u)), "k3mla_pool_stats")
        return t.value, u.value

    def share_prefix(self, dst_slot: int, src_slot: int, n_tokens: int) -> int:
        """Map src_slot's first ceil(n_tokens / 64) pages into the empty dst_slot (status code)."""
        return int(load().k3mla_pool_share_prefix(self._h, dst_slot, src_slot, n_tokens))

    def cow(self, slot: int, pos: int):
        """Before writing token `pos`: None if the slot owns the page (or a negative status code),
        else the (src_page, dst_page) copy to run first."""
        s, d = ctypes.c_int32(), ctypes.c_int32()
        rc = int(load().k3mla_pool_cow(self._h, slot, pos, ctypes.byref(s), ctypes.byref(d)))
        if rc == 1:
            return s.value, d.value
        return None if rc == 0 else rc

    def refs(self, page: int) -> int:
        return int(load().k3mla_pool_page_refs(self._h, page))

    def close(self):
        if self._h:
            load().k3mla_pool_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
