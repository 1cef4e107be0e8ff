"""prefill_dsa_indexer_gb300: the DSA sparse-attention layer on one GB300 GPU.

Python binding of libdsa (include/dsa.h).  Every function here only
marshals torch tensors into pointers and sizes and calls the C ABI of the
same name; all arithmetic runs in the library's CUDA kernels.  There is no
CPU fallback: importing the package on a machine without the built library
raises, and calling it with CPU tensors raises.

The layer (vLLM blog "Day-0 support for Kimi K3.1 Pro", section "Sparse
attention in K3.1 Pro"): indexer logits over every cached token -> exact
top-k (2,048) -> page-to-slot translation -> sparse absorbed MLA over the
selected tokens' latents.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

from . import inputs  # noqa: F401  (seeded synthetic inputs)

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdsa.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_WORKSPACE, ERR_TIMEOUT, ERR_BOUNDS, ERR_RANGE = \
    0, -1, -2, -3, -4, -5, -6, -7
KEY_FP8, KEY_MXFP4, LATENT_FP8, LATENT_NVFP4 = 1, 2, 3, 4
PAGE_SIZE = 64
INDEX_HEADS, INDEX_DIM, LATENT_DIM, VALUE_DIM = 32, 128, 576, 512
DEFAULT_SM_SCALE = 1.0 / math.sqrt(192.0)


class DsaError(RuntimeError):
    pass


class _Cache(ctypes.Structure):
    _fields_ = [("base", ctypes.c_void_p), ("format", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("num_pages", ctypes.c_int64), ("tensor_scale", ctypes.c_float)]


class _Rows(ctypes.Structure):
    _fields_ = [("block_table", ctypes.c_void_p), ("bt_stride", ctypes.c_int64), ("num_requests", ctypes.c_int32),
                ("row_req", ctypes.c_void_p), ("row_ctx", ctypes.c_void_p), ("num_rows", ctypes.c_int32),
                ("max_ctx", ctypes.c_int32), ("rows_per_group", ctypes.c_int32)]


_lib = None


def load_library(path: str | None = None):
    """Load libdsa.so; raises if it has not been built (no fallback)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise DsaError(f"libdsa.so not found at {p}: build it with prefill_dsa_indexer_gb300.build.build()")
    lib = ctypes.CDLL(p)
    P, I32, I64, F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    lib.dsa_version.restype = ctypes.c_int
    lib.dsa_status_string.restype = ctypes.c_char_p
    lib.dsa_status_string.argtypes = [ctypes.c_int]
    lib.dsa_indexer_logits.restype = ctypes.c_int
    lib.dsa_indexer_logits.argtypes = [ctypes.POINTER(_Cache), ctypes.POINTER(_Rows), P, P, P, I64, P, P]
    lib.dsa_topk.restype = ctypes.c_int
    lib.dsa_topk.argtypes = [P, I64, P, I32, I32, I32, P, P, P, ctypes.c_size_t, P]
    lib.dsa_topk_workspace_size.restype = ctypes.c_size_t
    lib.dsa_topk_workspace_size.argtypes = [I32, I32, I32]
    lib.dsa_page_to_slot.restype = ctypes.c_int
    lib.dsa_page_to_slot.argtypes = [ctypes.POINTER(_Rows), I64, P, I32, P, P, P]
    for name in ("dsa_sparse_mla_decode", "dsa_sparse_mla_prefill"):
        fn = getattr(lib, name)
        fn.restype = ctypes.c_int
        fn.argtypes = [ctypes.POINTER(_Cache), P, I32, P, I32, I32, F, P, P, P, P, ctypes.c_size_t, P]
    lib.dsa_sparse_mla_decode_noalloc.restype = ctypes.c_int
    lib.dsa_sparse_mla_decode_noalloc.argtypes = [ctypes.POINTER(_Cache), P, I32, P, I32, I32, F, P, P, P, P]
    lib.dsa_cache_insert.restype = ctypes.c_int
    lib.dsa_cache_insert.argtypes = [ctypes.POINTER(_Cache), ctypes.POINTER(_Cache), P, I32, P, P, P, P]
    lib.dsa_sparse_mla_workspace_size.restype = ctypes.c_size_t
    lib.dsa_sparse_mla_workspace_size.argtypes = [I32, I32, I32]
    lib.dsa_indexer_logits_hist.restype = ctypes.c_int
    lib.dsa_indexer_logits_hist.argtypes = [ctypes.POINTER(_Cache), ctypes.POINTER(_Rows), P, P, P, I64, P, P, P]
    lib.dsa_topk_hist.restype = ctypes.c_int
    lib.dsa_topk_hist.argtypes = [P, I64, P, I32, I32, I32, P, P, P, P]
    lib.dsa_indexer_topk.restype = ctypes.c_int
    lib.dsa_indexer_topk.argtypes = [ctypes.POINTER(_Cache), ctypes.POINTER(_Rows), P, P, I32, P, P, P,
                                     ctypes.c_size_t, P]
    lib.dsa_indexer_topk_workspace_size.restype = ctypes.c_size_t
    lib.dsa_indexer_topk_workspace_size.argtypes = [I32, I32]
    lib.dsa_topk_slots.restype = ctypes.c_int
    lib.dsa_topk_slots.argtypes = [P, I64, ctypes.POINTER(_Rows), I64, I32, P, P, P, P, ctypes.c_size_t, P]
    lib.dsa_selftest_wait_timeout.restype = ctypes.c_int
    lib.dsa_selftest_wait_timeout.argtypes = [P, P]
    lib.dsa_topk_slots_warm.restype = ctypes.c_int
    lib.dsa_topk_slots_warm.argtypes = [P, I64, ctypes.POINTER(_Rows), ctypes.POINTER(_Cache), I32, P, P, P, P,
                                        ctypes.c_size_t, P]
    lib.dsa_sparse_mla_decode_prepare.restype = ctypes.c_int
    lib.dsa_sparse_mla_decode_prepare.argtypes = [ctypes.POINTER(_Cache), P, I32, I32, I32, P, P, ctypes.c_size_t, P]
    lib.dsa_sparse_mla_decode_prepared.restype = ctypes.c_int
    lib.dsa_sparse_mla_decode_prepared.argtypes = [ctypes.POINTER(_Cache), P, I32, P, I32, I32, F, P, P, P, P,
                                                   ctypes.c_size_t, P]
    lib.dsa_msa_block_scores.restype = ctypes.c_int
    lib.dsa_msa_block_scores.argtypes = [P, I64, ctypes.POINTER(_Rows), P, P, I64, P, P]
    lib.dsa_msa_select.restype = ctypes.c_int
    lib.dsa_msa_select.argtypes = [P, I64, P, I32, I32, P, P, P]
    lib.dsa_msa_attention.restype = ctypes.c_int
    lib.dsa_msa_attention.argtypes = [P, I64, F, F, ctypes.POINTER(_Rows), P, F, I32, P, F, P, P, P,
                                      ctypes.c_size_t, P, P]
    lib.dsa_msa_attention_workspace_size.restype = ctypes.c_size_t
    lib.dsa_msa_attention_workspace_size.argtypes = [I32, I32]
    if path is None:
        _lib = lib
    return lib


EXPORTED = ("dsa_version", "dsa_status_string", "dsa_indexer_logits", "dsa_topk", "dsa_page_to_slot",
            "dsa_sparse_mla_decode", "dsa_sparse_mla_prefill", "dsa_sparse_mla_workspace_size",
            "dsa_sparse_mla_decode_noalloc", "dsa_cache_insert", "dsa_indexer_logits_hist", "dsa_topk_hist",
            "dsa_indexer_topk", "dsa_indexer_topk_workspace_size", "dsa_topk_slots", "dsa_topk_workspace_size",
            "dsa_sparse_mla_decode_prepare", "dsa_sparse_mla_decode_prepared", "dsa_msa_block_scores",
            "dsa_msa_select", "dsa_msa_attention", "dsa_msa_attention_workspace_size", "dsa_topk_slots_warm",
            "dsa_selftest_wait_timeout")
HIST_BINS = 65536
NOALLOC_MAX_ROWS = 8


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise DsaError("libdsa takes device tensors only")
    if not t.is_contiguous():
        raise DsaError("libdsa takes contiguous tensors only")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(rc: int, what: str):
    if rc != OK:
        msg = load_library().dsa_status_string(rc).decode()
        raise DsaError(f"{what}: {msg} ({rc})")


def new_status(device=None) -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=device or "cuda")


def check_status(status: torch.Tensor, what: str = "device status"):
    """Synchronise-free read of a device status word (the caller has synchronised)."""
    v = int(status.item())
    if v != OK:
        raise DsaError(f"{what}: {load_library().dsa_status_string(v).decode()} ({v})")


def _cache(pool: torch.Tensor, fmt: int, tensor_scale: float = 1.0) -> _Cache:
    return _Cache(_ptr(pool), fmt, PAGE_SIZE, pool.shape[0], tensor_scale)


def _rows(block_table, row_req, row_ctx, max_ctx, rows_per_group=1) -> _Rows:
    return _Rows(_ptr(block_table), block_table.shape[1], block_table.shape[0], _ptr(row_req), _ptr(row_ctx),
                 row_ctx.shape[0], int(max_ctx), int(rows_per_group))


def indexer_logits(index_pool, key_fmt, block_table, row_req, row_ctx, max_ctx, q_idx, head_w, rows_per_group=1,
                   logits=None, status=None, stream=None):
    """dsa_indexer_logits: fp32 logits [R, max_ctx] (t >= row_ctx[r] untouched)."""
    R = row_ctx.shape[0]
    if logits is None:
        logits = torch.empty((R, max(int(max_ctx), 1)), dtype=torch.float32, device=q_idx.device)
    c, r = _cache(index_pool, key_fmt), _rows(block_table, row_req, row_ctx, max_ctx, rows_per_group)
    rc = load_library().dsa_indexer_logits(ctypes.byref(c), ctypes.byref(r), _ptr(q_idx), _ptr(head_w),
                                           _ptr(logits), logits.stride(0), _ptr(status), _stream(stream))
    _check(rc, "dsa_indexer_logits")
    return logits


def topk_workspace_size(num_rows: int, max_ctx: int, k: int = 2048) -> int:
    """dsa_topk_workspace_size: bytes of the histogram top-k's workspace (0: the shape needs none)."""
    return int(load_library().dsa_topk_workspace_size(num_rows, max_ctx, k))


def _ws(workspace):
    return (_ptr(workspace), workspace.numel() * workspace.element_size()) if workspace is not None else (None, 0)


def topk(logits, row_ctx, max_ctx, k=2048, out=None, status=None, stream=None, workspace=None):
    """dsa_topk: int32 [R, k] selected positions, ascending, -1 padded (`workspace`: optional, see
    topk_workspace_size)."""
    R = row_ctx.shape[0]
    if out is None:
        out = torch.empty((R, k), dtype=torch.int32, device=logits.device)
    wp, wb = _ws(workspace)
    rc = load_library().dsa_topk(_ptr(logits), logits.stride(0), _ptr(row_ctx), R, int(max_ctx), int(k), _ptr(out),
                                 _ptr(status), wp, wb, _stream(stream))
    _check(rc, "dsa_topk")
    return out


def new_hist(num_rows: int, device=None) -> torch.Tensor:
    """A zeroed per-row histogram for indexer_logits_hist / topk_hist (uint32 bits in int32)."""
    return torch.zeros((num_rows, HIST_BINS), dtype=torch.int32, device=device or "cuda")


def indexer_logits_hist(index_pool, key_fmt, block_table, row_req, row_ctx, max_ctx, q_idx, head_w, hist,
                        rows_per_group=1, logits=None, status=None, stream=None):
    """dsa_indexer_logits_hist: indexer_logits that also adds every logit to the zeroed histogram `hist`."""
    R = row_ctx.shape[0]
    if logits is None:
        logits = torch.empty((R, max(int(max_ctx), 1)), dtype=torch.float32, device=q_idx.device)
    c, r = _cache(index_pool, key_fmt), _rows(block_table, row_req, row_ctx, max_ctx, rows_per_group)
    rc = load_library().dsa_indexer_logits_hist(ctypes.byref(c), ctypes.byref(r), _ptr(q_idx), _ptr(head_w),
                                                _ptr(logits), logits.stride(0), _ptr(hist), _ptr(status),
                                                _stream(stream))
    _check(rc, "dsa_indexer_logits_hist")
    return logits


def topk_hist(logits, row_ctx, max_ctx, hist, k=2048, out=None, status=None, stream=None):
    """dsa_topk_hist: topk starting from the scorer's histogram of these logits (left zeroed)."""
    R = row_ctx.shape[0]
    if out is None:
        out = torch.empty((R, k), dtype=torch.int32, device=logits.device)
    rc = load_library().dsa_topk_hist(_ptr(logits), logits.stride(0), _ptr(row_ctx), R, int(max_ctx), int(k),
                                      _ptr(hist), _ptr(out), _ptr(status), _stream(stream))
    _check(rc, "dsa_topk_hist")
    return out


def indexer_topk_workspace_size(num_rows: int, max_ctx: int) -> int:
    return int(load_library().dsa_indexer_topk_workspace_size(int(num_rows), int(max_ctx)))


def indexer_topk(index_pool, key_fmt, block_table, row_req, row_ctx, max_ctx, q_idx, head_w, workspace, k=2048,
                 rows_per_group=1, out=None, status=None, stream=None):
    """dsa_indexer_topk: scorer + top-k in one call; `workspace` (uint8, zeroed before its first use)."""
    R = row_ctx.shape[0]
    if out is None:
        out = torch.empty((R, k), dtype=torch.int32, device=q_idx.device)
    c, r = _cache(index_pool, key_fmt), _rows(block_table, row_req, row_ctx, max_ctx, rows_per_group)
    rc = load_library().dsa_indexer_topk(ctypes.byref(c), ctypes.byref(r), _ptr(q_idx), _ptr(head_w), int(k),
                                         _ptr(out), _ptr(status), _ptr(workspace), workspace.numel(),
                                         _stream(stream))
    _check(rc, "dsa_indexer_topk")
    return out


def topk_slots(logits, block_table, row_req, row_ctx, max_ctx, pool_pages, k=2048, out=None, slots=None,
               status=None, stream=None, workspace=None):
    """dsa_topk_slots: (idx int32 [R, k], slots int32 [R, k]) — top-k with the page -> slot translation."""
    R = row_ctx.shape[0]
    if out is None:
        out = torch.empty((R, k), dtype=torch.int32, device=logits.device)
    if slots is None:
        slots = torch.empty((R, k), dtype=torch.int32, device=logits.device)
    r = _rows(block_table, row_req, row_ctx, max_ctx)
    wp, wb = _ws(workspace)
    rc = load_library().dsa_topk_slots(_ptr(logits), logits.stride(0), ctypes.byref(r), int(pool_pages), int(k),
                                       _ptr(out), _ptr(slots), _ptr(status), wp, wb, _stream(stream))
    _check(rc, "dsa_topk_slots")
    return out, slots


def topk_slots_warm(logits, block_table, row_req, row_ctx, max_ctx, lat_pool, lat_fmt, k=2048, out=None,
                    slots=None, status=None, stream=None, workspace=None):
    """dsa_topk_slots_warm: topk_slots whose output pass also prefetches the selected FP8 latents into L2."""
    R = row_ctx.shape[0]
    if out is None:
        out = torch.empty((R, k), dtype=torch.int32, device=logits.device)
    if slots is None:
        slots = torch.empty((R, k), dtype=torch.int32, device=logits.device)
    r = _rows(block_table, row_req, row_ctx, max_ctx)
    c = _cache(lat_pool, lat_fmt)
    wp, wb = _ws(workspace)
    rc = load_library().dsa_topk_slots_warm(_ptr(logits), logits.stride(0), ctypes.byref(r), ctypes.byref(c), int(k),
                                            _ptr(out), _ptr(slots), _ptr(status), wp, wb, _stream(stream))
    _check(rc, "dsa_topk_slots_warm")
    return out, slots


def page_to_slot(block_table, row_req, row_ctx, max_ctx, pool_pages, idx, out=None, status=None, stream=None):
    """dsa_page_to_slot: int32 [R, k] physical slots (-1 stays -1)."""
    if out is None:
        out = torch.empty_like(idx)
    r = _rows(block_table, row_req, row_ctx, max_ctx)
    rc = load_library().dsa_page_to_slot(ctypes.byref(r), int(pool_pages), _ptr(idx), idx.shape[1], _ptr(out),
                                         _ptr(status), _stream(stream))
    _check(rc, "dsa_page_to_slot")
    return out


def cache_insert(idx_pool, key_fmt, lat_pool, lat_fmt, tensor_scale, slots, index_keys, latents, status=None,
                 stream=None):
    """dsa_cache_insert: quantise new tokens (bf16 [n,128] keys, [n,576] latents) into the pools in place."""
    ci, cl = _cache(idx_pool, key_fmt), _cache(lat_pool, lat_fmt, tensor_scale)
    rc = load_library().dsa_cache_insert(ctypes.byref(ci), ctypes.byref(cl), _ptr(slots), slots.shape[0],
                                         _ptr(index_keys), _ptr(latents), _ptr(status), _stream(stream))
    _check(rc, "dsa_cache_insert")


def sparse_mla_workspace_size(num_rows, num_heads, k) -> int:
    return int(load_library().dsa_sparse_mla_workspace_size(num_rows, num_heads, k))


def _mla(name, lat_pool, lat_fmt, tensor_scale, q, slots, sm_scale, out, lse, workspace, status, stream):
    R, H, _ = q.shape
    k = slots.shape[1]
    if out is None:
        out = torch.empty((R, H, VALUE_DIM), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((R, H), dtype=torch.float32, device=q.device)
    ws_ptr, ws_bytes = None, 0
    if name in ("dsa_sparse_mla_decode", "dsa_sparse_mla_decode_prepared"):
        need = sparse_mla_workspace_size(R, H, k)
        if workspace is None and need:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        if workspace is not None:
            ws_ptr, ws_bytes = _ptr(workspace), workspace.numel() * workspace.element_size()
    c = _cache(lat_pool, lat_fmt, tensor_scale)
    rc = getattr(load_library(), name)(ctypes.byref(c), _ptr(q), H, _ptr(slots), R, k, float(sm_scale), _ptr(out),
                                       _ptr(lse), _ptr(status), ws_ptr, ws_bytes, _stream(stream))
    _check(rc, name)
    return out, lse


def sparse_mla_decode(lat_pool, lat_fmt, tensor_scale, q, slots, sm_scale=DEFAULT_SM_SCALE, out=None, lse=None,
                      workspace=None, status=None, stream=None):
    """dsa_sparse_mla_decode: (out fp32 [R, H, 512], lse fp32 [R, H]); q is bf16 (or its int16 bits)."""
    return _mla("dsa_sparse_mla_decode", lat_pool, lat_fmt, tensor_scale, q, slots, sm_scale, out, lse, workspace,
                status, stream)


def sparse_mla_decode_noalloc(lat_pool, lat_fmt, tensor_scale, q, slots, out, lse, sm_scale=DEFAULT_SM_SCALE,
                              status=None, stream=None):
    """dsa_sparse_mla_decode_noalloc: as sparse_mla_decode, with the split-K scratch kept in the
    library's own fixed device array instead of a workspace (for callers that cannot allocate;
    at most NOALLOC_MAX_ROWS rows).  `out` and `lse` must be preallocated."""
    R, H, _ = q.shape
    c = _cache(lat_pool, lat_fmt, tensor_scale)
    rc = load_library().dsa_sparse_mla_decode_noalloc(ctypes.byref(c), _ptr(q), H, _ptr(slots), R, slots.shape[1],
                                                      float(sm_scale), _ptr(out), _ptr(lse), _ptr(status),
                                                      _stream(stream))
    _check(rc, "dsa_sparse_mla_decode_noalloc")
    return out, lse


def sparse_mla_decode_prepare(lat_pool, lat_fmt, tensor_scale, q, k, workspace, status=None, stream=None):
    """dsa_sparse_mla_decode_prepare: the rows' queries into the workspace in the kernel's layout."""
    R, H, _ = q.shape
    c = _cache(lat_pool, lat_fmt, tensor_scale)
    rc = load_library().dsa_sparse_mla_decode_prepare(ctypes.byref(c), _ptr(q), H, R, int(k), _ptr(status),
                                                      _ptr(workspace), workspace.numel() * workspace.element_size(),
                                                      _stream(stream))
    _check(rc, "dsa_sparse_mla_decode_prepare")


def sparse_mla_decode_prepared(lat_pool, lat_fmt, tensor_scale, q, slots, sm_scale=DEFAULT_SM_SCALE, out=None,
                               lse=None, workspace=None, status=None, stream=None):
    """dsa_sparse_mla_decode_prepared: sparse_mla_decode after sparse_mla_decode_prepare on `workspace`."""
    return _mla("dsa_sparse_mla_decode_prepared", lat_pool, lat_fmt, tensor_scale, q, slots, sm_scale, out, lse,
                workspace, status, stream)


def sparse_mla_prefill(lat_pool, lat_fmt, tensor_scale, q, slots, sm_scale=DEFAULT_SM_SCALE, out=None, lse=None,
                       status=None, stream=None):
    return _mla("dsa_sparse_mla_prefill", lat_pool, lat_fmt, tensor_scale, q, slots, sm_scale, out, lse, None,
                status, stream)


def selftest_wait_timeout(status, stream=None):
    """dsa_selftest_wait_timeout: a kernel whose bounded wait runs out; status gets DSA_ERR_TIMEOUT."""
    _check(load_library().dsa_selftest_wait_timeout(_ptr(status), _stream(stream)), "dsa_selftest_wait_timeout")


# ------------------------------------------------------------------ MSA block-sparse variant
MSA_PAGE, MSA_GROUPS, MSA_BLOCKS = 128, 4, 16


def msa_block_scores(idx_pool, block_table, row_req, row_ctx, max_ctx, q_idx, rows_per_group=1, scores=None,
                     status=None, stream=None):
    """dsa_msa_block_scores: fp32 [R, 4, ceil(max_ctx / 128)] block-max index scores."""
    R = row_ctx.shape[0]
    nb = max((int(max_ctx) + MSA_PAGE - 1) // MSA_PAGE, 1)
    if scores is None:
        scores = torch.empty((R, MSA_GROUPS, nb), dtype=torch.float32, device=q_idx.device)
    r = _rows(block_table, row_req, row_ctx, max_ctx, rows_per_group)
    rc = load_library().dsa_msa_block_scores(_ptr(idx_pool), idx_pool.shape[0], ctypes.byref(r), _ptr(q_idx),
                                             _ptr(scores), scores.shape[-1], _ptr(status), _stream(stream))
    _check(rc, "dsa_msa_block_scores")
    return scores


def msa_select(scores, row_ctx, max_ctx, blocks=None, status=None, stream=None):
    """dsa_msa_select: int32 [R, 4, 16] selected blocks, ascending, -1 padded."""
    R = row_ctx.shape[0]
    if blocks is None:
        blocks = torch.empty((R, MSA_GROUPS, MSA_BLOCKS), dtype=torch.int32, device=scores.device)
    rc = load_library().dsa_msa_select(_ptr(scores), scores.shape[-1], _ptr(row_ctx), R, int(max_ctx), _ptr(blocks),
                                       _ptr(status), _stream(stream))
    _check(rc, "dsa_msa_select")
    return blocks


def msa_attention_workspace_size(num_rows, heads_per_group) -> int:
    return int(load_library().dsa_msa_attention_workspace_size(int(num_rows), int(heads_per_group)))


def msa_attention(kv_pool, k_scale, v_scale, block_table, row_req, row_ctx, max_ctx, q, q_scale, blocks, sm_scale,
                  out=None, lse=None, workspace=None, status=None, stream=None):
    """dsa_msa_attention: (out fp32 [R, H, 128], lse fp32 [R, H]); q is e4m3 codes [R, H, 128]."""
    R, H, _ = q.shape
    hpg = H // MSA_GROUPS
    if out is None:
        out = torch.empty((R, H, 128), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((R, H), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = torch.empty(max(msa_attention_workspace_size(R, hpg), 1), dtype=torch.uint8, device=q.device)
    r = _rows(block_table, row_req, row_ctx, max_ctx)
    rc = load_library().dsa_msa_attention(_ptr(kv_pool), kv_pool.shape[0], float(k_scale), float(v_scale),
                                          ctypes.byref(r), _ptr(q), float(q_scale), hpg, _ptr(blocks),
                                          float(sm_scale), _ptr(out), _ptr(lse), _ptr(workspace),
                                          workspace.numel() * workspace.element_size(), _ptr(status),
                                          _stream(stream))
    _check(rc, "dsa_msa_attention")
    return out, lse


class Layer:
    """One DSA layer invocation over resident caches: indexer -> top-k -> slots -> sparse MLA.

    Buffers are allocated once per shape and reused, so repeated calls (and
    CUDA-graph capture of `run`) allocate nothing.
    """

    def __init__(self, idx_pool, key_fmt, lat_pool, lat_fmt, tensor_scale, block_table, max_ctx, num_rows,
                 num_heads=96, k=2048, rows_per_group=1, prefill=False, sm_scale=DEFAULT_SM_SCALE, device="cuda",
                 single_pass=False):
        self.idx_pool, self.key_fmt = idx_pool, key_fmt
        self.lat_pool, self.lat_fmt, self.tensor_scale = lat_pool, lat_fmt, float(tensor_scale)
        self.block_table, self.max_ctx, self.k = block_table, int(max_ctx), int(k)
        self.rows_per_group, self.prefill, self.sm_scale = rows_per_group, prefill, sm_scale
        R, H = int(num_rows), int(num_heads)
        self.logits = torch.empty((R, max(self.max_ctx, 1)), dtype=torch.float32, device=device)
        self.idx = torch.empty((R, self.k), dtype=torch.int32, device=device)
        self.slots = torch.empty((R, self.k), dtype=torch.int32, device=device)
        # outputs and log-sum-exps in one buffer, so one copy moves a step's results
        self.outputs = torch.empty(R * H * (VALUE_DIM + 1), dtype=torch.float32, device=device)
        self.out = self.outputs[:R * H * VALUE_DIM].view(R, H, VALUE_DIM)
        self.lse = self.outputs[R * H * VALUE_DIM:].view(R, H)
        need = 0 if prefill else sparse_mla_workspace_size(R, H, self.k)
        self.workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
        # the histogram top-k's counts and candidates (few long rows; none otherwise)
        tk = topk_workspace_size(R, self.max_ctx, self.k)
        self.topk_workspace = torch.empty(tk, dtype=torch.uint8, device=device) if tk > 0 else None
        self.status = new_status(device)
        # single pass: the scorer builds each row's histogram and the top-k starts from it (opt-in:
        # on one GB300 the scorer's histogram atomics cost more than the selection saves)
        self.single_pass = single_pass
        self.hist = new_hist(R, device) if single_pass else None

    def score(self, row_req, row_ctx, q_idx, head_w, stream=None):
        """Indexer logits (and, single pass, their histogram)."""
        if self.single_pass:
            indexer_logits_hist(self.idx_pool, self.key_fmt, self.block_table, row_req, row_ctx, self.max_ctx, q_idx,
                                head_w, self.hist, self.rows_per_group, logits=self.logits, status=self.status,
                                stream=stream)
        else:
            indexer_logits(self.idx_pool, self.key_fmt, self.block_table, row_req, row_ctx, self.max_ctx, q_idx,
                           head_w, self.rows_per_group, logits=self.logits, status=self.status, stream=stream)

    def select(self, row_req, row_ctx, q_mla, stream=None, prepared=False):
        """Top-k, page -> slot and sparse MLA over the scored logits (`prepared`: prepare() ran already)."""
        self.select_tokens(row_req, row_ctx, stream=stream)
        return self.attend(q_mla, stream=stream, prepared=prepared)

    def select_tokens(self, row_req, row_ctx, stream=None):
        """Top-k and page -> slot over the scored logits (into self.idx, self.slots)."""
        if self.single_pass:
            topk_hist(self.logits, row_ctx, self.max_ctx, self.hist, self.k, out=self.idx, status=self.status,
                      stream=stream)
            page_to_slot(self.block_table, row_req, row_ctx, self.max_ctx, self.lat_pool.shape[0], self.idx,
                         out=self.slots, status=self.status, stream=stream)
        elif not self.prefill:  # decode: top-k with page -> slot, warming L2 with the chosen latents
            topk_slots_warm(self.logits, self.block_table, row_req, row_ctx, self.max_ctx, self.lat_pool,
                            self.lat_fmt, self.k, out=self.idx, slots=self.slots, status=self.status, stream=stream,
                            workspace=self.topk_workspace)
        else:  # top-k with the page -> slot translation in its output pass
            topk_slots(self.logits, self.block_table, row_req, row_ctx, self.max_ctx, self.lat_pool.shape[0], self.k,
                       out=self.idx, slots=self.slots, status=self.status, stream=stream,
                       workspace=self.topk_workspace)

    def attend(self, q_mla, stream=None, prepared=False):
        """Sparse MLA over self.slots (`prepared`: prepare() ran already for these queries)."""
        if self.prefill:
            sparse_mla_prefill(self.lat_pool, self.lat_fmt, self.tensor_scale, q_mla, self.slots, self.sm_scale,
                               out=self.out, lse=self.lse, status=self.status, stream=stream)
        elif prepared:
            sparse_mla_decode_prepared(self.lat_pool, self.lat_fmt, self.tensor_scale, q_mla, self.slots,
                                       self.sm_scale, out=self.out, lse=self.lse, workspace=self.workspace,
                                       status=self.status, stream=stream)
        else:
            sparse_mla_decode(self.lat_pool, self.lat_fmt, self.tensor_scale, q_mla, self.slots, self.sm_scale,
                              out=self.out, lse=self.lse, workspace=self.workspace, status=self.status,
                              stream=stream)
        return self.out, self.lse

    def prepare(self, q_mla, stream=None):
        """Decode query conversion (independent of the scorer and the top-k; may run beside the top-k,
        which leaves most SMs free, and must be ordered before attend(prepared=True))."""
        if not self.prefill:
            sparse_mla_decode_prepare(self.lat_pool, self.lat_fmt, self.tensor_scale, q_mla, self.k, self.workspace,
                                      status=self.status, stream=stream)

    def run(self, row_req, row_ctx, q_idx, head_w, q_mla, stream=None):
        self.score(row_req, row_ctx, q_idx, head_w, stream=stream)
        return self.select(row_req, row_ctx, q_mla, stream=stream)
