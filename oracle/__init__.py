"""CPU oracle for the DSA layer hot path (test infrastructure only).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports it and shares no code with it.

The arithmetic lives in ``dsa_oracle.c`` (plain C, double precision, OpenMP
over rows).  This module compiles it with gcc on first use and exposes thin
numpy wrappers.  Source of every definition: the vLLM blog post "Day-0
support for Kimi K3.1 Pro", section "Sparse attention in K3.1 Pro", and for
the block-sparse variant the vLLM blog post "Day-0 support for
MiniMax-M3.1-Flash", section "MSA primer"; the formulas are restated in
``dsa_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dsa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

KEY_FP8, KEY_MXFP4, LATENT_FP8, LATENT_NVFP4 = 1, 2, 3, 4
OK, ERR_ARG, ERR_BOUNDS = 0, -1, -6


def build(force: bool = False, extra_flags: tuple[str, ...] = (), out: str | None = None) -> str:
    """Compile dsa_oracle.c into a shared library (gcc, -O2, OpenMP)."""
    out = out or _LIB_PATH
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    tmp = out + ".tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-fopenmp", *extra_flags, _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def load(path: str | None = None):
    global _lib
    with _lock:
        if path is None and _lib is not None:
            return _lib
        lib = ctypes.CDLL(path or build())
        P, I64, I32, D = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
        lib.oracle_e4m3_decode.restype = D
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e2m1_decode.restype = D
        lib.oracle_e2m1_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e8m0_decode.restype = D
        lib.oracle_e8m0_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_bf16_decode.restype = D
        lib.oracle_bf16_decode.argtypes = [ctypes.c_uint16]
        lib.oracle_index_page_bytes.restype = I64
        lib.oracle_index_page_bytes.argtypes = [I32]
        lib.oracle_latent_page_bytes.restype = I64
        lib.oracle_latent_page_bytes.argtypes = [I32]
        lib.oracle_indexer_logits.restype = I32
        lib.oracle_indexer_logits.argtypes = [P, I32, I64, P, I64, P, P, I32, P, P, P, I64]
        lib.oracle_topk_f32.restype = I32
        lib.oracle_topk_f32.argtypes = [P, I64, P, I32, I32, P]
        lib.oracle_topk_f64.restype = I32
        lib.oracle_topk_f64.argtypes = [P, I64, P, I32, I32, P]
        lib.oracle_page_to_slot.restype = I32
        lib.oracle_page_to_slot.argtypes = [P, I64, P, I32, P, I32, P]
        lib.oracle_sparse_mla.restype = I32
        lib.oracle_sparse_mla.argtypes = [P, I32, I64, D, P, I32, P, I32, I32, D, P, P]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_e2m1_encode.restype = ctypes.c_uint8
        lib.oracle_e2m1_encode.argtypes = [ctypes.c_float]
        lib.oracle_cache_insert.restype = I32
        lib.oracle_cache_insert.argtypes = [P, I32, P, I32, ctypes.c_float, I64, P, I32, P, P]
        lib.oracle_msa_index_page_bytes.restype = I64
        lib.oracle_msa_index_page_bytes.argtypes = []
        lib.oracle_msa_kv_page_bytes.restype = I64
        lib.oracle_msa_kv_page_bytes.argtypes = []
        lib.oracle_msa_block_scores.restype = I32
        lib.oracle_msa_block_scores.argtypes = [P, I64, P, I64, P, P, I32, P, P, I64]
        lib.oracle_msa_select_f64.restype = I32
        lib.oracle_msa_select_f64.argtypes = [P, I64, P, I32, P]
        lib.oracle_msa_select_f32.restype = I32
        lib.oracle_msa_select_f32.argtypes = [P, I64, P, I32, P]
        lib.oracle_msa_attention.restype = I32
        lib.oracle_msa_attention.argtypes = [P, I64, D, D, P, I64, P, P, I32, P, D, I32, P, D, P, P]
        lib.oracle_num_threads.restype = I32
        lib.oracle_set_num_threads.argtypes = [I32]
        if path is None:
            _lib = lib
        return lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


def e4m3_decode(code: int, lib=None) -> float:
    return (lib or load()).oracle_e4m3_decode(code)


def e2m1_decode(nib: int, lib=None) -> float:
    return (lib or load()).oracle_e2m1_decode(nib)


def e8m0_decode(code: int, lib=None) -> float:
    return (lib or load()).oracle_e8m0_decode(code)


def bf16_decode(bits: int, lib=None) -> float:
    return (lib or load()).oracle_bf16_decode(bits)


def index_page_bytes(fmt: int, lib=None) -> int:
    return (lib or load()).oracle_index_page_bytes(fmt)


def latent_page_bytes(fmt: int, lib=None) -> int:
    return (lib or load()).oracle_latent_page_bytes(fmt)


def indexer_logits(idx_pool, fmt, block_table, row_req, row_ctx, q_idx, w, lib=None):
    """Return float64 logits [R, max(row_ctx)] (NaN where t >= row_ctx[r])."""
    lib = lib or load()
    pool = _c(idx_pool, np.uint8)
    bt = _c(block_table, np.int32)
    rq, rc = _c(row_req, np.int32), _c(row_ctx, np.int32)
    q, wv = _c(q_idx, np.uint8), _c(w, np.float32)
    R = rc.shape[0]
    width = max(int(rc.max()) if R else 0, 1)
    out = np.full((R, width), np.nan, dtype=np.float64)
    num_pages = pool.size // index_page_bytes(fmt, lib)
    rcode = lib.oracle_indexer_logits(_p(pool), fmt, num_pages, _p(bt), bt.shape[1], _p(rq), _p(rc), R,
                                      _p(q), _p(wv), _p(out), width)
    if rcode != OK:
        raise ValueError(f"oracle_indexer_logits failed: {rcode}")
    return out


def topk_f32(logits, row_ctx, k, lib=None):
    lib = lib or load()
    lg, rc = _c(logits, np.float32), _c(row_ctx, np.int32)
    R = rc.shape[0]
    out = np.empty((R, k), dtype=np.int32)
    rcode = lib.oracle_topk_f32(_p(lg), lg.shape[1], _p(rc), R, k, _p(out))
    if rcode != OK:
        raise ValueError(f"oracle_topk_f32 failed: {rcode}")
    return out


def topk_f64(logits, row_ctx, k, lib=None):
    lib = lib or load()
    lg, rc = _c(logits, np.float64), _c(row_ctx, np.int32)
    R = rc.shape[0]
    out = np.empty((R, k), dtype=np.int32)
    rcode = lib.oracle_topk_f64(_p(lg), lg.shape[1], _p(rc), R, k, _p(out))
    if rcode != OK:
        raise ValueError(f"oracle_topk_f64 failed: {rcode}")
    return out


def page_to_slot(block_table, row_req, idx, lib=None):
    lib = lib or load()
    bt, rq, ix = _c(block_table, np.int32), _c(row_req, np.int32), _c(idx, np.int32)
    R, k = ix.shape
    out = np.empty((R, k), dtype=np.int32)
    lib.oracle_page_to_slot(_p(bt), bt.shape[1], _p(rq), R, _p(ix), k, _p(out))
    return out


def sparse_mla(lat_pool, fmt, tensor_scale, q_bf16_bits, slots, sm_scale, lib=None):
    """q_bf16_bits: uint16 [R, H, 576]; slots: int32 [R, k].
    Returns (out float64 [R, H, 512], lse float64 [R, H])."""
    lib = lib or load()
    pool = _c(lat_pool, np.uint8)
    q = _c(q_bf16_bits, np.uint16)
    sl = _c(slots, np.int32)
    R, H, _ = q.shape
    k = sl.shape[1]
    out = np.empty((R, H, 512), dtype=np.float64)
    lse = np.empty((R, H), dtype=np.float64)
    num_pages = pool.size // latent_page_bytes(fmt, lib)
    rcode = lib.oracle_sparse_mla(_p(pool), fmt, num_pages, float(tensor_scale), _p(q), H, _p(sl), R, k,
                                  float(sm_scale), _p(out), _p(lse))
    if rcode != OK:
        raise ValueError(f"oracle_sparse_mla failed: {rcode}")
    return out, lse


def e4m3_encode(x: float, lib=None) -> int:
    return (lib or load()).oracle_e4m3_encode(x)


def e2m1_encode(x: float, lib=None) -> int:
    return (lib or load()).oracle_e2m1_encode(x)


def cache_insert(idx_pool, key_fmt, lat_pool, lat_fmt, tensor_scale, slots, keys_bf16_bits, lat_bf16_bits, lib=None):
    """Write new tokens into copies of the pools; returns (idx_pool, lat_pool) numpy copies."""
    lib = lib or load()
    ip = np.array(idx_pool, dtype=np.uint8, copy=True, order="C")
    lp = np.array(lat_pool, dtype=np.uint8, copy=True, order="C")
    sl = _c(slots, np.int32)
    k = _c(keys_bf16_bits, np.uint16)
    x = _c(lat_bf16_bits, np.uint16)
    num_pages = ip.shape[0] if ip.ndim == 2 else ip.size // index_page_bytes(key_fmt, lib)
    rc = lib.oracle_cache_insert(_p(ip), key_fmt, _p(lp), lat_fmt, float(tensor_scale), num_pages, _p(sl),
                                 sl.shape[0], _p(k), _p(x))
    if rc != OK:
        raise ValueError(f"oracle_cache_insert failed: {rc}")
    return ip, lp


# ------------------------------------------------------------------ MSA

MSA_GROUPS, MSA_BLOCKS, MSA_PAGE = 4, 16, 128


def msa_block_scores(idx_pool, block_table, row_req, row_ctx, q_idx, lib=None):
    """float64 block scores [R, 4, ceil(max(row_ctx) / 128)] (NaN past a row's blocks)."""
    lib = lib or load()
    pool = _c(idx_pool, np.uint8)
    bt, rq, rc = _c(block_table, np.int32), _c(row_req, np.int32), _c(row_ctx, np.int32)
    q = _c(q_idx, np.uint8)
    R = rc.shape[0]
    width = max((int(rc.max()) + MSA_PAGE - 1) // MSA_PAGE if R else 0, 1)
    out = np.full((R, MSA_GROUPS, width), np.nan, dtype=np.float64)
    num_pages = pool.size // lib.oracle_msa_index_page_bytes()
    rcode = lib.oracle_msa_block_scores(_p(pool), num_pages, _p(bt), bt.shape[1], _p(rq), _p(rc), R, _p(q),
                                        _p(out), width)
    if rcode != OK:
        raise ValueError(f"oracle_msa_block_scores failed: {rcode}")
    return out


def msa_select(scores, row_ctx, lib=None):
    """Selected blocks int32 [R, 4, 16] from block scores [R, 4, W] (float32: decided in fp32)."""
    lib = lib or load()
    sc = np.asarray(scores)
    fn = lib.oracle_msa_select_f32 if sc.dtype == np.float32 else lib.oracle_msa_select_f64
    sc = _c(sc, np.float32 if sc.dtype == np.float32 else np.float64)
    rc = _c(row_ctx, np.int32)
    R = rc.shape[0]
    out = np.empty((R, MSA_GROUPS, MSA_BLOCKS), dtype=np.int32)
    fn(_p(sc), sc.shape[-1], _p(rc), R, _p(out))
    return out


def msa_attention(kv_pool, k_scale, v_scale, block_table, row_req, row_ctx, q_codes, q_scale, blocks, sm_scale,
                  lib=None):
    """q_codes: uint8 e4m3 [R, 4 * hpg, 128] (times q_scale); blocks: int32 [R, 4, 16].
    Returns (out float64 [R, H, 128], lse float64 [R, H])."""
    lib = lib or load()
    pool = _c(kv_pool, np.uint8)
    bt, rq, rc = _c(block_table, np.int32), _c(row_req, np.int32), _c(row_ctx, np.int32)
    q, bl = _c(q_codes, np.uint8), _c(blocks, np.int32)
    R, H, _ = q.shape
    out = np.empty((R, H, 128), dtype=np.float64)
    lse = np.empty((R, H), dtype=np.float64)
    num_pages = pool.size // lib.oracle_msa_kv_page_bytes()
    rcode = lib.oracle_msa_attention(_p(pool), num_pages, float(k_scale), float(v_scale), _p(bt), bt.shape[1],
                                     _p(rq), _p(rc), R, _p(q), float(q_scale), H // MSA_GROUPS, _p(bl),
                                     float(sm_scale), _p(out),
                                     _p(lse))
    if rcode != OK:
        raise ValueError(f"oracle_msa_attention failed: {rcode}")
    return out, lse


def num_threads(lib=None) -> int:
    return (lib or load()).oracle_num_threads()
