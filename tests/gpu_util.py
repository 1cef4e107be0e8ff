"""Helpers shared by the GPU parity tests: run the CUDA path through the
C-ABI binding and compare with the oracle on the same seeded bytes."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
import prefill_dsa_indexer_gb300 as P
from prefill_dsa_indexer_gb300 import inputs as I
from tests import oracle_pins as pins

SM_SCALE = 1.0 / math.sqrt(192.0)
ORACLE_FMT = {I.KEY_FP8: oracle.KEY_FP8, I.KEY_MXFP4: oracle.KEY_MXFP4, I.LATENT_FP8: oracle.LATENT_FP8,
              I.LATENT_NVFP4: oracle.LATENT_NVFP4}


def gpu_inputs(wl: I.Workload, where: str = "cpu") -> I.Inputs:
    """Generate on `where` (cpu for small cases), return a cuda copy."""
    inp = I.make_inputs(wl, device=where)
    return inp.to("cuda") if where == "cpu" else inp


def run_indexer(inp: I.Inputs, status=None):
    return P.indexer_logits(inp.idx_pool, inp.wl.key_fmt, inp.block_table, inp.row_req, inp.row_ctx, inp.max_ctx,
                            inp.q_idx, inp.head_w, inp.wl.rows_per_group, status=status)


def logit_bound(inp: I.Inputs, rows=None):
    """Per-entry accumulation-error bound 2^-13 * sum_h w_h s_t sum_i |q_hi k_ti| (numpy, from decoded bytes)."""
    bt, rq, rc = inp.np("block_table"), inp.np("row_req"), inp.np("row_ctx")
    q = np.abs(pins.ref_e4m3(inp.np("q_idx")))
    w = inp.np("head_w").astype(np.float64)
    pool = inp.np("idx_pool")
    rows = range(len(rc)) if rows is None else rows
    out = {}
    for r in rows:
        t = np.arange(rc[r])
        slots = bt[rq[r], t // 64].astype(np.int64) * 64 + t % 64
        k, s = pins.ref_index_keys(pool, inp.wl.key_fmt, slots)
        out[r] = 2.0 ** -13 * ((w[r] @ (q[r] @ np.abs(k).T)) * s) + 1e-30
    return out


def oracle_logits(inp: I.Inputs, rows=None):
    bt, rq, rc = inp.np("block_table"), inp.np("row_req"), inp.np("row_ctx")
    q, w = inp.np("q_idx"), inp.np("head_w")
    if rows is not None:
        rows = np.asarray(rows)
        return oracle.indexer_logits(inp.np("idx_pool"), ORACLE_FMT[inp.wl.key_fmt], bt, rq[rows], rc[rows], q[rows],
                                     w[rows])
    return oracle.indexer_logits(inp.np("idx_pool"), ORACLE_FMT[inp.wl.key_fmt], bt, rq, rc, q, w)


def mla_errors(got: np.ndarray, ref: np.ndarray):
    d = got.astype(np.float64) - ref
    max_abs = float(np.abs(d).max()) if d.size else 0.0
    rel_l2 = float(np.linalg.norm(d) / max(np.linalg.norm(ref), 1e-30))
    return max_abs, rel_l2


def set_diff_within_band(gpu_idx: np.ndarray, ora_idx: np.ndarray, ora_logits_row: np.ndarray, k: int,
                         rel: float = 1e-3):
    """Tokens selected by only one side must score within rel * |s_k| of the k-th oracle score."""
    g = set(int(x) for x in gpu_idx if x >= 0)
    o = set(int(x) for x in ora_idx if x >= 0)
    diff = g ^ o
    if not diff:
        return True, 0
    vals = ora_logits_row[: len(ora_logits_row)]
    vals = vals[~np.isnan(vals)]
    kth = np.sort(vals)[::-1][min(k, len(vals)) - 1]
    ok = all(abs(ora_logits_row[t] - kth) <= rel * abs(kth) for t in diff)
    return ok, len(diff)
