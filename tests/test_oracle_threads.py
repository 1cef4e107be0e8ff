"""The oracle's results do not depend on how many host threads it runs on, and repeated runs
are bit-identical (its OpenMP loops split rows, never a sum)."""
import numpy as np

import oracle
from prefill_dsa_indexer_gb300 import inputs as I


def _layer(inp, wl):
    lg = oracle.indexer_logits(inp.np("idx_pool"), wl.key_fmt, inp.np("block_table"), inp.np("row_req"),
                               inp.np("row_ctx"), inp.np("q_idx"), inp.np("head_w"))
    idx = oracle.topk_f64(lg, inp.np("row_ctx"), wl.k)
    sl = oracle.page_to_slot(inp.np("block_table"), inp.np("row_req"), idx)
    out, lse = oracle.sparse_mla(inp.np("lat_pool"), wl.lat_fmt, inp.tensor_scale, inp.np("q_mla"), sl,
                                 1.0 / np.sqrt(192.0))
    return lg, idx, sl, out, lse


def _msa(inp):
    sc = oracle.msa_block_scores(inp.np("idx_pool"), inp.np("block_table"), inp.np("row_req"), inp.np("row_ctx"),
                                 inp.np("q_idx"))
    blocks = oracle.msa_select(sc, inp.np("row_ctx"))
    out, lse = oracle.msa_attention(inp.np("kv_pool"), inp.k_scale, inp.v_scale, inp.np("block_table"),
                                    inp.np("row_req"), inp.np("row_ctx"), inp.np("q"), inp.q_scale, blocks,
                                    1.0 / np.sqrt(128.0))
    return sc, blocks, out, lse


def _same(a, b):
    for x, y in zip(a, b):
        assert np.array_equal(x, y, equal_nan=True)


def test_thread_count_does_not_change_results():
    lib = oracle.load()
    n = oracle.num_threads()
    wl = I.small_workload("threads", [1500, 3100, 2049, 700, 2600, 4000], k=512, heads=16, seed=41)
    inp = I.make_inputs(wl, device="cpu")
    mwl = I.small_msa_workload("threads", [2500, 5000, 900], rows_per_req=2, rows_per_group=2, heads_per_group=8,
                               seed=42)
    minp = I.make_msa_inputs(mwl, device="cpu")
    try:
        lib.oracle_set_num_threads(1)
        one, mone = _layer(inp, wl), _msa(minp)
        lib.oracle_set_num_threads(max(n, 4))
        many, mmany = _layer(inp, wl), _msa(minp)
        again = _layer(inp, wl)
    finally:
        lib.oracle_set_num_threads(n)
    _same(one, many)
    _same(many, again)
    _same(mone, mmany)
