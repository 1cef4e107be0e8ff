"""Full-size workloads, in the launch configuration bench.py times (the
`Layer` chain over GPU-generated inputs), checked on sampled rows that the
oracle can afford one by one:

  * indexer logits of a sampled row within the accumulation bound;
  * the row's top-k set equals the oracle's up to ties inside the 1e-3 band,
    and is bit-exactly the oracle's selection over the GPU's own logits;
  * the row's attention output within the FP8 (NVFP4) tolerance, on the
    GPU's own selection;
  * every row: selection sorted ascending, in range, no duplicates.
"""
import numpy as np
import pytest
import torch

import oracle
import prefill_dsa_indexer_gb300 as P
from prefill_dsa_indexer_gb300 import inputs as I
from tests import gpu_util as U

pytestmark = pytest.mark.gpu

CASES = {
    # name: sampled rows
    "decode_b8_128k_fp8": [0, 5],
    "decode_b32_16k_64k": [3, 31],
    "verify_b4_256k": [2, 13],
    "prefill_8k_on_56k": [0, 4097, 8191],
    "verify_b1_1m": [3],
    "decode_b8_128k_fp4": [2, 7],
}


@pytest.fixture(scope="module", autouse=True)
def built():
    from prefill_dsa_indexer_gb300 import build
    build.build()


@pytest.mark.parametrize("name", list(CASES))
def test_fullsize_sampled(name):
    wl = I.workload(name)
    inp = I.make_inputs(wl, device="cuda")
    prefill = wl.rows_per_req > 8
    layer = P.Layer(inp.idx_pool, wl.key_fmt, inp.lat_pool, wl.lat_fmt, inp.tensor_scale, inp.block_table,
                    inp.max_ctx, wl.num_rows, wl.heads, wl.k, wl.rows_per_group, prefill=prefill)
    out, lse = layer.run(inp.row_req, inp.row_ctx, inp.q_idx, inp.head_w, inp.q_mla)
    torch.cuda.synchronize()
    P.check_status(layer.status)
    rc = inp.np("row_ctx")
    idx = layer.idx.cpu().numpy()
    # every row: a valid selection
    for r in range(wl.num_rows):
        n = min(wl.k, int(rc[r]))
        sel = idx[r, :n]
        assert np.all(sel >= 0) and np.all(sel < rc[r]) and np.all(np.diff(sel) > 0), r
        assert np.all(idx[r, n:] == -1), r
    rows = CASES[name]
    ref_lg = U.oracle_logits(inp, rows)
    gpu_lg = layer.logits.cpu().numpy()
    bound = U.logit_bound(inp, rows)
    ora_idx = oracle.topk_f64(np.nan_to_num(ref_lg, nan=-np.inf), rc[rows], wl.k)
    # the selection of the sampled rows is exactly the oracle's over the GPU's own logits
    assert np.array_equal(idx[rows], oracle.topk_f32(gpu_lg[rows], rc[rows], wl.k))
    for i, r in enumerate(rows):
        d = np.abs(gpu_lg[r, :rc[r]].astype(np.float64) - ref_lg[i, :rc[r]])
        assert np.all(d <= bound[r]), (r, float((d / bound[r]).max()))
        ok, nd = U.set_diff_within_band(idx[r], ora_idx[i], ref_lg[i], wl.k)
        assert ok, (r, nd)
    # every row: the slots are the oracle's translation of the GPU's selection
    all_slots = layer.slots.cpu().numpy()
    assert np.array_equal(all_slots, oracle.page_to_slot(inp.np("block_table"), inp.np("row_req"), idx))
    # attention on the GPU's own selection for the sampled rows
    gslots = all_slots[rows]
    ref_o, ref_l = oracle.sparse_mla(inp.np("lat_pool"), U.ORACLE_FMT[wl.lat_fmt], inp.tensor_scale,
                                     inp.np("q_mla")[rows], gslots, U.SM_SCALE)
    tol = 3e-2 if wl.lat_fmt == I.LATENT_NVFP4 else 1e-2
    max_abs, rel = U.mla_errors(out.cpu().numpy()[rows], ref_o)
    assert max_abs <= 2e-2 and rel <= tol, (max_abs, rel)
    assert np.all(np.abs(lse.cpu().numpy()[rows] - ref_l) <= 2e-3)
