"""dsa_sparse_mla_decode_noalloc against dsa_sparse_mla_decode.

The no-alloc variant serves callers that cannot allocate device memory (a
host framework that has reserved the device's memory for its own pools, a
plugin that only sees the tensors it is handed, a latency-critical loop that
must not call cudaMalloc): its split-K scratch lives in a fixed array inside
the library instead of a caller workspace.  This file is collected last so a
run that stops at the first failure has already run every other test; it
also passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

import prefill_dsa_indexer_gb300 as P
from prefill_dsa_indexer_gb300 import inputs as I
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from prefill_dsa_indexer_gb300 import build
    build.build()
    P.load_library()


def _case(seed, ctx, lat=I.LATENT_FP8):
    wl = I.small_workload("noalloc", ctx, lat_fmt=lat, seed=seed)
    inp = U.gpu_inputs(wl)
    rng = np.random.default_rng(seed)
    rc, bt, rq = inp.np("row_ctx"), inp.np("block_table"), inp.np("row_req")
    idx = np.full((len(rc), 2048), -1, dtype=np.int32)
    for r, L in enumerate(rc):
        n = min(2048, L)
        idx[r, :n] = np.sort(rng.choice(L, size=n, replace=False))
    slots = torch.from_numpy(U.oracle.page_to_slot(bt, rq, idx)).cuda()
    return wl, inp, slots


def _close(a, b):
    max_abs, rel = U.mla_errors(a.cpu().numpy(), b.cpu().numpy().astype(np.float64))
    return max_abs <= 2e-2 and rel <= 1e-2


def test_noalloc_matches_decode_on_two_calls_in_a_row():
    for seed, ctx, lat in ((41, [3000, 5000, 2100, 70, 2600, 4400, 3900, 2048], I.LATENT_FP8),
                           (42, [3000, 2500], I.LATENT_NVFP4)):
        wl, inp, slots = _case(seed, ctx, lat)
        R = wl.num_rows
        ref_o, ref_l = P.sparse_mla_decode(inp.lat_pool, lat, inp.tensor_scale, inp.q_mla, slots)
        for _ in range(2):
            out = torch.full((R, wl.heads, 512), float("nan"), device="cuda")
            lse = torch.full((R, wl.heads), float("nan"), device="cuda")
            st = P.new_status()
            P.sparse_mla_decode_noalloc(inp.lat_pool, lat, inp.tensor_scale, inp.q_mla, slots, out, lse, status=st)
            torch.cuda.synchronize()
            P.check_status(st)
            assert _close(out, ref_o)
            assert torch.allclose(lse, ref_l, rtol=0, atol=2e-3)


def test_noalloc_rejects_more_rows_than_its_scratch_holds():
    wl, inp, slots = _case(43, [3000] * (P.NOALLOC_MAX_ROWS + 1))
    out = torch.empty((wl.num_rows, wl.heads, 512), device="cuda")
    lse = torch.empty((wl.num_rows, wl.heads), device="cuda")
    with pytest.raises(P.DsaError, match="workspace"):
        P.sparse_mla_decode_noalloc(inp.lat_pool, I.LATENT_FP8, inp.tensor_scale, inp.q_mla, slots, out, lse)
