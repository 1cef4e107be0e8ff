"""Calls that merge or split steps of the path: top-k with the page -> slot
translation in its output pass (equal to dsa_topk then dsa_page_to_slot, and
to the oracle's selection and slots; with the L2 warm-up of the chosen
latents, equal to it bit for bit), and the decode attention split into
query preparation + attention (equal bit for bit to the single call)."""
import numpy as np
import pytest
import torch

import oracle
import prefill_dsa_indexer_gb300 as P
from prefill_dsa_indexer_gb300 import inputs as I
from tests import gpu_util as U
from tests.test_gpu_parity import INDEXER_CASES, TOPK_CASES, _wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from prefill_dsa_indexer_gb300 import build
    build.build()
    P.load_library()


@pytest.mark.parametrize("case", sorted(TOPK_CASES))
def test_topk_slots_matches_oracle(case):
    v, ctx, k = TOPK_CASES[case]
    R, width = v.shape
    rng = np.random.default_rng(11)
    pages = (width + 63) // 64
    pool_pages = R * pages + 5
    bt = np.stack([rng.permutation(pool_pages)[:pages] for _ in range(R)]).astype(np.int32)
    row_req = np.arange(R, dtype=np.int32)
    st = P.new_status()
    idx, slots = P.topk_slots(torch.from_numpy(v).cuda(), torch.from_numpy(bt).cuda(), torch.from_numpy(row_req).cuda(),
                              torch.from_numpy(ctx).cuda(), width, pool_pages, k, status=st)
    torch.cuda.synchronize()
    P.check_status(st)
    ref = oracle.topk_f32(v, ctx, k)
    assert np.array_equal(idx.cpu().numpy(), ref)
    assert np.array_equal(slots.cpu().numpy(), oracle.page_to_slot(bt, row_req, ref))


def test_topk_slots_on_indexer_logits():
    inp = U.gpu_inputs(INDEXER_CASES["ragged"])
    lg = U.run_indexer(inp)
    st = P.new_status()
    idx, slots = P.topk_slots(lg, inp.block_table, inp.row_req, inp.row_ctx, inp.max_ctx, inp.lat_pool.shape[0], 2048,
                              status=st)
    torch.cuda.synchronize()
    P.check_status(st)
    ref = oracle.topk_f32(lg.cpu().numpy(), inp.np("row_ctx"), 2048)
    assert np.array_equal(idx.cpu().numpy(), ref)
    assert np.array_equal(slots.cpu().numpy(), oracle.page_to_slot(inp.np("block_table"), inp.np("row_req"), ref))


@pytest.mark.parametrize("lat", [I.LATENT_FP8, I.LATENT_NVFP4])
@pytest.mark.parametrize("k", [2048, 100])
def test_topk_slots_warm_equals_topk_slots(lat, k):
    # warming L2 with the chosen latents changes no output
    inp = U.gpu_inputs(_wl("warm", [1, 100, 2048, 2049, 5000, 9000], lat=lat, k=k, seed=29))
    lg = U.run_indexer(inp)
    st = P.new_status()
    a_idx, a_sl = P.topk_slots(lg, inp.block_table, inp.row_req, inp.row_ctx, inp.max_ctx, inp.lat_pool.shape[0], k,
                               status=st)
    b_idx, b_sl = P.topk_slots_warm(lg, inp.block_table, inp.row_req, inp.row_ctx, inp.max_ctx, inp.lat_pool,
                                    inp.wl.lat_fmt, k, status=st)
    torch.cuda.synchronize()
    P.check_status(st)
    assert torch.equal(a_idx, b_idx) and torch.equal(a_sl, b_sl)


@pytest.mark.parametrize("lat", [I.LATENT_FP8, I.LATENT_NVFP4])
@pytest.mark.parametrize("k", [2048, 300, 100])
def test_decode_prepare_then_prepared_equals_decode(lat, k):
    wl = _wl("prep", [5000, 3000, 2500], lat=lat, k=k, seed=23)
    inp = U.gpu_inputs(wl)
    lg = U.run_indexer(inp)
    idx = P.topk(lg, inp.row_ctx, inp.max_ctx, k)
    slots = P.page_to_slot(inp.block_table, inp.row_req, inp.row_ctx, inp.max_ctx, inp.lat_pool.shape[0], idx)
    R, H = inp.q_mla.shape[0], inp.q_mla.shape[1]
    ws = torch.empty(max(P.sparse_mla_workspace_size(R, H, k), 256), dtype=torch.uint8, device="cuda")
    st = P.new_status()
    o1, l1 = P.sparse_mla_decode(inp.lat_pool, lat, inp.tensor_scale, inp.q_mla, slots, workspace=ws, status=st)
    o1, l1 = o1.clone(), l1.clone()
    ws2 = torch.empty_like(ws)
    P.sparse_mla_decode_prepare(inp.lat_pool, lat, inp.tensor_scale, inp.q_mla, k, ws2, status=st)
    o2, l2 = P.sparse_mla_decode_prepared(inp.lat_pool, lat, inp.tensor_scale, inp.q_mla, slots, workspace=ws2,
                                          status=st)
    torch.cuda.synchronize()
    P.check_status(st)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
