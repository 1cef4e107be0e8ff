"""Single-pass scorer + top-k (the scorer's epilogue builds each row's histogram of
logit keys; the top-k starts from it): bit-exact against the oracle's top-k of
the same logits, the histogram equal to its definition and left zeroed, and the
fused call reusable on one workspace.

The histogram's definition (dsa.h): bin = top 16 bits of the order-preserving
32-bit key of the fp32 logit (negative floats: all bits flipped; others: sign
bit set; -0 folds onto +0; NaN is key 0).  It is restated here in numpy so the
top-k path can also be fed logits the scorer did not produce (heavy ties)."""
import numpy as np
import pytest
import torch

import oracle
import prefill_dsa_indexer_gb300 as P
from tests import gpu_util as U
from tests.test_gpu_parity import INDEXER_CASES, TOPK_CASES

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from prefill_dsa_indexer_gb300 import build
    build.build()
    P.load_library()


def order_keys(v: np.ndarray) -> np.ndarray:
    f = np.ascontiguousarray(v, dtype=np.float32)
    u = f.view(np.uint32).copy()
    u[u == 0x80000000] = 0
    neg = (u & 0x80000000) != 0
    key = np.where(neg, ~u, u | np.uint32(0x80000000)).astype(np.uint32)
    key[np.isnan(f)] = 0
    return key


def histogram(logits: np.ndarray, row_ctx: np.ndarray) -> np.ndarray:
    h = np.zeros((len(row_ctx), P.HIST_BINS), dtype=np.int64)
    for r, n in enumerate(row_ctx):
        if n > 0:
            h[r] = np.bincount(order_keys(logits[r, :n]) >> 16, minlength=P.HIST_BINS)
    return h


@pytest.mark.parametrize("case", sorted(TOPK_CASES))
def test_topk_hist_bit_exact(case):
    v, ctx, k = TOPK_CASES[case]
    hist = torch.from_numpy(histogram(v, ctx).astype(np.uint32).view(np.int32)).cuda()
    st = P.new_status()
    got = P.topk_hist(torch.from_numpy(v).cuda(), torch.from_numpy(ctx).cuda(), v.shape[1], hist, k, status=st)
    torch.cuda.synchronize()
    P.check_status(st)
    assert np.array_equal(got.cpu().numpy(), oracle.topk_f32(v, ctx, k))
    assert int(torch.count_nonzero(hist)) == 0  # left zeroed for the next scorer call


@pytest.mark.parametrize("case", ["ragged", "verify_g4", "pairs_g2", "prefill_g8", "mxfp4_ragged",
                                  "mxfp4_verify_g4", "tiny_4k"])
def test_scorer_histogram_and_topk(case):
    inp = U.gpu_inputs(INDEXER_CASES[case])
    R = inp.row_ctx.shape[0]
    plain = U.run_indexer(inp)
    hist = P.new_hist(R)
    st = P.new_status()
    lg = P.indexer_logits_hist(inp.idx_pool, inp.wl.key_fmt, inp.block_table, inp.row_req, inp.row_ctx,
                               inp.max_ctx, inp.q_idx, inp.head_w, hist, inp.wl.rows_per_group, status=st)
    torch.cuda.synchronize()
    P.check_status(st)
    rc = inp.np("row_ctx")
    lg_np, plain_np = lg.cpu().numpy(), plain.cpu().numpy()
    for r in range(R):  # the same logits as the plain scorer, bit for bit
        assert np.array_equal(lg_np[r, :rc[r]].view(np.uint32), plain_np[r, :rc[r]].view(np.uint32))
    assert np.array_equal(hist.cpu().numpy().view(np.uint32).astype(np.int64), histogram(lg_np, rc))
    for k in (2048, 37):
        if k != 2048:  # the histogram is consumed: rebuild it for the second k
            P.indexer_logits_hist(inp.idx_pool, inp.wl.key_fmt, inp.block_table, inp.row_req, inp.row_ctx,
                                  inp.max_ctx, inp.q_idx, inp.head_w, hist, inp.wl.rows_per_group, logits=lg,
                                  status=st)
        idx = P.topk_hist(lg, inp.row_ctx, inp.max_ctx, hist, k, status=st)
        torch.cuda.synchronize()
        P.check_status(st)
        assert np.array_equal(idx.cpu().numpy(), oracle.topk_f32(lg_np, rc, k))
        assert int(torch.count_nonzero(hist)) == 0


@pytest.mark.parametrize("case", ["ragged", "verify_g4", "mxfp4_ragged"])
def test_fused_indexer_topk_twice(case):
    inp = U.gpu_inputs(INDEXER_CASES[case])
    R = inp.row_ctx.shape[0]
    ws = torch.zeros(P.indexer_topk_workspace_size(R, inp.max_ctx), dtype=torch.uint8, device="cuda")
    ref = oracle.topk_f32(U.run_indexer(inp).cpu().numpy(), inp.np("row_ctx"), 2048)
    st = P.new_status()
    for _ in range(2):  # the call leaves its histogram zeroed, so the workspace is reusable
        got = P.indexer_topk(inp.idx_pool, inp.wl.key_fmt, inp.block_table, inp.row_req, inp.row_ctx, inp.max_ctx,
                             inp.q_idx, inp.head_w, ws, 2048, inp.wl.rows_per_group, status=st)
        torch.cuda.synchronize()
        P.check_status(st)
        assert np.array_equal(got.cpu().numpy(), ref)
