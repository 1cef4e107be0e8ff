"""Failure detection without a GPU fault: a kernel's bounded wait runs out on a barrier that
nothing arrives on, the device status word reports DSA_ERR_TIMEOUT, and the context keeps
working (the next layer call is still exact)."""
import time

import numpy as np
import pytest
import torch

import oracle
import prefill_dsa_indexer_gb300 as P
from prefill_dsa_indexer_gb300 import inputs as I
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from prefill_dsa_indexer_gb300 import build
    build.build()
    P.load_library()


def test_wait_limit_reports_timeout_and_context_survives():
    st = P.new_status()
    t0 = time.time()
    P.selftest_wait_timeout(st)
    torch.cuda.synchronize()
    waited = time.time() - t0
    assert int(st.item()) == P.ERR_TIMEOUT
    assert waited < 30.0  # the wait is bounded (about two seconds of SM clock)
    with pytest.raises(P.DsaError):
        P.check_status(st)
    # the same context still runs the path exactly
    inp = U.gpu_inputs(I.workload("decode_tiny_4k"))
    st2 = P.new_status()
    lg = P.indexer_logits(inp.idx_pool, inp.wl.key_fmt, inp.block_table, inp.row_req, inp.row_ctx, inp.max_ctx,
                          inp.q_idx, inp.head_w, status=st2)
    idx = P.topk(lg, inp.row_ctx, inp.max_ctx, 2048, status=st2)
    torch.cuda.synchronize()
    P.check_status(st2)
    ref = oracle.topk_f32(lg.cpu().numpy(), inp.np("row_ctx"), 2048)
    assert np.array_equal(idx.cpu().numpy(), ref)


def test_selftest_needs_a_status_word():
    with pytest.raises(P.DsaError):
        P._check(P.load_library().dsa_selftest_wait_timeout(None, P._stream(None)), "selftest")
