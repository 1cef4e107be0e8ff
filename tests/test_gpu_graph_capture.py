"""One decode step captured as a CUDA graph (query preparation on a parallel branch, scorer,
top-k with slots and L2 warm-up, sparse attention), replayed with new queries copied into its
input buffers, gives bit for bit the results of the same calls made eagerly."""
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


def test_graph_replay_equals_eager_calls():
    ctx = [3000, 9000, 2100, 6000]
    wl = I.small_workload("graph", ctx, seed=31)
    a = U.gpu_inputs(wl)
    b = U.gpu_inputs(I.small_workload("graph", ctx, seed=32))  # other queries and weights, same shapes
    layer = P.Layer(a.idx_pool, wl.key_fmt, a.lat_pool, wl.lat_fmt, a.tensor_scale, a.block_table, a.max_ctx,
                    wl.num_rows)

    def eager(q_idx, head_w, q_mla):
        o, l = layer.run(a.row_req, a.row_ctx, q_idx, head_w, q_mla)
        return o.clone(), l.clone(), layer.idx.clone(), layer.slots.clone()

    want_a = eager(a.q_idx, a.head_w, a.q_mla)
    want_b = eager(b.q_idx, b.head_w, b.q_mla)
    torch.cuda.synchronize()
    P.check_status(layer.status)

    # the graph reads its queries from these buffers
    d = {"row_req": a.row_req.clone(), "row_ctx": a.row_ctx.clone(), "q_idx": a.q_idx.clone(),
         "head_w": a.head_w.clone(), "q_mla": a.q_mla.clone()}
    cap, side = torch.cuda.Stream(), torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cap):
        with torch.cuda.graph(g, stream=cap):
            # the shape bench.py times: scorer, then the query prep on a side branch beside the top-k
            layer.score(d["row_req"], d["row_ctx"], d["q_idx"], d["head_w"])
            side.wait_stream(cap)
            with torch.cuda.stream(side):
                layer.prepare(d["q_mla"])
            layer.select_tokens(d["row_req"], d["row_ctx"])
            cap.wait_stream(side)
            layer.attend(d["q_mla"], prepared=True)
    torch.cuda.current_stream().wait_stream(cap)

    def replayed(src):
        for n in ("q_idx", "head_w", "q_mla"):
            d[n].copy_(getattr(src, n))
        g.replay()
        torch.cuda.synchronize()
        return layer.out.clone(), layer.lse.clone(), layer.idx.clone(), layer.slots.clone()

    for src, want in ((b, want_b), (a, want_a), (b, want_b)):
        got = replayed(src)
        for x, y in zip(got, want):
            assert torch.equal(x, y)
    P.check_status(layer.status)
