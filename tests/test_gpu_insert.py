"""dsa_cache_insert (new-token quantise + cache write) against the oracle:
the whole pools must be byte-identical after the insert (the quantisation
is fully specified in fp32 with round-to-nearest-even codes)."""
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


def _bf16(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16)


@pytest.mark.parametrize("key_fmt,lat_fmt", [(I.KEY_FP8, I.LATENT_FP8), (I.KEY_MXFP4, I.LATENT_NVFP4),
                                             (I.KEY_FP8, I.LATENT_NVFP4), (I.KEY_MXFP4, I.LATENT_FP8)])
def test_insert_bytes_match_oracle(key_fmt, lat_fmt):
    rng = np.random.default_rng(key_fmt * 10 + lat_fmt)
    pages, n = 6, 300
    keys = rng.standard_normal((n, 128)) * rng.uniform(1e-3, 30, (n, 1))
    lats = rng.standard_normal((n, 576)) * rng.uniform(0.1, 3, (n, 1))
    keys[0] = 0.0
    keys[1, :32] = 0.0                       # an all-zero MX block
    keys[2] *= 1e-30                         # tiny values (subnormal scales)
    lats[3, :16] = 0.0                       # an all-zero NVFP4 block
    lats[4] *= 1e3                           # saturating latents
    slots = rng.permutation(pages * 64)[:n].astype(np.int32)
    slots[::17] = -1
    ip0 = rng.integers(0, 256, (pages, I.index_page_bytes(key_fmt)), dtype=np.uint8)
    lp0 = rng.integers(0, 256, (pages, I.latent_page_bytes(lat_fmt)), dtype=np.uint8)
    ts = 0.0137
    kb, lb = _bf16(keys), _bf16(lats)
    ip, lp = torch.from_numpy(ip0).cuda(), torch.from_numpy(lp0).cuda()
    st = P.new_status()
    P.cache_insert(ip, key_fmt, lp, lat_fmt, ts, torch.from_numpy(slots).cuda(), kb.cuda(), lb.cuda(), status=st)
    torch.cuda.synchronize()
    P.check_status(st)
    ref_ip, ref_lp = oracle.cache_insert(ip0, key_fmt, lp0, lat_fmt, ts, slots, kb.numpy().view(np.uint16),
                                         lb.numpy().view(np.uint16))
    assert np.array_equal(ip.cpu().numpy(), ref_ip)
    assert np.array_equal(lp.cpu().numpy(), ref_lp)


def test_insert_then_layer_reads_it():
    """Tokens written by the insert are read back by the indexer and the MLA: a request whose
    whole cache came from dsa_cache_insert scores and attends like the oracle on those bytes."""
    wl = I.small_workload("ins", [700], seed=3)
    inp = I.make_inputs(wl).to("cuda")
    rng = np.random.default_rng(5)
    keys = _bf16(rng.standard_normal((700, 128))).cuda()
    lats = _bf16(rng.standard_normal((700, 576))).cuda()
    t = np.arange(700)
    slots = (inp.np("block_table")[0, t // 64].astype(np.int64) * 64 + t % 64).astype(np.int32)
    P.cache_insert(inp.idx_pool, wl.key_fmt, inp.lat_pool, wl.lat_fmt, inp.tensor_scale,
                   torch.from_numpy(slots).cuda(), keys, lats)
    lg = P.indexer_logits(inp.idx_pool, wl.key_fmt, inp.block_table, inp.row_req, inp.row_ctx, inp.max_ctx,
                          inp.q_idx, inp.head_w)
    torch.cuda.synchronize()
    ref = oracle.indexer_logits(inp.np("idx_pool"), 1, inp.np("block_table"), inp.np("row_req"), inp.np("row_ctx"),
                                inp.np("q_idx"), inp.np("head_w"))
    bound = U.logit_bound(inp, [0])[0]
    d = np.abs(lg.cpu().numpy()[0, :700].astype(np.float64) - ref[0, :700])
    assert np.all(d <= bound[:700]), float((d / bound[:700]).max())
