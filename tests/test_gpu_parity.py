"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Tolerances (written here, derived from the arithmetic and the method's
stated bounds):
  * indexer logits: FP8 products are exact and accumulate in fp32 on the
    tensor cores, so |gpu - exact| <= 2^-13 * sum_h w_h s_t sum_i |q_hi k_ti|;
  * top-k: bit-exact against the oracle's selection on the SAME (gpu) logits;
  * end to end, a token selected by only one side must score within 1e-3
    relative of the k-th oracle score;
  * sparse MLA: max-abs <= 2e-2 and rel-L2 <= 1e-2 (FP8 latents), 3e-2
    (NVFP4 latents); lse within 2e-3.
"""
import math

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


def _wl(name, ctx, rows=1, group=1, lat=I.LATENT_FP8, heads=96, k=2048, seed=5, key=I.KEY_FP8):
    return I.small_workload(name, ctx, rows_per_req=rows, rows_per_group=group, key_fmt=key, lat_fmt=lat,
                            heads=heads, k=k, seed=seed)


INDEXER_CASES = {
    "tiny_4k": I.workload("decode_tiny_4k"),
    "ragged": _wl("ragged", [1, 63, 64, 65, 127, 128, 129, 193, 255, 256, 257, 2047, 2048, 2049, 3000, 5000]),
    # more row groups than one decode launch plans for: the call splits into several launches
    "many_rows": _wl("many", [200 + 37 * (i % 11) for i in range(300)]),
    "verify_g4": _wl("verify", [3000, 4100], rows=4, group=4),
    "pairs_g2": _wl("pairs", [700, 1500, 2500], rows=2, group=2),
    "prefill_g8": _wl("prefill", [3000], rows=64, group=8),
    "mxfp4_ragged": _wl("mx", [1, 64, 65, 129, 2049, 5000], key=I.KEY_MXFP4),
    "mxfp4_verify_g4": _wl("mxv", [3000, 4100], rows=4, group=4, key=I.KEY_MXFP4),
    "mxfp4_prefill_g8": _wl("mxp", [2500], rows=32, group=8, key=I.KEY_MXFP4),
    # steady state of the persistent MXFP4 grid: every CTA runs several tiles, so the stage,
    # accumulator and scale-factor rings all wrap (8 x 80K keys = 2,560 tiles of 256 for G = 1;
    # 4 x 4 rows x 40K = 1,252 tiles of 128 for G = 4; 3 x 2 rows x 60K for G = 2)
    "mxfp4_steady_g1": _wl("mxs1", [80000 + 997 * i for i in range(8)], key=I.KEY_MXFP4, seed=61),
    "mxfp4_steady_g4": _wl("mxs4", [40000, 39001, 40013, 38500], rows=4, group=4, key=I.KEY_MXFP4, seed=62),
    "mxfp4_steady_g2": _wl("mxs2", [60000, 59003, 61111], rows=2, group=2, key=I.KEY_MXFP4, seed=63),
}


def _check_logits(inp, got):
    ref = U.oracle_logits(inp)
    bound = U.logit_bound(inp)
    rc = inp.np("row_ctx")
    for r in range(len(rc)):
        g = got[r, :rc[r]].astype(np.float64)
        d = np.abs(g - ref[r, :rc[r]])
        assert np.all(d <= bound[r]), (r, float(d.max()), float((d / bound[r]).max()))


@pytest.mark.parametrize("case", sorted(INDEXER_CASES))
def test_indexer_logits(case):
    inp = U.gpu_inputs(INDEXER_CASES[case])
    st = P.new_status()
    lg = U.run_indexer(inp, st)
    torch.cuda.synchronize()
    P.check_status(st)
    _check_logits(inp, lg.cpu().numpy())


def _mx_scale_bytes(inp, rows_tokens):
    """(byte offsets of each listed token's four e8m0 scales) in the MXFP4 index pool."""
    bt, rq = inp.np("block_table"), inp.np("row_req")
    offs = []
    for r, t in rows_tokens:
        slot = int(bt[rq[r], t // 64]) * 64 + t % 64
        offs.append((slot // 64) * I.index_page_bytes(I.KEY_MXFP4) + 64 * 64 + (slot % 64) * 4)
    return offs


def test_mxfp4_keys_exact_over_wide_block_exponent_spread():
    # keys whose four 32-value blocks sit up to 130 binades apart: each block's partial product is
    # scaled on its own, so the logits stay within the accumulation bound of the exact values
    inp = U.gpu_inputs(_wl("mxw", [5000, 3000], key=I.KEY_MXFP4, seed=64))
    rng = np.random.default_rng(64)
    pool = inp.idx_pool.cpu().numpy().reshape(-1)
    toks = [(0, int(t)) for t in rng.choice(5000, 1500, replace=False)] + \
           [(1, int(t)) for t in rng.choice(3000, 900, replace=False)]
    spreads = np.array([[131, 109, 97, 128], [127, 27, 147, 60], [20, 150, 85, 126], [140, 140, 10, 139]])
    for i, off in enumerate(_mx_scale_bytes(inp, toks)):
        pool[off:off + 4] = spreads[i % 4]
    inp.idx_pool.copy_(torch.from_numpy(pool.reshape(inp.idx_pool.shape)))
    st = P.new_status()
    lg = U.run_indexer(inp, st)
    torch.cuda.synchronize()
    P.check_status(st)
    _check_logits(inp, lg.cpu().numpy())


def test_mxfp4_nan_scale_of_a_visible_key_is_range_error():
    # the e8m0 code 0xff is NaN in the MX format: a visible key that carries it is reported
    inp = U.gpu_inputs(_wl("mxn", [3000], key=I.KEY_MXFP4, seed=65))
    pool = inp.idx_pool.cpu().numpy().reshape(-1)
    off = _mx_scale_bytes(inp, [(0, 1234)])[0]
    pool[off + 2] = 0xFF
    inp.idx_pool.copy_(torch.from_numpy(pool.reshape(inp.idx_pool.shape)))
    st = P.new_status()
    U.run_indexer(inp, st)
    torch.cuda.synchronize()
    assert int(st.item()) == P.ERR_RANGE


def test_indexer_leaves_masked_entries_untouched():
    inp = U.gpu_inputs(_wl("mask", [100, 1000]))
    lg = torch.full((2, 1000), 12345.0, device="cuda")
    P.indexer_logits(inp.idx_pool, I.KEY_FP8, inp.block_table, inp.row_req, inp.row_ctx, inp.max_ctx, inp.q_idx,
                     inp.head_w, logits=lg)
    torch.cuda.synchronize()
    assert torch.all(lg[0, 100:] == 12345.0)
    assert torch.all(lg[0, :100] != 12345.0)


def _topk_cases():
    rng = np.random.default_rng(3)
    cases = {}
    v = rng.standard_normal((6, 9000)).astype(np.float32)
    cases["normal"] = (v, np.array([9000, 8999, 4096, 2049, 2048, 17], dtype=np.int32), 2048)
    t = (rng.integers(0, 50, (4, 6000)) / 8).astype(np.float32)  # heavy ties
    cases["ties"] = (t, np.array([6000, 5000, 3000, 2100], dtype=np.int32), 2048)
    c = np.zeros((2, 5000), dtype=np.float32)
    c[1, ::3] = -0.0
    cases["all_equal_signed_zero"] = (c, np.array([5000, 5000], dtype=np.int32), 2048)
    big = (rng.standard_normal((2, 200000)) * 10 + 100).astype(np.float32)  # several CTAs per row
    cases["long_rows"] = (big, np.array([200000, 150001], dtype=np.int32), 2048)
    # chunks longer than the shared-memory copy: each CTA re-reads its tail from global memory
    tail = rng.standard_normal((2, 700000)).astype(np.float32)
    cases["cached_tail"] = (tail, np.array([700000, 400003], dtype=np.int32), 2048)
    # more keys equal to the threshold than the candidate list holds: the cluster refines alone
    # to a single key, every CTA counting its own keys above and equal to it
    tb = rng.uniform(0.0, 3.0, (3, 100000)).astype(np.float32)
    tb[0, :20000] = rng.uniform(-1.0, 1.0, 20000)
    tb[0, rng.choice(20000, 5000, replace=False)] = 2.0
    tb[1, rng.choice(100000, 8000, replace=False)] = 3.5
    tb[2, :] = 1.0
    tb[2, rng.choice(100000, 50, replace=False)] = 9.0
    cases["ties_beyond_candidates"] = (tb, np.array([20000, 100000, 100000], dtype=np.int32), 2048)
    # a threshold bin of ~1,500 equal keys in a row cut over several CTAs: the cluster gathers
    # many candidates from its peers and refines them by histogram rounds, not by ranking
    tp = rng.uniform(0.0, 1.0, (2, 100000)).astype(np.float32)
    tp[:, rng.choice(100000, 1500, replace=False)] = 2.0
    tp[0, rng.choice(100000, 1000, replace=False)] = 3.0
    cases["ties_many_candidates"] = (tp, np.array([100000, 99999], dtype=np.int32), 2048)
    # 12 rows of 150K keys: the co-residency check picks a cluster size that need not be a power of
    # two, so the reduce-scatter's bin slices do not divide the histogram evenly
    mid = rng.standard_normal((12, 150000)).astype(np.float32)
    cases["twelve_rows_150k"] = (mid, np.array([150000 - 977 * i for i in range(12)], dtype=np.int32), 2048)
    s = rng.standard_normal((3, 3000)).astype(np.float32)
    cases["small_k"] = (s, np.array([3000, 10, 1], dtype=np.int32), 5)
    w = np.concatenate([np.full((1, 3000), 1e30, np.float32), np.full((1, 3000), -1e30, np.float32)])
    w[0, 1500:] = np.float32(1e-30)
    cases["extremes"] = (w, np.array([3000, 3000], dtype=np.int32), 2048)
    return cases


TOPK_CASES = _topk_cases()


@pytest.mark.parametrize("case", sorted(TOPK_CASES))
def test_topk_bit_exact(case):
    v, ctx, k = TOPK_CASES[case]
    st = P.new_status()
    got = P.topk(torch.from_numpy(v).cuda(), torch.from_numpy(ctx).cuda(), v.shape[1], k, status=st)
    torch.cuda.synchronize()
    P.check_status(st)
    ref = oracle.topk_f32(v, ctx, k)
    assert np.array_equal(got.cpu().numpy(), ref)


def _hist_select_cases():
    """Rows long enough for the histogram selection (a workspace is given): plain, tied and
    concentrated scores, so both the candidate path and the whole-row fallback (a threshold bin of
    more keys than the select kernel holds) are exercised."""
    rng = np.random.default_rng(17)
    cases = {}
    n = 300000  # more chunks than the select kernel's rows get CTAs at two per SM
    v = rng.standard_normal((4, n)).astype(np.float32)
    cases["normal_4x300k"] = (v, np.array([n - 4099 * i for i in range(4)], dtype=np.int32), 2048)
    t = (rng.integers(0, 40, (3, n)) / 8).astype(np.float32)  # ties at the threshold across chunks
    cases["ties"] = (t, np.array([n, 270000, 45000], dtype=np.int32), 2048)
    c = rng.standard_normal((3, n)).astype(np.float32)
    c[0, 10000:13000] += 50.0  # the whole selection inside one early chunk: it cannot pass it all on
    c[1, n - 3000:] += 50.0  # inside the chunk of the most recent tokens
    c[2, ::97] += 50.0  # spread evenly
    cases["concentrated"] = (c, np.array([n, n, n], dtype=np.int32), 2048)
    z = np.zeros((2, n), dtype=np.float32)
    z[1, ::3] = -0.0
    cases["all_equal"] = (z, np.array([n, n - 1], dtype=np.int32), 2048)
    m = rng.standard_normal((5, n)).astype(np.float32)
    cases["short_and_long"] = (m, np.array([n, 100, 2048, 2049, 33333], dtype=np.int32), 2048)
    w = rng.standard_normal((4, n)).astype(np.float32)
    cases["long_k100"] = (w, np.array([n, n - 1, 150000, 80000], dtype=np.int32), 100)
    b = rng.standard_normal((8, 140000)).astype(np.float32) * 40.0 + 150.0  # a decode batch of 8 long rows
    cases["b8_140k"] = (b, np.array([140000] * 6 + [131073, 70001], dtype=np.int32), 2048)
    o = rng.standard_normal((3, 262147)).astype(np.float32)  # odd row stride: unaligned rows, ragged tails
    cases["odd_stride"] = (o, np.array([262147, 200001, 150003], dtype=np.int32), 2048)
    return cases


HIST_SELECT_CASES = _hist_select_cases()


@pytest.mark.parametrize("case", sorted(HIST_SELECT_CASES))
def test_topk_hist_select_bit_exact(case):
    v, ctx, k = HIST_SELECT_CASES[case]
    R, width = v.shape
    need = P.topk_workspace_size(R, width, k)
    assert need > 0  # these shapes take the histogram selection
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    st = P.new_status()
    got = P.topk(torch.from_numpy(v).cuda(), torch.from_numpy(ctx).cuda(), width, k, status=st, workspace=ws)
    torch.cuda.synchronize()
    P.check_status(st)
    assert np.array_equal(got.cpu().numpy(), oracle.topk_f32(v, ctx, k))


def test_topk_hist_select_rejects_a_small_workspace():
    v, ctx, k = HIST_SELECT_CASES["normal_4x300k"]
    ws = torch.empty(P.topk_workspace_size(v.shape[0], v.shape[1], k) - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(P.DsaError, match="workspace"):
        P.topk(torch.from_numpy(v).cuda(), torch.from_numpy(ctx).cuda(), v.shape[1], k, workspace=ws)


def _topk_ws(R, n, k):
    need = P.topk_workspace_size(R, n, k)
    assert need > 0  # the histogram selection
    return torch.empty(need, dtype=torch.uint8, device="cuda")


@pytest.mark.parametrize("n,long_rows", [(5000, False), (300000, True)])
def test_topk_reports_a_nan_logit(n, long_rows):
    """A NaN logit is DSA_ERR_RANGE on both selection paths; the other rows stay exact."""
    v = np.random.default_rng(3).standard_normal((2, n)).astype(np.float32)
    v[1, n // 2] = np.nan
    ctx = np.array([n, n], dtype=np.int32)
    st = P.new_status()
    got = P.topk(torch.from_numpy(v).cuda(), torch.from_numpy(ctx).cuda(), n, 2048, status=st,
                 workspace=_topk_ws(2, n, 2048) if long_rows else None)
    torch.cuda.synchronize()
    assert int(st.item()) == P.ERR_RANGE
    assert np.array_equal(got.cpu().numpy()[0], oracle.topk_f32(v[:1], ctx[:1], 2048)[0])


@pytest.mark.parametrize("n,long_rows", [(5000, False), (300000, True)])
def test_topk_clamps_and_reports_a_row_past_max_ctx(n, long_rows):
    """row_ctx above max_ctx is DSA_ERR_BOUNDS; that row is selected over max_ctx keys."""
    v = np.random.default_rng(4).standard_normal((2, n)).astype(np.float32)
    st = P.new_status()
    got = P.topk(torch.from_numpy(v).cuda(), torch.tensor([n, n + 7], dtype=torch.int32, device="cuda"), n, 2048,
                 status=st, workspace=_topk_ws(2, n, 2048) if long_rows else None)
    torch.cuda.synchronize()
    assert int(st.item()) == P.ERR_BOUNDS
    assert np.array_equal(got.cpu().numpy(), oracle.topk_f32(v, np.array([n, n], dtype=np.int32), 2048))


def test_topk_on_indexer_logits_bit_exact():
    inp = U.gpu_inputs(INDEXER_CASES["ragged"])
    lg = U.run_indexer(inp)
    idx = P.topk(lg, inp.row_ctx, inp.max_ctx, 2048)
    torch.cuda.synchronize()
    ref = oracle.topk_f32(lg.cpu().numpy(), inp.np("row_ctx"), 2048)
    assert np.array_equal(idx.cpu().numpy(), ref)


def test_page_to_slot_exact():
    inp = U.gpu_inputs(INDEXER_CASES["ragged"])
    rng = np.random.default_rng(9)
    rc = inp.np("row_ctx")
    idx = np.full((len(rc), 64), -1, dtype=np.int32)
    for r, L in enumerate(rc):
        n = min(64, L)
        idx[r, :n] = np.sort(rng.choice(L, size=n, replace=False))
    st = P.new_status()
    got = P.page_to_slot(inp.block_table, inp.row_req, inp.row_ctx, inp.max_ctx, inp.num_pages,
                         torch.from_numpy(idx).cuda(), status=st)
    torch.cuda.synchronize()
    P.check_status(st)
    ref = oracle.page_to_slot(inp.np("block_table"), inp.np("row_req"), idx)
    assert np.array_equal(got.cpu().numpy(), ref)


def test_page_to_slot_reports_bounds():
    inp = U.gpu_inputs(_wl("b", [100]))
    idx = torch.tensor([[0, 99, 100, -1]], dtype=torch.int32, device="cuda")  # 100 >= ctx
    st = P.new_status()
    got = P.page_to_slot(inp.block_table, inp.row_req, inp.row_ctx, inp.max_ctx, inp.num_pages, idx, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == P.ERR_BOUNDS
    assert got[0, 2].item() == -1 and got[0, 3].item() == -1


def _mla_case(inp, k, n_valid=None, seed=0):
    """Random distinct positions per row (sorted), -1 padded; physical slots."""
    rng = np.random.default_rng(seed)
    rc, bt, rq = inp.np("row_ctx"), inp.np("block_table"), inp.np("row_req")
    idx = np.full((len(rc), k), -1, dtype=np.int32)
    for r, L in enumerate(rc):
        n = min(k, L) if n_valid is None else min(n_valid, L)
        idx[r, :n] = np.sort(rng.choice(L, size=n, replace=False))
    return oracle.page_to_slot(bt, rq, idx)


MLA_CASES = {
    "fp8_decode_k2048": (_wl("m1", [3000, 5000, 2100]), 2048, None, "decode"),
    "fp8_decode_ragged": (_wl("m2", [3000, 70, 1]), 2048, None, "decode"),
    "fp8_prefill_k2048": (_wl("m3", [2500, 4000]), 2048, None, "prefill"),
    "fp8_decode_partial": (_wl("m4", [3000, 3000]), 2048, 1000, "decode"),
    "fp8_prefill_k100": (_wl("m5", [3000, 40]), 100, None, "prefill"),
    "fp8_heads64": (_wl("m6", [3000], heads=64), 2048, None, "decode"),
    "fp8_heads16": (_wl("m7", [3000], heads=16), 512, None, "prefill"),
    "nvfp4_decode": (_wl("m8", [3000, 2500], lat=I.LATENT_NVFP4), 2048, None, "decode"),
    "nvfp4_prefill": (_wl("m9", [2600], lat=I.LATENT_NVFP4), 2048, None, "prefill"),
}


@pytest.mark.parametrize("case", sorted(MLA_CASES))
def test_sparse_mla(case):
    wl, k, nv, mode = MLA_CASES[case]
    inp = U.gpu_inputs(wl)
    slots = _mla_case(inp, k, nv)
    st = P.new_status()
    fn = P.sparse_mla_decode if mode == "decode" else P.sparse_mla_prefill
    out, lse = fn(inp.lat_pool, wl.lat_fmt, inp.tensor_scale, inp.q_mla, torch.from_numpy(slots).cuda(),
                  U.SM_SCALE, status=st)
    torch.cuda.synchronize()
    P.check_status(st)
    ref_o, ref_l = oracle.sparse_mla(inp.np("lat_pool"), U.ORACLE_FMT[wl.lat_fmt], inp.tensor_scale, inp.np("q_mla"),
                                     slots, U.SM_SCALE)
    tol = 3e-2 if wl.lat_fmt == I.LATENT_NVFP4 else 1e-2
    max_abs, rel = U.mla_errors(out.cpu().numpy(), ref_o)
    assert max_abs <= 2e-2 and rel <= tol, (max_abs, rel)
    gl = lse.cpu().numpy()
    assert np.array_equal(np.isneginf(gl), np.isneginf(ref_l))
    fin = np.isfinite(ref_l)
    assert np.all(np.abs(gl[fin] - ref_l[fin]) <= 2e-3)


def _mla_check(inp, wl, slots, mode, q=None):
    """Run one attention call and compare it with the oracle on the same selection."""
    q = inp.q_mla if q is None else q
    st = P.new_status()
    fn = P.sparse_mla_decode if mode == "decode" else P.sparse_mla_prefill
    out, lse = fn(inp.lat_pool, wl.lat_fmt, inp.tensor_scale, q, torch.from_numpy(slots).cuda(), U.SM_SCALE,
                  status=st)
    torch.cuda.synchronize()
    P.check_status(st)
    ref_o, ref_l = oracle.sparse_mla(inp.np("lat_pool"), U.ORACLE_FMT[wl.lat_fmt], inp.tensor_scale,
                                     q.cpu().numpy(), slots, U.SM_SCALE)
    max_abs, rel = U.mla_errors(out.cpu().numpy(), ref_o)
    assert max_abs <= 2e-2 and rel <= 1e-2, (max_abs, rel)
    gl = lse.cpu().numpy()
    assert np.array_equal(np.isneginf(gl), np.isneginf(ref_l))
    fin = np.isfinite(ref_l)
    assert np.all(np.abs(gl[fin] - ref_l[fin]) <= 2e-3 * np.maximum(1.0, np.abs(ref_l[fin])))


@pytest.mark.parametrize("qmul", [4.0, 16.0])
def test_prefill_scores_spread_over_many_binades(qmul):
    """Queries scaled by a power of two (exact in bf16) spread each head's scores over tens of log2 units,
    so along a row of 64-token tiles the running max moves up many times and the accumulated output and
    sum of those heads are rescaled."""
    wl = _wl("spread", [3000, 2600, 2300], seed=11)
    inp = U.gpu_inputs(wl)
    slots = _mla_case(inp, 2048, seed=3)
    q = (inp.q_mla.view(torch.bfloat16) * qmul).view(torch.int16)
    _mla_check(inp, wl, slots, "prefill", q)


def test_prefill_leading_tiles_without_tokens():
    """The first three tiles of a row hold only unused slots (-1), a middle tile is partly empty, and
    the row ends in a ragged tile: the running max starts at the first valid token."""
    wl = _wl("lead", [3000, 3000], seed=12)
    inp = U.gpu_inputs(wl)
    slots = _mla_case(inp, 1000, seed=4)
    slots = np.concatenate([np.full((2, 192), -1, np.int32), slots], axis=1)  # 1192 = 18 tiles + 40
    slots[0, 500:530] = -1
    _mla_check(inp, wl, slots, "prefill")


@pytest.mark.parametrize("k", [1, 64, 100, 128])
def test_fp8_decode_single_part(k):
    """Decode rows whose selection fits one 128-token part run as one CTA per row (no split merge)."""
    wl = _wl("single", [3000, 90, 2048], seed=13)
    inp = U.gpu_inputs(wl)
    slots = _mla_case(inp, k, seed=5)
    _mla_check(inp, wl, slots, "decode")


def test_sparse_mla_empty_rows():
    inp = U.gpu_inputs(_wl("e", [300, 300]))
    slots = np.full((2, 2048), -1, dtype=np.int32)
    slots[1, :5] = U.oracle.page_to_slot(inp.np("block_table"), inp.np("row_req")[1:], np.arange(5, dtype=np.int32)[None])
    out, lse = P.sparse_mla_decode(inp.lat_pool, I.LATENT_FP8, inp.tensor_scale, inp.q_mla,
                                   torch.from_numpy(slots).cuda())
    torch.cuda.synchronize()
    assert torch.all(out[0] == 0) and torch.all(torch.isneginf(lse[0]))
    assert torch.all(torch.isfinite(lse[1]))


INDEXER_CASES["fp4_both"] = _wl("fp4", [3000, 4500], key=I.KEY_MXFP4, lat=I.LATENT_NVFP4)


@pytest.mark.parametrize("name", ["decode_tiny_4k", "ragged", "verify_g4", "prefill_g8", "fp4_both"])
def test_layer_end_to_end(name):
    wl = INDEXER_CASES.get(name) or I.workload(name)
    inp = U.gpu_inputs(wl)
    prefill = wl.rows_per_group == 8
    layer = P.Layer(inp.idx_pool, wl.key_fmt, inp.lat_pool, wl.lat_fmt, inp.tensor_scale, inp.block_table,
                    inp.max_ctx, wl.num_rows, wl.heads, wl.k, wl.rows_per_group, prefill=prefill)
    out, lse = layer.run(inp.row_req, inp.row_ctx, inp.q_idx, inp.head_w, inp.q_mla)
    torch.cuda.synchronize()
    P.check_status(layer.status)
    ref_lg = U.oracle_logits(inp)
    ora_idx = oracle.topk_f64(np.nan_to_num(ref_lg, nan=-np.inf), inp.np("row_ctx"), wl.k)
    gpu_idx = layer.idx.cpu().numpy()
    for r in range(wl.num_rows):
        ok, nd = U.set_diff_within_band(gpu_idx[r], ora_idx[r], ref_lg[r], wl.k)
        assert ok, (r, nd)
    # the slots the attention read are the oracle's translation of the GPU's selection
    gslots = layer.slots.cpu().numpy()
    assert np.array_equal(gslots, oracle.page_to_slot(inp.np("block_table"), inp.np("row_req"), gpu_idx))
    # attention parity on the GPU's own selection
    ref_o, _ = oracle.sparse_mla(inp.np("lat_pool"), U.ORACLE_FMT[wl.lat_fmt], inp.tensor_scale, inp.np("q_mla"),
                                 gslots, U.SM_SCALE)
    max_abs, rel = U.mla_errors(out.cpu().numpy(), ref_o)
    tol = 3e-2 if wl.lat_fmt == I.LATENT_NVFP4 else 1e-2
    assert max_abs <= 2e-2 and rel <= tol, (max_abs, rel)


def test_layer_deterministic_and_batch_invariant():
    wl = _wl("inv", [3000, 5000, 4100, 2200], seed=21)
    inp = U.gpu_inputs(wl)
    layer = P.Layer(inp.idx_pool, wl.key_fmt, inp.lat_pool, wl.lat_fmt, inp.tensor_scale, inp.block_table,
                    inp.max_ctx, wl.num_rows)
    runs = []
    for _ in range(3):
        o, l = layer.run(inp.row_req, inp.row_ctx, inp.q_idx, inp.head_w, inp.q_mla)
        runs.append((o.clone(), l.clone(), layer.idx.clone()))
    torch.cuda.synchronize()
    for o, l, i in runs[1:]:
        assert torch.equal(o, runs[0][0]) and torch.equal(l, runs[0][1]) and torch.equal(i, runs[0][2])
    # row 2 alone gives the bit-identical result
    one = P.Layer(inp.idx_pool, wl.key_fmt, inp.lat_pool, wl.lat_fmt, inp.tensor_scale, inp.block_table,
                  inp.max_ctx, 1)
    o1, l1 = one.run(inp.row_req[2:3].contiguous(), inp.row_ctx[2:3].contiguous(), inp.q_idx[2:3].contiguous(),
                     inp.head_w[2:3].contiguous(), inp.q_mla[2:3].contiguous())
    torch.cuda.synchronize()
    assert torch.equal(one.idx[0], runs[0][2][2])
    assert torch.equal(o1[0], runs[0][0][2]) and torch.equal(l1[0], runs[0][1][2])
