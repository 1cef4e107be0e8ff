"""Parity of the MSA block-sparse variant (through the C ABI) with the CPU oracle.

Tolerances (written here, derived from the arithmetic):
  * block scores: FP8 products are exact and accumulate in fp32 on the tensor
    cores, so each token's score is within 2^-13 * sum_i |q_i k_ti| of exact,
    and a block max within the largest such bound over the block's tokens;
  * selection: bit-exact against the oracle's selection on the SAME (gpu)
    fp32 scores; end to end, a block chosen by only one side must score within
    1e-3 relative of the oracle's 15th-best score of that (row, group);
  * attention (FP8 queries, K and V; fp16 P): max-abs <= 2e-2 and rel-L2 <=
    1e-2 against the oracle on the same blocks; lse within 2e-3.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import prefill_dsa_indexer_gb300 as P
from prefill_dsa_indexer_gb300 import inputs as I
from tests import oracle_pins as pins

pytestmark = pytest.mark.gpu

SM_SCALE = 1.0 / math.sqrt(128.0)


@pytest.fixture(scope="module", autouse=True)
def built():
    from prefill_dsa_indexer_gb300 import build
    build.build()
    P.load_library()


def _wl(name, ctx, rows=1, group=1, hpg=16, seed=11):
    return I.small_msa_workload(name, ctx, rows_per_req=rows, rows_per_group=group, heads_per_group=hpg, seed=seed)


CASES = {
    "tiny_4k": I.msa_workload("msa_decode_tiny_4k"),
    "ragged": _wl("ragged", [1, 127, 128, 129, 2047, 2048, 2049, 2177, 5000, 9000]),
    "pairs_g2": _wl("pairs", [1500, 4100, 7000], rows=2, group=2),
    "verify_g4": _wl("verify", [3000, 6000], rows=4, group=4),
    "verify_g8": _wl("verify8", [2600, 9000], rows=8, group=8, hpg=32),
    "heads64": _wl("h64", [3000, 20000], hpg=64),
    "heads48": _wl("h48", [5000], hpg=48),
    "long_128k": _wl("long", [131072 - 5]),  # 1024 blocks: every selection warp holds 128 candidates
}


def _inputs(wl):
    return I.make_msa_inputs(wl, device="cpu").to("cuda")


def _score_bound(inp):
    """Per (row, group, block): 2^-13 * max over the block's visible tokens of sum_i |q_gi k_ti|."""
    bt, rq, rc = inp.np("block_table"), inp.np("row_req"), inp.np("row_ctx")
    pool = inp.np("idx_pool").reshape(-1, I.MSA_PAGE, I.MSA_DIM)
    q = np.abs(pins.ref_e4m3(inp.np("q_idx")))  # [R, 4, 128]
    R = len(rc)
    W = max((int(rc.max()) + 127) // 128, 1)
    out = np.zeros((R, 4, W))
    for r in range(R):
        nb = (rc[r] + 127) // 128
        for b in range(nb):
            n = min(128, rc[r] - 128 * b)
            k = np.abs(pins.ref_e4m3(pool[bt[rq[r], b], :n]))  # [n, 128]
            out[r, :, b] = 2.0 ** -13 * (q[r] @ k.T).max(axis=1)
    return out


def _gpu_scores(inp, status):
    return P.msa_block_scores(inp.idx_pool, inp.block_table, inp.row_req, inp.row_ctx, inp.max_ctx, inp.q_idx,
                              inp.wl.rows_per_group, status=status)


@pytest.mark.parametrize("case", sorted(CASES))
def test_msa_block_scores(case):
    inp = _inputs(CASES[case])
    st = P.new_status()
    got = _gpu_scores(inp, st).cpu().numpy().astype(np.float64)
    torch.cuda.synchronize()
    P.check_status(st)
    ref = oracle.msa_block_scores(inp.np("idx_pool"), inp.np("block_table"), inp.np("row_req"), inp.np("row_ctx"),
                                  inp.np("q_idx"))
    bound = _score_bound(inp)
    rc = inp.np("row_ctx")
    for r in range(len(rc)):
        nb = (rc[r] + 127) // 128
        d = np.abs(got[r, :, :nb] - ref[r, :, :nb])
        assert np.all(d <= bound[r, :, :nb] + 1e-30), (case, r, float(d.max()))


@pytest.mark.parametrize("case", sorted(CASES))
def test_msa_select_bit_exact(case):
    inp = _inputs(CASES[case])
    st = P.new_status()
    sc = _gpu_scores(inp, st)
    got = P.msa_select(sc, inp.row_ctx, inp.max_ctx, status=st).cpu().numpy()
    torch.cuda.synchronize()
    P.check_status(st)
    ref = oracle.msa_select(sc.cpu().numpy(), inp.np("row_ctx"))
    assert np.array_equal(got, ref), case


def test_msa_select_ties_and_nan():
    # constructed scores: equal values resolve to the lower block; NaN never wins
    R, W = 3, 40
    rc = torch.tensor([40 * 128, 17 * 128 - 5, 16 * 128], dtype=torch.int32, device="cuda")
    sc = torch.zeros((R, 4, W), dtype=torch.float32)
    sc[:, 0, :] = 1.0                                  # all tied
    sc[:, 1, :] = torch.arange(W, dtype=torch.float32)  # increasing
    sc[:, 2, ::3] = float("nan")
    sc[:, 2, 1::3] = -0.0
    sc[:, 3, :] = -torch.arange(W, dtype=torch.float32)
    sc = sc.cuda()
    st = P.new_status()
    got = P.msa_select(sc, rc, 40 * 128, status=st).cpu().numpy()
    torch.cuda.synchronize()
    P.check_status(st)
    ref = oracle.msa_select(sc.cpu().numpy(), rc.cpu().numpy())
    assert np.array_equal(got, ref)
    assert list(got[0, 0]) == list(range(15)) + [39]


@pytest.mark.parametrize("case", sorted(CASES))
def test_msa_attention(case):
    inp = _inputs(CASES[case])
    st = P.new_status()
    sc = _gpu_scores(inp, st)
    blocks = P.msa_select(sc, inp.row_ctx, inp.max_ctx, status=st)
    out, lse = P.msa_attention(inp.kv_pool, inp.k_scale, inp.v_scale, inp.block_table, inp.row_req, inp.row_ctx,
                               inp.max_ctx, inp.q, inp.q_scale, blocks, SM_SCALE, status=st)
    torch.cuda.synchronize()
    P.check_status(st)
    ref_o, ref_l = oracle.msa_attention(inp.np("kv_pool"), inp.k_scale, inp.v_scale, inp.np("block_table"),
                                        inp.np("row_req"), inp.np("row_ctx"), inp.np("q"), inp.q_scale,
                                        blocks.cpu().numpy(), SM_SCALE)
    o = out.cpu().numpy().astype(np.float64)
    err = np.abs(o - ref_o)
    rel = np.linalg.norm(o - ref_o) / max(np.linalg.norm(ref_o), 1e-30)
    assert err.max() <= 2e-2 and rel <= 1e-2, (case, float(err.max()), float(rel))
    l = lse.cpu().numpy().astype(np.float64)
    fin = np.isfinite(ref_l)
    assert np.array_equal(fin, np.isfinite(l))
    assert np.abs(l[fin] - ref_l[fin]).max() <= 2e-3


def test_msa_end_to_end_selection_band():
    inp = _inputs(CASES["ragged"])
    st = P.new_status()
    sc = _gpu_scores(inp, st)
    got = P.msa_select(sc, inp.row_ctx, inp.max_ctx, status=st).cpu().numpy()
    torch.cuda.synchronize()
    P.check_status(st)
    ref_sc = oracle.msa_block_scores(inp.np("idx_pool"), inp.np("block_table"), inp.np("row_req"),
                                     inp.np("row_ctx"), inp.np("q_idx"))
    ref = oracle.msa_select(ref_sc, inp.np("row_ctx"))
    rc = inp.np("row_ctx")
    for r in range(len(rc)):
        nb = (rc[r] + 127) // 128
        for g in range(4):
            a, b = set(got[r, g]) - {-1}, set(ref[r, g]) - {-1}
            if a == b:
                continue
            s = ref_sc[r, g, :nb - 1]
            kth = np.sort(s)[::-1][14]
            for blk in a ^ b:
                assert abs(s[blk] - kth) <= 1e-3 * abs(kth), (r, g, blk)


def test_msa_empty_and_unused_slots():
    # a row whose blocks are all -1 attends to nothing: out = 0, lse = -inf
    inp = _inputs(_wl("e", [300, 3000]))
    blocks = torch.full((2, 4, 16), -1, dtype=torch.int32, device="cuda")
    blocks[1, :, 0] = 0
    st = P.new_status()
    out, lse = P.msa_attention(inp.kv_pool, inp.k_scale, inp.v_scale, inp.block_table, inp.row_req, inp.row_ctx,
                               inp.max_ctx, inp.q, inp.q_scale, blocks, SM_SCALE, status=st)
    torch.cuda.synchronize()
    P.check_status(st)
    assert torch.all(out[0] == 0) and torch.all(torch.isinf(lse[0])) and torch.all(lse[0] < 0)
    ref_o, _ = oracle.msa_attention(inp.np("kv_pool"), inp.k_scale, inp.v_scale, inp.np("block_table"),
                                    inp.np("row_req"), inp.np("row_ctx"), inp.np("q"), inp.q_scale,
                                    blocks.cpu().numpy(), SM_SCALE)
    assert np.abs(out.cpu().numpy() - ref_o).max() <= 2e-2
