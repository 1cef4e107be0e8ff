"""dsa_sparse_mla_decode_noalloc against the oracle and against dsa_sparse_mla_decode.

The no-alloc variant serves callers that cannot allocate device memory (a
host framework that has reserved the device's memory for its own pools, a
plugin that only sees the tensors it is handed, a latency-critical loop that
must not call cudaMalloc): its split-K scratch lives in a fixed array inside
the library instead of a caller workspace.

Each call is checked against the CPU oracle at the attention tolerances
(max-abs 2e-2, rel-L2 1e-2 for FP8 latents, 3e-2 for NVFP4; lse within
2e-3), and bit for bit against dsa_sparse_mla_decode with a caller
workspace: both run the same kernels on the same inputs, so any difference
would come from the shared scratch.  Two calls run in a row; a larger call
leaves the scratch dirty before a smaller one; k <= 128 uses no scratch.

This file is collected last so a run that stops at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
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


def _case(seed, ctx, lat=I.LATENT_FP8, k=2048):
    wl = I.small_workload("noalloc", ctx, lat_fmt=lat, seed=seed, k=k)
    inp = U.gpu_inputs(wl)
    rng = np.random.default_rng(seed)
    rc, bt, rq = inp.np("row_ctx"), inp.np("block_table"), inp.np("row_req")
    idx = np.full((len(rc), k), -1, dtype=np.int32)
    for r, L in enumerate(rc):
        n = min(k, L)
        idx[r, :n] = np.sort(rng.choice(L, size=n, replace=False))
    slots = oracle.page_to_slot(bt, rq, idx)
    return wl, inp, slots


def _noalloc(inp, lat, slots_dev):
    R, H = inp.q_mla.shape[0], inp.q_mla.shape[1]
    out = torch.full((R, H, 512), float("nan"), device="cuda")
    lse = torch.full((R, H), float("nan"), device="cuda")
    st = P.new_status()
    P.sparse_mla_decode_noalloc(inp.lat_pool, lat, inp.tensor_scale, inp.q_mla, slots_dev, out, lse, status=st)
    torch.cuda.synchronize()
    P.check_status(st)
    return out, lse


def _check_against_oracle(inp, lat, slots, out, lse):
    ref_o, ref_l = oracle.sparse_mla(inp.np("lat_pool"), U.ORACLE_FMT[lat], inp.tensor_scale, inp.np("q_mla"), slots,
                                     U.SM_SCALE)
    tol = 3e-2 if lat == I.LATENT_NVFP4 else 1e-2
    max_abs, rel = U.mla_errors(out.cpu().numpy(), ref_o)
    assert max_abs <= 2e-2 and rel <= tol, (max_abs, rel)
    gl = lse.cpu().numpy()
    assert np.array_equal(np.isneginf(gl), np.isneginf(ref_l))
    fin = np.isfinite(ref_l)
    assert np.all(np.abs(gl[fin] - ref_l[fin]) <= 2e-3)


CASES = {
    "fp8_8rows": (41, [3000, 5000, 2100, 70, 2600, 4400, 3900, 2048], I.LATENT_FP8, 2048),
    "nvfp4_2rows": (42, [3000, 2500], I.LATENT_NVFP4, 2048),
    "fp8_k100_no_scratch": (44, [3000, 90, 400], I.LATENT_FP8, 100),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_noalloc_matches_oracle_and_decode_on_two_calls_in_a_row(case):
    seed, ctx, lat, k = CASES[case]
    wl, inp, slots = _case(seed, ctx, lat, k)
    sd = torch.from_numpy(slots).cuda()
    ref_o, ref_l = P.sparse_mla_decode(inp.lat_pool, lat, inp.tensor_scale, inp.q_mla, sd)
    torch.cuda.synchronize()
    for _ in range(2):
        out, lse = _noalloc(inp, lat, sd)
        _check_against_oracle(inp, lat, slots, out, lse)
        assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)


def test_noalloc_after_a_larger_call_left_the_scratch_dirty():
    big_wl, big, big_slots = _case(45, [4000] * P.NOALLOC_MAX_ROWS)
    _noalloc(big, I.LATENT_FP8, torch.from_numpy(big_slots).cuda())
    wl, inp, slots = _case(46, [3500, 2200], I.LATENT_FP8)
    sd = torch.from_numpy(slots).cuda()
    out, lse = _noalloc(inp, I.LATENT_FP8, sd)
    _check_against_oracle(inp, I.LATENT_FP8, slots, out, lse)
    ref_o, ref_l = P.sparse_mla_decode(inp.lat_pool, I.LATENT_FP8, inp.tensor_scale, inp.q_mla, sd)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)


def test_noalloc_rejects_more_rows_than_its_scratch_holds():
    wl, inp, slots = _case(43, [3000] * (P.NOALLOC_MAX_ROWS + 1))
    out = torch.empty((wl.num_rows, wl.heads, 512), device="cuda")
    lse = torch.empty((wl.num_rows, wl.heads), device="cuda")
    with pytest.raises(P.DsaError, match="workspace"):
        P.sparse_mla_decode_noalloc(inp.lat_pool, I.LATENT_FP8, inp.tensor_scale, inp.q_mla,
                                    torch.from_numpy(slots).cuda(), out, lse)
