"""The synthetic inputs follow their stated recipe: context lengths and query-row positions of
the named workloads, unshared pages drawn from a larger pool, poisoned slots that hold no
token, and FP8 scales that map each token's (or the pool's) largest magnitude to 448."""
import numpy as np

from prefill_dsa_indexer_gb300 import inputs as I
from tests import oracle_pins as pins


def test_named_workload_shapes():
    b32 = I.workload("decode_b32_16k_64k")
    assert len(b32.ctx) == 32 and all(16384 <= L <= 65536 for L in b32.ctx)
    assert np.array_equal(b32.row_ctx(), np.asarray(b32.ctx))
    for name in ("decode_b8_128k_fp8", "decode_b8_128k_fp4"):
        wl = I.workload(name)
        assert wl.ctx == [131072] * 8 and wl.rows_per_req == 1 and wl.k == 2048 and wl.heads == 96
    v = I.workload("verify_b4_256k")  # four verify rows per request, scored together
    assert v.rows_per_group == 4 and list(v.row_ctx()[:4]) == [262141, 262142, 262143, 262144]
    assert np.array_equal(v.row_req(), np.repeat(np.arange(4), 4))
    p = I.workload("prefill_8k_on_56k")  # row j sees 57,345 + j tokens
    assert np.array_equal(p.row_ctx(), 57345 + np.arange(8192))
    assert I.workload("verify_b1_1m").ctx == [1 << 20]


def test_pages_are_unshared_and_from_a_larger_pool():
    for name in ("decode_b8_128k_fp8", "decode_b32_16k_64k", "verify_b4_256k"):
        wl = I.workload(name)
        bt, total = I._paging(wl)
        used = [bt[b, :(L + 63) // 64] for b, L in enumerate(wl.ctx)]
        flat = np.concatenate(used)
        assert len(np.unique(flat)) == len(flat)  # no page serves two requests or two positions
        assert flat.min() >= 0 and flat.max() < total
        assert total == len(flat) + max(1, int(len(flat) * wl.extra_pages))


def _check_pools(wl):
    inp = I.make_inputs(wl, device="cpu")
    idx, lat, bt = inp.np("idx_pool"), inp.np("lat_pool"), inp.np("block_table")
    used = np.zeros((idx.shape[0], 64), dtype=bool)
    for b, L in enumerate(wl.ctx):
        t = np.arange(L)
        used[bt[b, t // 64], t % 64] = True
    # slots that hold no token (tail of a request's last page, free pages) carry NaN codes
    if wl.key_fmt == I.KEY_FP8:
        codes = idx[:, :64 * 128].reshape(-1, 64, 128)
        scales = idx[:, 64 * 128:].copy().view(np.float32).reshape(-1, 64)
        assert np.all(codes[~used] == 0x7F) and np.all(np.isnan(scales[~used]))
        # the per-token scale is amax / 448: every token's largest code magnitude is 448
        mags = np.abs(pins.ref_e4m3(codes[used]))
        assert np.all(mags.max(axis=1) == 448.0)
        assert np.all(scales[used] > 0)
    if wl.key_fmt == I.KEY_MXFP4:  # unused slots: NaN block scales (e8m0 0xFF)
        assert np.all(idx[:, 64 * 64:].reshape(-1, 64, 4)[~used] == 0xFF)
    if wl.lat_fmt == I.LATENT_NVFP4:  # unused slots: every byte of the three regions 0x7F
        assert np.all(lat[:, :64 * 256].reshape(-1, 64, 256)[~used] == 0x7F)
        assert np.all(lat[:, 64 * 288:].reshape(-1, 64, 64)[~used] == 0x7F)
    if wl.lat_fmt == I.LATENT_FP8:
        rows = lat.reshape(-1, 64, 576)
        assert np.all(rows[~used] == 0x7F)
        # the per-tensor scale is amax / 448 over the used pool
        assert np.abs(pins.ref_e4m3(rows[used])).max() == 448.0
        assert inp.tensor_scale > 0


def test_generated_pools_follow_the_recipe():
    _check_pools(I.small_workload("recipe_fp8", [100, 4096, 700], seed=51))
    _check_pools(I.small_workload("recipe_fp4", [300, 1000], key_fmt=I.KEY_MXFP4, lat_fmt=I.LATENT_NVFP4, seed=52))


def test_same_seed_same_inputs():
    wl = I.small_workload("seeded", [900, 2000], seed=53)
    a, b = I.make_inputs(wl, device="cpu"), I.make_inputs(wl, device="cpu")
    for n in ("idx_pool", "lat_pool", "block_table", "q_idx", "head_w", "q_mla"):
        assert np.array_equal(a.np(n), b.np(n)), n  # byte images, integers and NaN-free floats
    assert a.tensor_scale == b.tensor_scale
