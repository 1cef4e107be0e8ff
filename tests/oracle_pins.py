"""Pins of the CPU oracle against facts that do not come from the oracle.

Each ``pin_*`` function takes a loaded oracle library (so the planted-mistake
test can hand it a deliberately broken build) and raises AssertionError when
the oracle disagrees with:

* library routines (torch's float8_e4m3fn and bfloat16 decoders, numpy
  matmul/softmax/argsort),
* the pages' printed figures (tests/golden/*.txt, each with its source),
* brute force on tiny inputs, written independently here,
* closed forms and invariants of the method (one-hot head weights, k >= L
  giving dense attention, a single selected token, equal scores, paging
  and head-padding invariance).
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch

import oracle
from prefill_dsa_indexer_gb300 import inputs as I

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# ------------------------------------------------------- independent decoders

def ref_e4m3(codes) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8))
    return t.view(torch.float8_e4m3fn).to(torch.float64).numpy()


E2M1 = np.array([float(v) for _, v in _golden("e2m1_values.txt")])


def ref_e8m0(codes) -> np.ndarray:
    c = np.asarray(codes, dtype=np.int64)
    return np.where(c == 255, np.nan, np.ldexp(1.0, (c - 127).astype(np.int32)))


def _unpack(packed) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 15
    out[..., 1::2] = p >> 4
    return out


def ref_index_keys(pool, fmt, slots):
    """Decode index keys of physical slots -> (k [n,128] f64, scale [n])."""
    pool = np.asarray(pool)
    pages, j = slots // 64, slots % 64
    if fmt == I.KEY_FP8:
        codes = pool[:, :64 * 128].reshape(-1, 64, 128)[pages, j]
        sc = pool[:, 64 * 128:].copy().view(np.float32).reshape(-1, 64)[pages, j].astype(np.float64)
        return ref_e4m3(codes), sc
    codes = _unpack(pool[:, :64 * 64].reshape(-1, 64, 64)[pages, j])
    e = pool[:, 64 * 64:].reshape(-1, 64, 4)[pages, j]
    k = E2M1[codes] * np.repeat(ref_e8m0(e), 32, axis=-1)
    return k, np.ones(len(slots))


def ref_latents(pool, fmt, tensor_scale, slots):
    pool = np.asarray(pool)
    pages, j = slots // 64, slots % 64
    if fmt == I.LATENT_FP8:
        return ref_e4m3(pool.reshape(-1, 64, 576)[pages, j]) * tensor_scale
    codes = _unpack(pool[:, :64 * 256].reshape(-1, 64, 256)[pages, j])
    sc = ref_e4m3(pool[:, 64 * 256:64 * 288].reshape(-1, 64, 32)[pages, j])
    rope = ref_e4m3(pool[:, 64 * 288:].reshape(-1, 64, 64)[pages, j]) * tensor_scale
    return np.concatenate([E2M1[codes] * np.repeat(sc, 16, axis=-1), rope], axis=-1)


def ref_bf16(bits) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16))
    return t.view(torch.bfloat16).to(torch.float64).numpy()


# ------------------------------------------------------------- brute force

def brute_logits(inp: I.Inputs):
    """sum_h w_h * relu(s_t * q_h . k_t), numpy float64."""
    bt, rq, rc = inp.np("block_table"), inp.np("row_req"), inp.np("row_ctx")
    q = ref_e4m3(inp.np("q_idx"))
    w = inp.np("head_w").astype(np.float64)
    out = np.full((len(rc), int(rc.max())), np.nan)
    for r in range(len(rc)):
        t = np.arange(rc[r])
        slots = bt[rq[r], t // 64].astype(np.int64) * 64 + t % 64
        k, s = ref_index_keys(inp.np("idx_pool"), inp.wl.key_fmt, slots)
        a = (q[r] @ k.T) * s[None, :]
        out[r, :rc[r]] = (w[r][:, None] * np.maximum(a, 0.0)).sum(axis=0)
    return out


def brute_topk(vals, n, k):
    v = np.asarray(vals[:n], dtype=np.float64)
    order = np.lexsort((np.arange(n), -v))
    sel = np.sort(order[:min(k, n)]).astype(np.int32)
    return np.concatenate([sel, -np.ones(k - len(sel), dtype=np.int32)])


def dense_attention(q, kv, sm_scale):
    """q [H,576], kv [n,576] -> (O [H,512], lse [H]) with numpy softmax."""
    s = (q @ kv.T) * sm_scale
    m = s.max(axis=1, keepdims=True)
    p = np.exp(s - m)
    l = p.sum(axis=1, keepdims=True)
    return (p / l) @ kv[:, :512], (m + np.log(l))[:, 0]


def _tiny(fmt_key=I.KEY_FP8, fmt_lat=I.LATENT_FP8, ctx=(150, 77), rows=1, heads=8, seed=3):
    wl = I.small_workload("tiny", list(ctx), rows_per_req=rows, rows_per_group=rows, key_fmt=fmt_key,
                          lat_fmt=fmt_lat, k=64, heads=heads, seed=seed)
    return I.make_inputs(wl)


# -------------------------------------------------------------------- pins

def pin_e4m3(lib):
    ref = ref_e4m3(np.arange(256, dtype=np.uint8))
    got = np.array([oracle.e4m3_decode(c, lib) for c in range(256)])
    assert np.array_equal(np.isnan(got), np.isnan(ref)), "e4m3 NaN codes"
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok]), "e4m3 values"
    assert np.array_equal(np.signbit(got[ok]), np.signbit(ref[ok])), "e4m3 signs"


def pin_e2m1(lib):
    got = np.array([oracle.e2m1_decode(c, lib) for c in range(16)])
    assert np.array_equal(got, E2M1) and np.array_equal(np.signbit(got), np.signbit(E2M1)), "e2m1 table"


def pin_e8m0(lib):
    for code, val in _golden("e8m0_semantics.txt"):
        got = oracle.e8m0_decode(int(code, 16), lib)
        if val == "nan":
            assert math.isnan(got), code
        else:
            assert got == 2.0 ** int(val), (code, got)
    allc = np.array([oracle.e8m0_decode(c, lib) for c in range(256)])
    ref = ref_e8m0(np.arange(256))
    assert np.array_equal(np.isnan(allc), np.isnan(ref)) and np.array_equal(allc[:255], ref[:255])


def pin_bf16(lib):
    rng = np.random.default_rng(5)
    bits = np.concatenate([rng.integers(0, 1 << 16, 2000), [0, 0x8000, 0x3F80, 0x7F7F, 0x0001]]).astype(np.uint16)
    ref = ref_bf16(bits)
    got = np.array([oracle.bf16_decode(int(b), lib) for b in bits])
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok]) and np.array_equal(np.isnan(got), np.isnan(ref))


def pin_byte_widths(lib):
    g = {k: float(v) for k, v in _golden("byte_widths.txt")}
    assert oracle.index_page_bytes(oracle.KEY_FP8, lib) == 64 * g["index_fp8"]
    assert oracle.index_page_bytes(oracle.KEY_MXFP4, lib) == 64 * g["index_mxfp4"]
    assert oracle.latent_page_bytes(oracle.LATENT_FP8, lib) == 64 * g["latent_fp8"]
    assert oracle.latent_page_bytes(oracle.LATENT_NVFP4, lib) == 64 * g["latent_nvfp4"]
    # the generator's layouts agree with the oracle's
    assert I.index_page_bytes(I.KEY_FP8) == oracle.index_page_bytes(oracle.KEY_FP8, lib)
    assert I.index_page_bytes(I.KEY_MXFP4) == oracle.index_page_bytes(oracle.KEY_MXFP4, lib)
    assert I.latent_page_bytes(I.LATENT_FP8) == oracle.latent_page_bytes(oracle.LATENT_FP8, lib)
    assert I.latent_page_bytes(I.LATENT_NVFP4) == oracle.latent_page_bytes(oracle.LATENT_NVFP4, lib)
    # derived figures: MXFP4 saving and the long-context DSA byte fraction
    assert round(100 * (1 - g["index_mxfp4"] / g["index_fp8"]), 1) == g["mxfp4_index_saving_pct"]
    L = 1 << 30
    frac = (g["index_fp8"] * L + g["latent_fp8"] * 2048) / (g["latent_fp8"] * L)
    assert round(100 * frac) == g["dsa_fraction_long_ctx_pct"]
    # 2048 candidates: 8 B (fp32 score + int32 id) vs 4 B (score only)
    assert g["candidates"] * 8 / 1024 == g["candidate_exchange_kib_before"]
    assert g["candidates"] * 4 / 1024 == g["candidate_exchange_kib_after"]


def pin_indexer_bruteforce(lib, fmt=I.KEY_FP8):
    inp = _tiny(fmt_key=fmt, ctx=(150, 77, 64, 1), seed=11)
    got = oracle.indexer_logits(inp.np("idx_pool"), fmt, inp.np("block_table"), inp.np("row_req"),
                                inp.np("row_ctx"), inp.np("q_idx"), inp.np("head_w"), lib=lib)
    ref = brute_logits(inp)
    assert np.array_equal(np.isnan(got), np.isnan(ref)), "causal extent"
    ok = ~np.isnan(ref)
    np.testing.assert_allclose(got[ok], ref[ok], rtol=1e-12, atol=0)


def pin_indexer_special_cases(lib):
    inp = _tiny(ctx=(200,), seed=12)
    w = np.zeros((1, 32), dtype=np.float32)
    w[0, 5] = 1.0
    got = oracle.indexer_logits(inp.np("idx_pool"), 1, inp.np("block_table"), inp.np("row_req"),
                                inp.np("row_ctx"), inp.np("q_idx"), w, lib=lib)[0]
    t = np.arange(200)
    slots = inp.np("block_table")[0, t // 64].astype(np.int64) * 64 + t % 64
    k, s = ref_index_keys(inp.np("idx_pool"), 1, slots)
    q5 = ref_e4m3(inp.np("q_idx")[0, 5])
    assert np.array_equal(got, np.maximum(s * (k @ q5), 0.0)), "one-hot head weight"
    # negating the query flips every dot: relu keeps exactly the other half
    q_neg = inp.np("q_idx").copy() ^ np.uint8(0x80)
    got_n = oracle.indexer_logits(inp.np("idx_pool"), 1, inp.np("block_table"), inp.np("row_req"),
                                  inp.np("row_ctx"), q_neg, w, lib=lib)[0]
    assert np.array_equal(got_n, np.maximum(-s * (k @ q5), 0.0)), "sign of the dot"
    assert np.all((got == 0) | (got_n == 0)), "relu: a dot and its negation cannot both survive"


def pin_indexer_paging_invariance(lib):
    a = _tiny(ctx=(300, 130), seed=13)
    # same values, different physical pages: rebuild the pools under a permutation
    perm = np.random.default_rng(1).permutation(a.num_pages).astype(np.int32)
    inv = np.argsort(perm)
    pool_b = a.np("idx_pool")[inv]           # page p moves to perm[p]
    bt_b = perm[a.np("block_table")]
    la = oracle.indexer_logits(a.np("idx_pool"), 1, a.np("block_table"), a.np("row_req"), a.np("row_ctx"),
                               a.np("q_idx"), a.np("head_w"), lib=lib)
    lb = oracle.indexer_logits(pool_b, 1, bt_b, a.np("row_req"), a.np("row_ctx"), a.np("q_idx"),
                               a.np("head_w"), lib=lib)
    assert np.array_equal(la, lb, equal_nan=True), "paging invariance"


def pin_topk(lib):
    rng = np.random.default_rng(21)
    n_rows, width, k = 6, 500, 64
    vals = rng.integers(-20, 20, size=(n_rows, width)).astype(np.float32) / 4  # many ties
    vals[1] = 0.0
    vals[1, ::7] = -0.0                                                        # signed zeros tie
    ctx = np.array([500, 500, 64, 63, 1, 0], dtype=np.int32)
    got = oracle.topk_f32(vals, ctx, k, lib=lib)
    for r in range(n_rows):
        assert np.array_equal(got[r], brute_topk(vals[r], ctx[r], k)), r
    assert np.array_equal(got[1], np.arange(k)), "ties go to the lower index"
    assert np.array_equal(got[3, :63], np.arange(63)) and np.all(got[3, 63:] == -1), "k >= L returns all"
    got64 = oracle.topk_f64(vals.astype(np.float64), ctx, k, lib=lib)
    assert np.array_equal(got, got64)


def pin_page_to_slot(lib):
    bt = np.array([[5, 2, 9], [7, 0, 3]], dtype=np.int32)
    idx = np.array([[0, 63, 64, 130, -1], [1, 70, 191, -1, -1]], dtype=np.int32)
    got = oracle.page_to_slot(bt, np.array([0, 1], dtype=np.int32), idx, lib=lib)
    want = np.array([[320, 383, 128, 578, -1], [449, 6, 255, -1, -1]], dtype=np.int32)
    assert np.array_equal(got, want)


def _mla_case(lib, fmt=I.LATENT_FP8, seed=31, n_sel=40, heads=8):
    inp = _tiny(fmt_lat=fmt, ctx=(150,), heads=heads, seed=seed)
    rng = np.random.default_rng(seed)
    t = np.sort(rng.choice(150, size=n_sel, replace=False))
    slots = inp.np("block_table")[0, t // 64].astype(np.int64) * 64 + t % 64
    sl = np.full((1, 64), -1, dtype=np.int32)
    sl[0, :n_sel] = slots
    return inp, sl, slots


def pin_mla_dense_restricted(lib, fmt=I.LATENT_FP8):
    inp, sl, slots = _mla_case(lib, fmt)
    sm = 1 / math.sqrt(192)
    out, lse = oracle.sparse_mla(inp.np("lat_pool"), fmt, inp.tensor_scale, inp.np("q_mla"), sl, sm, lib=lib)
    kv = ref_latents(inp.np("lat_pool"), fmt, inp.tensor_scale, slots)
    o_ref, lse_ref = dense_attention(ref_bf16(inp.np("q_mla")[0]), kv, sm)
    np.testing.assert_allclose(out[0], o_ref, rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(lse[0], lse_ref, rtol=1e-12, atol=1e-12)


def pin_mla_full_selection_is_dense_causal(lib):
    # k >= L: the selection is every visible token -> dense causal MLA
    inp = _tiny(ctx=(100,), heads=4, seed=33)
    logits = oracle.indexer_logits(inp.np("idx_pool"), 1, inp.np("block_table"), inp.np("row_req"),
                                   inp.np("row_ctx"), inp.np("q_idx"), inp.np("head_w"), lib=lib)
    idx = oracle.topk_f64(logits, inp.np("row_ctx"), 128, lib=lib)
    assert np.array_equal(idx[0, :100], np.arange(100)) and np.all(idx[0, 100:] == -1)
    sl = oracle.page_to_slot(inp.np("block_table"), inp.np("row_req"), idx, lib=lib)
    sm = 1 / math.sqrt(192)
    out, _ = oracle.sparse_mla(inp.np("lat_pool"), 3, inp.tensor_scale, inp.np("q_mla"), sl, sm, lib=lib)
    t = np.arange(100)
    slots = inp.np("block_table")[0, t // 64].astype(np.int64) * 64 + t % 64
    kv = ref_latents(inp.np("lat_pool"), 3, inp.tensor_scale, slots)
    o_ref, _ = dense_attention(ref_bf16(inp.np("q_mla")[0]), kv, sm)
    np.testing.assert_allclose(out[0], o_ref, rtol=1e-9, atol=1e-12)


def pin_mla_closed_forms(lib):
    inp, sl, slots = _mla_case(lib, seed=35)
    sm = 1 / math.sqrt(192)
    kv = ref_latents(inp.np("lat_pool"), 3, inp.tensor_scale, slots)
    one = np.full_like(sl, -1)
    one[0, 0] = sl[0, 3]
    out, lse = oracle.sparse_mla(inp.np("lat_pool"), 3, inp.tensor_scale, inp.np("q_mla"), one, sm, lib=lib)
    assert np.array_equal(out[0], np.broadcast_to(kv[3, :512], out[0].shape)), "single token -> its latent"
    s3 = ref_bf16(inp.np("q_mla")[0]) @ kv[3] * sm
    np.testing.assert_allclose(lse[0], s3, rtol=1e-12, atol=1e-12)
    zq = np.zeros_like(inp.np("q_mla"))
    out, lse = oracle.sparse_mla(inp.np("lat_pool"), 3, inp.tensor_scale, zq, sl, sm, lib=lib)
    np.testing.assert_allclose(out[0], np.broadcast_to(kv[:, :512].mean(axis=0), out[0].shape), rtol=1e-12,
                               atol=1e-14)
    np.testing.assert_allclose(lse[0], np.log(len(slots)), rtol=1e-12)
    empty = np.full_like(sl, -1)
    out, lse = oracle.sparse_mla(inp.np("lat_pool"), 3, inp.tensor_scale, inp.np("q_mla"), empty, sm, lib=lib)
    assert np.all(out == 0) and np.all(np.isneginf(lse)), "empty selection"


def pin_mla_invariances(lib):
    inp, sl, slots = _mla_case(lib, seed=37, heads=6)
    sm = 1 / math.sqrt(192)
    q = inp.np("q_mla")
    out, lse = oracle.sparse_mla(inp.np("lat_pool"), 3, inp.tensor_scale, q, sl, sm, lib=lib)
    # head padding: adding heads leaves the original heads bit-identical
    qpad = np.concatenate([q, np.zeros((1, 2, 576), dtype=np.uint16)], axis=1)
    out_p, lse_p = oracle.sparse_mla(inp.np("lat_pool"), 3, inp.tensor_scale, qpad, sl, sm, lib=lib)
    assert np.array_equal(out_p[:, :6], out) and np.array_equal(lse_p[:, :6], lse)
    # selection order does not matter (up to rounding)
    perm = sl.copy()
    perm[0, :len(slots)] = sl[0, :len(slots)][::-1]
    out_r, _ = oracle.sparse_mla(inp.np("lat_pool"), 3, inp.tensor_scale, q, perm, sm, lib=lib)
    np.testing.assert_allclose(out_r, out, rtol=1e-12, atol=1e-13)


def _nearest_even(x, values, codes):
    """Brute force: the representable value closest to x; ties to the code with an even
    mantissa bit (lowest code bit 0)."""
    d = [abs(x - v) for v in values]
    best = min(d)
    cands = [c for c, dd in zip(codes, d) if dd == best]
    even = [c for c in cands if c % 2 == 0]
    return (even or cands)[0]


def pin_e4m3_encode(lib):
    rng = np.random.default_rng(17)
    xs = np.concatenate([rng.standard_normal(4000) * 50, rng.standard_normal(2000) * 1e-2,
                         rng.uniform(-460, 460, 2000)]).astype(np.float32)
    # every midpoint between neighbouring finite codes (ties) and every code value itself
    vals = ref_e4m3(np.arange(0x7F, dtype=np.uint8))
    mids = ((vals[1:] + vals[:-1]) / 2).astype(np.float32)
    xs = np.concatenate([xs, vals.astype(np.float32), mids, -mids, [0.0, -0.0]]).astype(np.float32)
    got = np.array([oracle.e4m3_encode(float(x), lib) for x in xs], dtype=np.uint8)
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, ref), "e4m3 encode vs torch cast (RNE)"
    for big in (448.0, 463.9, 464.0, 1e6, -1e6):
        assert oracle.e4m3_encode(big, lib) == (0x7E | (0x80 if big < 0 else 0)), "saturation"
    assert oracle.e4m3_encode(float("nan"), lib) == 0x7F


def pin_e2m1_encode(lib):
    mags = list(E2M1[:8])
    rng = np.random.default_rng(18)
    xs = np.concatenate([rng.uniform(-7, 7, 3000), [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, 9.0, -5.0]])
    for x in xs.astype(np.float32):
        a = min(abs(float(x)), 6.0)
        want = _nearest_even(a, mags, list(range(8))) | (8 if np.signbit(x) else 0)
        assert oracle.e2m1_encode(float(x), lib) == want, float(x)


def _bf16_bits(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(
        np.uint16)


def pin_cache_insert(lib):
    """New tokens written into each format: FP8 bytes equal torch's RNE cast of the fp32
    quotients; MXFP4/NVFP4 codes equal brute-force nearest-even choices; every written
    value decodes back within half a code step."""
    rng = np.random.default_rng(19)
    n, pages = 40, 4
    keys = _bf16_bits(rng.standard_normal((n, 128)) * rng.uniform(0.01, 10, (n, 1)))
    lats = _bf16_bits(rng.standard_normal((n, 576)))
    keys[3, :] = 0  # an all-zero key
    slots = rng.permutation(pages * 64)[:n].astype(np.int32)
    slots[5] = -1
    ts = 0.0123
    kf = ref_bf16(keys).astype(np.float32)
    xf = ref_bf16(lats).astype(np.float32)
    for kfmt, lfmt in ((oracle.KEY_FP8, oracle.LATENT_FP8), (oracle.KEY_MXFP4, oracle.LATENT_NVFP4)):
        ip0 = np.zeros((pages, oracle.index_page_bytes(kfmt, lib)), np.uint8)
        lp0 = np.zeros((pages, oracle.latent_page_bytes(lfmt, lib)), np.uint8)
        ip, lp = oracle.cache_insert(ip0, kfmt, lp0, lfmt, ts, slots, keys, lats, lib=lib)
        ok = slots >= 0
        sl = slots[ok]
        if kfmt == oracle.KEY_FP8:
            amax = np.abs(kf[ok]).max(axis=1)
            sc = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
            want = torch.from_numpy((kf[ok] / sc[:, None]).astype(np.float32)).to(torch.float8_e4m3fn).view(
                torch.uint8).numpy()
            codes = ip[:, :64 * 128].reshape(-1, 64, 128)[sl // 64, sl % 64]
            got_sc = ip[:, 64 * 128:].copy().view(np.float32).reshape(-1, 64)[sl // 64, sl % 64]
            assert np.array_equal(codes, want) and np.array_equal(got_sc, sc), "FP8 key insert"
            wantl = torch.from_numpy((xf[ok] / np.float32(ts)).astype(np.float32)).to(torch.float8_e4m3fn).view(
                torch.uint8).numpy()
            assert np.array_equal(lp.reshape(-1, 64, 576)[sl // 64, sl % 64], wantl), "FP8 latent insert"
        else:
            k, _ = ref_index_keys(ip, kfmt, sl.astype(np.int64))
            e = ip[:, 64 * 64:].reshape(-1, 64, 4)[sl // 64, sl % 64].astype(np.int64)
            for t in range(len(sl)):
                for b in range(4):
                    blk = kf[ok][t, 32 * b:32 * b + 32].astype(np.float64)
                    am = np.abs(blk).max()
                    E = 0 if am == 0 else int(np.clip(np.floor(np.log2(am)) - 2 + 127, 0, 254))
                    assert e[t, b] == E, "MX scale"
                    step = 2.0 ** (E - 127)
                    for d in range(0, 32, 7):
                        x = blk[d] / step
                        want = _nearest_even(min(abs(x), 6.0), mags := list(E2M1[:8]), list(range(8)))
                        assert abs(k[t, 32 * b + d]) == E2M1[want] * step, "MX element"
            kv = ref_latents(lp, lfmt, ts, sl.astype(np.int64))
            scs = ref_e4m3(lp[:, 64 * 256:64 * 288].reshape(-1, 64, 32)[sl // 64, sl % 64])
            for t in range(len(sl)):
                for b in range(0, 32, 5):
                    blk = xf[ok][t, 16 * b:16 * b + 16]
                    am = np.float32(np.abs(blk).max())
                    want_sc = torch.tensor([am / np.float32(6.0)], dtype=torch.float32).to(torch.float8_e4m3fn).to(
                        torch.float64).item()
                    assert scs[t, b] == want_sc, "NV scale"
                    for d in range(16):
                        x = float(np.float32(blk[d] / np.float32(want_sc))) if want_sc > 0 else 0.0
                        want = _nearest_even(min(abs(x), 6.0), list(E2M1[:8]), list(range(8)))
                        assert abs(kv[t, 16 * b + d]) == E2M1[want] * want_sc, "NV element"
            wantr = torch.from_numpy((xf[ok][:, 512:] / np.float32(ts)).astype(np.float32)).to(
                torch.float8_e4m3fn).to(torch.float64).numpy() * ts
            assert np.array_equal(kv[:, 512:], wantr), "NVFP4 RoPE dims"


# ------------------------------------------------------------------ MSA
#
# The block-sparse variant (vLLM blog "Day-0 support for MiniMax-M3.1-Flash",
# section "MSA primer"): block scores against numpy brute force, the block
# selection against the properties that make it unique, attention against
# numpy softmax and torch's grouped-query scaled_dot_product_attention.

def _msa_inputs(ctx=(300, 2200), rows=2, hpg=4, seed=5):
    wl = I.small_msa_workload("pin", list(ctx), rows_per_req=rows, rows_per_group=rows, heads_per_group=hpg,
                              seed=seed)
    return I.make_msa_inputs(wl)


def _msa_slots(bt, req, L):
    t = np.arange(L, dtype=np.int64)
    return bt[req, t // 128].astype(np.int64) * 128 + t % 128


def ref_msa_keys(idx_pool, slots):
    return ref_e4m3(np.asarray(idx_pool).reshape(-1, 128, 128)[slots // 128, slots % 128])


def ref_msa_kv(kv_pool, slots, g, which):
    return ref_e4m3(np.asarray(kv_pool).reshape(-1, 4, 2, 128, 128)[slots // 128, g, which, slots % 128])


def pin_msa_block_scores(lib):
    inp = _msa_inputs()
    pool, bt, rq, rc, qi = (inp.np(n) for n in ("idx_pool", "block_table", "row_req", "row_ctx", "q_idx"))
    # a key just past row 0's causal edge (visible to row 1 only) that would win its block
    edge = int(_msa_slots(bt, rq[1], rc[1])[-1])
    pool = pool.copy()
    pool.reshape(-1, 128, 128)[edge // 128, edge % 128] = np.where(ref_e4m3(qi[1, 0]) > 0, 0x7E, 0xFE)
    got = oracle.msa_block_scores(pool, bt, rq, rc, qi, lib=lib)
    for r in range(len(rc)):
        L = int(rc[r])
        k = ref_msa_keys(pool, _msa_slots(bt, rq[r], L))
        s = ref_e4m3(qi[r]) @ k.T                      # [4, L]
        nb = (L + 127) // 128
        pad = np.full((4, nb * 128), -np.inf)
        pad[:, :L] = s
        want = pad.reshape(4, nb, 128).max(axis=-1)
        assert np.allclose(got[r, :, :nb], want, rtol=1e-13, atol=0), "MSA block scores"
        assert np.all(np.isnan(got[r, :, nb:])), "MSA blocks past the context"
    assert got[1, 0, 2] > 1e4 and got[0, 0, 2] < 1e3, "MSA causal edge"
    # paging invariance: the same tokens on other pages score the same
    perm = np.random.default_rng(1).permutation(pool.shape[0])
    pool2 = np.empty_like(pool)
    pool2[perm] = pool
    got2 = oracle.msa_block_scores(pool2, perm[bt].astype(np.int32), rq, rc, qi, lib=lib)
    assert np.array_equal(np.nan_to_num(got, nan=7.0), np.nan_to_num(got2, nan=7.0)), "MSA paging"


def _check_msa_selection(S, nb, sel):
    """The selection is the unique list with these properties."""
    sel = [int(b) for b in sel]
    chosen = [b for b in sel if b >= 0]
    assert sel[len(chosen):] == [-1] * (16 - len(chosen)), "MSA -1 padding"
    assert chosen == sorted(set(chosen)), "MSA ascending, distinct"
    assert len(chosen) == min(nb, 16), "MSA block count"
    if nb == 0:
        return
    assert chosen[-1] == nb - 1, "MSA recent block kept"
    key = lambda b: (-(S[b] if S[b] == S[b] else -np.inf), b)
    order = np.lexsort((np.arange(nb - 1), [key(b)[0] for b in range(nb - 1)]))
    assert sorted(chosen[:-1]) == sorted(int(b) for b in order[:len(chosen) - 1]), "MSA best others"
    others = set(chosen[:-1])
    for u in range(nb - 1):
        if u in others:
            continue
        for c in others:
            assert key(c) < key(u), "MSA dominance"


def pin_msa_select(lib):
    rng = np.random.default_rng(9)
    cases = [0, 1, 5, 16, 17, 18, 40, 129]
    R = len(cases)
    W = max(cases)
    S = rng.integers(0, 6, size=(R, 4, W)).astype(np.float64)  # many ties
    S[3, 1, :] = 2.0                                             # all equal
    S[5, 2, 16] = -50.0                                          # recent block scores worst
    S[6, 0, 7] = np.nan                                          # a NaN never beats a number
    row_ctx = np.array([c * 128 - (c % 3) * 40 if c else 0 for c in cases], dtype=np.int32)
    nbs = [(int(L) + 127) // 128 for L in row_ctx]
    for dt in (np.float64, np.float32):
        sel = oracle.msa_select(S.astype(dt), row_ctx, lib=lib)
        for r in range(R):
            for g in range(4):
                _check_msa_selection(S[r, g], nbs[r], sel[r, g])
    assert 7 not in oracle.msa_select(S, row_ctx, lib=lib)[6, 0], "MSA NaN block"


def _msa_dense(inp, r, blocks, sm_scale):
    """numpy softmax attention of row r over its selected blocks."""
    bt, rq, rc = inp.np("block_table"), inp.np("row_req"), inp.np("row_ctx")
    q = ref_e4m3(inp.np("q")[r]) * inp.q_scale
    H = q.shape[0]
    hpg = H // 4
    L = int(rc[r])
    out, lse = np.zeros((H, 128)), np.full(H, -np.inf)
    for g in range(4):
        t = np.concatenate([np.arange(b * 128, min(b * 128 + 128, L)) for b in blocks[g] if b >= 0] or
                           [np.zeros(0, np.int64)])
        if t.size == 0:
            continue
        sl = bt[rq[r], t // 128].astype(np.int64) * 128 + t % 128
        K = ref_msa_kv(inp.kv_pool.numpy(), sl, g, 0) * inp.k_scale
        V = ref_msa_kv(inp.kv_pool.numpy(), sl, g, 1) * inp.v_scale
        s = sm_scale * (q[g * hpg:(g + 1) * hpg] @ K.T)
        m = s.max(axis=1, keepdims=True)
        p = np.exp(s - m)
        out[g * hpg:(g + 1) * hpg] = (p @ V) / p.sum(axis=1, keepdims=True)
        lse[g * hpg:(g + 1) * hpg] = m[:, 0] + np.log(p.sum(axis=1))
    return out, lse


def pin_msa_attention(lib):
    inp = _msa_inputs(ctx=(300, 2200), rows=2, hpg=4)
    rc = inp.np("row_ctx")
    sc = oracle.msa_block_scores(inp.np("idx_pool"), inp.np("block_table"), inp.np("row_req"), rc,
                                 inp.np("q_idx"), lib=lib)
    blocks = oracle.msa_select(sc, rc, lib=lib)
    blocks[3, 2, :] = -1                                  # an empty group
    sm = 128 ** -0.5
    out, lse = oracle.msa_attention(inp.np("kv_pool"), inp.k_scale, inp.v_scale, inp.np("block_table"),
                                    inp.np("row_req"), rc, inp.np("q"), inp.q_scale, blocks, sm, lib=lib)
    for r in range(len(rc)):
        o, l = _msa_dense(inp, r, blocks[r], sm)
        assert np.allclose(out[r], o, rtol=1e-10, atol=1e-12) and np.allclose(lse[r], l, rtol=1e-12), "MSA attention"
    assert np.all(out[3, 8:12] == 0) and np.all(np.isneginf(lse[3, 8:12])), "MSA empty group"


def pin_msa_full_selection_is_gqa_attention(lib):
    """nb <= 16: every block is selected, so MSA is dense causal grouped-query
    attention, as torch computes it (head h reads KV head h // (H / 4))."""
    inp = _msa_inputs(ctx=(700, 2048), rows=3, hpg=4, seed=8)
    rc, H = inp.np("row_ctx"), inp.q.shape[1]
    blocks = np.full((len(rc), 4, 16), -1, np.int32)
    for r, L in enumerate(rc):
        blocks[r, :, :(L + 127) // 128] = np.arange((L + 127) // 128)
    sm = 0.09
    out, lse = oracle.msa_attention(inp.np("kv_pool"), inp.k_scale, inp.v_scale, inp.np("block_table"),
                                    inp.np("row_req"), rc, inp.np("q"), inp.q_scale, blocks, sm, lib=lib)
    bt, rq = inp.np("block_table"), inp.np("row_req")
    for r, L in enumerate(rc):
        sl = _msa_slots(bt, rq[r], int(L))
        K = np.stack([ref_msa_kv(inp.kv_pool.numpy(), sl, g, 0) for g in range(4)]) * inp.k_scale
        V = np.stack([ref_msa_kv(inp.kv_pool.numpy(), sl, g, 1) for g in range(4)]) * inp.v_scale
        q = torch.from_numpy(ref_e4m3(inp.np("q")[r]) * inp.q_scale)[None, :, None, :]
        want = torch.nn.functional.scaled_dot_product_attention(
            q, torch.from_numpy(K)[None], torch.from_numpy(V)[None], scale=sm, enable_gqa=True)[0, :, 0]
        assert np.allclose(out[r], want.numpy(), rtol=1e-9, atol=1e-12), "MSA = dense GQA attention"
    assert out.shape[1] == H


def pin_msa_closed_forms(lib):
    inp = _msa_inputs(ctx=(1, 900), rows=1, hpg=2, seed=4)
    rc = inp.np("row_ctx")
    q0 = np.zeros_like(inp.np("q"))                      # equal scores -> mean of V, lse = log n
    blocks = np.full((2, 4, 16), -1, np.int32)
    blocks[0, :, 0] = 0
    blocks[1, :, :3] = [0, 4, 7]
    out, lse = oracle.msa_attention(inp.np("kv_pool"), inp.k_scale, inp.v_scale, inp.np("block_table"),
                                    inp.np("row_req"), rc, q0, inp.q_scale, blocks, 0.1, lib=lib)
    bt, rq = inp.np("block_table"), inp.np("row_req")
    t1 = np.concatenate([np.arange(0, 128), np.arange(512, 640), np.arange(896, 900)])
    for g in range(4):
        v0 = ref_msa_kv(inp.kv_pool.numpy(), _msa_slots(bt, rq[0], 1), g, 1)[0] * inp.v_scale
        assert np.allclose(out[0, 2 * g:2 * g + 2], v0, rtol=1e-13, atol=0), "MSA single token = its value"
        sl = bt[rq[1], t1 // 128].astype(np.int64) * 128 + t1 % 128
        vm = ref_msa_kv(inp.kv_pool.numpy(), sl, g, 1).mean(axis=0) * inp.v_scale
        assert np.allclose(out[1, 2 * g:2 * g + 2], vm, rtol=1e-11, atol=1e-14), "MSA equal scores = mean"
    assert np.allclose(lse[1], np.log(len(t1)), rtol=1e-13), "MSA lse of equal scores"
    assert np.allclose(lse[0], 0.0, atol=1e-15), "MSA lse of one token"


ALL_PINS = {
    "e4m3": pin_e4m3,
    "e2m1": pin_e2m1,
    "e8m0": pin_e8m0,
    "bf16": pin_bf16,
    "byte_widths": pin_byte_widths,
    "indexer_fp8": pin_indexer_bruteforce,
    "indexer_mxfp4": lambda lib: pin_indexer_bruteforce(lib, I.KEY_MXFP4),
    "indexer_special": pin_indexer_special_cases,
    "indexer_paging": pin_indexer_paging_invariance,
    "topk": pin_topk,
    "page_to_slot": pin_page_to_slot,
    "mla_dense_fp8": pin_mla_dense_restricted,
    "mla_dense_nvfp4": lambda lib: pin_mla_dense_restricted(lib, I.LATENT_NVFP4),
    "mla_full_selection": pin_mla_full_selection_is_dense_causal,
    "mla_closed_forms": pin_mla_closed_forms,
    "mla_invariances": pin_mla_invariances,
    "e4m3_encode": pin_e4m3_encode,
    "e2m1_encode": pin_e2m1_encode,
    "cache_insert": pin_cache_insert,
    "msa_block_scores": pin_msa_block_scores,
    "msa_select": pin_msa_select,
    "msa_attention": pin_msa_attention,
    "msa_full_selection": pin_msa_full_selection_is_gqa_attention,
    "msa_closed_forms": pin_msa_closed_forms,
}
