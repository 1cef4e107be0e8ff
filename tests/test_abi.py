"""The C-ABI library loads and exports every entry point include/dsa.h
declares; host-side argument checks reject bad calls before any launch.
No test here needs a GPU: every call below fails validation on the host
(or is pure host logic), so no CUDA context is created."""
import ctypes
import os
import re

import pytest

from prefill_dsa_indexer_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    import prefill_dsa_indexer_gb300 as P
    return P.load_library()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "dsa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w]+\s*\*?\s*(dsa_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_layer_calls():
    names = declared_functions()
    for n in ("dsa_indexer_logits", "dsa_topk", "dsa_page_to_slot", "dsa_sparse_mla_decode", "dsa_sparse_mla_prefill"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n


def test_python_binding_names_match_the_abi():
    import prefill_dsa_indexer_gb300 as P
    for n in declared_functions():
        if n in ("dsa_version", "dsa_status_string"):
            continue
        assert hasattr(P, n[len("dsa_"):]), n
    assert set(P.EXPORTED) == set(declared_functions())


def test_status_strings_and_version(lib):
    assert lib.dsa_version() >= 100
    for code in range(-7, 1):
        assert lib.dsa_status_string(code).decode() not in ("", "unknown status")
    assert lib.dsa_status_string(-99).decode() == "unknown status"


def test_workspace_size_is_host_logic(lib):
    # 2048 tokens split 128 per CTA -> 16 partial outputs of 96 x 512 fp16, (max, sum) per head
    # in fp32, and each row's query as 96 x 576 fp16
    got = lib.dsa_sparse_mla_workspace_size(4, 96, 2048)
    assert got >= 4 * 16 * 96 * 512 * 2 + 4 * 16 * 96 * 2 * 4 + 4 * 96 * 576 * 2
    assert lib.dsa_sparse_mla_workspace_size(4, 96, 128) == 0  # one split: no workspace
    assert lib.dsa_sparse_mla_workspace_size(4, 96, 129) > 0
    assert lib.dsa_sparse_mla_workspace_size(0, 96, 2048) == 0


def test_host_validation_rejects_before_launch(lib):
    import prefill_dsa_indexer_gb300 as P
    fake = ctypes.c_void_p(0x10000)
    # top-k: k outside [1, 2048]
    assert lib.dsa_topk(fake, 4096, fake, 1, 4096, 0, fake, None, None, 0, None) == P.ERR_UNSUPPORTED
    assert lib.dsa_topk(fake, 4096, fake, 1, 4096, 4096, fake, None, None, 0, None) == P.ERR_UNSUPPORTED
    # top-k: logits stride shorter than max_ctx
    assert lib.dsa_topk(fake, 100, fake, 1, 4096, 16, fake, None, None, 0, None) == P.ERR_INVALID_ARG
    # top-k: nothing to do
    assert lib.dsa_topk(None, 0, None, 0, 0, 16, None, None, None, 0, None) == P.OK
    # indexer: unsupported page size, rows_per_group, bt too narrow, null cache
    c = P._Cache(fake, P.KEY_FP8, 32, 10, 1.0)
    r = P._Rows(fake, 1, 1, fake, fake, 1, 64, 1)
    assert lib.dsa_indexer_logits(ctypes.byref(c), ctypes.byref(r), fake, fake, fake, 64, None, None) == P.ERR_UNSUPPORTED
    c = P._Cache(fake, P.KEY_FP8, 64, 10, 1.0)
    r = P._Rows(fake, 1, 1, fake, fake, 3, 64, 3)
    assert lib.dsa_indexer_logits(ctypes.byref(c), ctypes.byref(r), fake, fake, fake, 64, None, None) == P.ERR_UNSUPPORTED
    r = P._Rows(fake, 1, 1, fake, fake, 1, 4096, 1)
    assert lib.dsa_indexer_logits(ctypes.byref(c), ctypes.byref(r), fake, fake, fake, 4096, None, None) == P.ERR_INVALID_ARG
    assert lib.dsa_indexer_logits(None, ctypes.byref(r), fake, fake, fake, 4096, None, None) == P.ERR_INVALID_ARG
    # sparse MLA: head count not a multiple of 16 / too many heads; decode without workspace
    lc = P._Cache(fake, P.LATENT_FP8, 64, 10, 0.01)
    for H in (8, 100, 128):
        assert lib.dsa_sparse_mla_decode(ctypes.byref(lc), fake, H, fake, 1, 2048, 0.07, fake, fake, None, None, 0,
                                         None) == P.ERR_UNSUPPORTED
    assert lib.dsa_sparse_mla_decode(ctypes.byref(lc), fake, 96, fake, 1, 2048, 0.07, fake, fake, None, None, 0,
                                     None) == P.ERR_WORKSPACE
    bad = P._Cache(fake, 9, 64, 10, 0.01)
    assert lib.dsa_sparse_mla_prefill(ctypes.byref(bad), fake, 96, fake, 1, 2048, 0.07, fake, fake, None, None, 0,
                                      None) == P.ERR_UNSUPPORTED
    # no-alloc decode: shape errors get dsa_sparse_mla_decode's statuses before any scratch check
    na = lib.dsa_sparse_mla_decode_noalloc
    assert na(ctypes.byref(lc), fake, 96, fake, 8, 2049, 0.07, fake, fake, None, None) == P.ERR_UNSUPPORTED
    for H in (8, 100, 112, 128):
        assert na(ctypes.byref(lc), fake, H, fake, 1, 2048, 0.07, fake, fake, None, None) == P.ERR_UNSUPPORTED
    assert na(None, fake, 96, fake, 1, 2048, 0.07, fake, fake, None, None) == P.ERR_INVALID_ARG
    assert na(ctypes.byref(lc), fake, 96, fake, 1, 0, 0.07, fake, fake, None, None) == P.ERR_INVALID_ARG
    assert na(ctypes.byref(lc), fake, 96, fake, P.NOALLOC_MAX_ROWS + 1, 2048, 0.07, fake, fake, None,
              None) == P.ERR_WORKSPACE
    # page -> slot: k < 1
    r = P._Rows(fake, 1, 1, fake, fake, 1, 64, 1)
    assert lib.dsa_page_to_slot(ctypes.byref(r), 10, fake, 0, fake, None, None) == P.ERR_INVALID_ARG


def test_python_binding_refuses_cpu_tensors():
    import torch
    import prefill_dsa_indexer_gb300 as P
    x = torch.zeros(4, 8)
    with pytest.raises(P.DsaError):
        P.topk(x, torch.zeros(4, dtype=torch.int32), 8, 4)


def test_missing_library_raises_instead_of_falling_back(tmp_path):
    import prefill_dsa_indexer_gb300 as P
    with pytest.raises(P.DsaError):
        P.load_library(str(tmp_path / "libdsa.so"))


def test_host_validation_of_the_msa_insert_and_warm_calls(lib):
    import prefill_dsa_indexer_gb300 as P
    fake, odd = ctypes.c_void_p(0x10000), ctypes.c_void_p(0x10004)
    rows = lambda n, ctx, stride, g=1: P._Rows(fake, stride, 1, fake, fake, n, ctx, g)
    # MSA block scores: row groups of 1, 2, 4 or 8; block table, scores and alignment checked
    r = rows(3, 256, 2, 3)
    assert lib.dsa_msa_block_scores(fake, 10, ctypes.byref(r), fake, fake, 2, None, None) == P.ERR_UNSUPPORTED
    r = rows(1, 1024, 2)
    assert lib.dsa_msa_block_scores(fake, 10, ctypes.byref(r), fake, fake, 8, None, None) == P.ERR_INVALID_ARG
    r = rows(1, 256, 2)
    assert lib.dsa_msa_block_scores(fake, 10, ctypes.byref(r), fake, fake, 1, None, None) == P.ERR_INVALID_ARG
    assert lib.dsa_msa_block_scores(odd, 10, ctypes.byref(r), fake, fake, 2, None, None) == P.ERR_INVALID_ARG
    assert lib.dsa_msa_block_scores(fake, 10, ctypes.byref(rows(0, 256, 2)), fake, fake, 2, None, None) == P.OK
    # MSA selection: counts, score stride, the shared-memory bound on blocks per row
    assert lib.dsa_msa_select(fake, 2, fake, -1, 256, fake, None, None) == P.ERR_INVALID_ARG
    assert lib.dsa_msa_select(fake, 1, fake, 1, 256, fake, None, None) == P.ERR_INVALID_ARG
    assert lib.dsa_msa_select(fake, 1 << 20, fake, 1, (1 << 21) + 128, fake, None, None) == P.ERR_UNSUPPORTED
    assert lib.dsa_msa_select(None, 0, None, 0, 0, None, None, None) == P.OK
    # MSA attention: heads per group a multiple of 16 in [16, 64]; positive finite scales; workspace
    r = rows(1, 256, 2)
    for hpg in (8, 24, 80):
        assert lib.dsa_msa_attention(fake, 10, 1.0, 1.0, ctypes.byref(r), fake, 1.0, hpg, fake, 0.09, fake, fake,
                                     fake, 1 << 30, None, None) == P.ERR_UNSUPPORTED
    assert lib.dsa_msa_attention(fake, 10, 0.0, 1.0, ctypes.byref(r), fake, 1.0, 16, fake, 0.09, fake, fake,
                                 fake, 1 << 30, None, None) == P.ERR_INVALID_ARG
    assert lib.dsa_msa_attention(fake, 10, 1.0, 1.0, ctypes.byref(r), fake, 1.0, 16, fake, 0.09, fake, fake,
                                 None, 0, None, None) == P.ERR_WORKSPACE
    # cache insert: page size, formats, matching pools, a positive latent scale
    ic, lc = P._Cache(fake, P.KEY_FP8, 64, 10, 1.0), P._Cache(fake, P.LATENT_FP8, 64, 10, 0.01)
    assert lib.dsa_cache_insert(ctypes.byref(P._Cache(fake, P.KEY_FP8, 32, 10, 1.0)), ctypes.byref(lc), fake, 1,
                                fake, fake, None, None) == P.ERR_UNSUPPORTED
    assert lib.dsa_cache_insert(ctypes.byref(P._Cache(fake, P.LATENT_FP8, 64, 10, 1.0)), ctypes.byref(lc), fake, 1,
                                fake, fake, None, None) == P.ERR_UNSUPPORTED
    assert lib.dsa_cache_insert(ctypes.byref(ic), ctypes.byref(P._Cache(fake, P.LATENT_FP8, 64, 11, 0.01)), fake,
                                1, fake, fake, None, None) == P.ERR_INVALID_ARG
    assert lib.dsa_cache_insert(ctypes.byref(ic), ctypes.byref(P._Cache(fake, P.LATENT_FP8, 64, 10, 0.0)), fake,
                                1, fake, fake, None, None) == P.ERR_INVALID_ARG
    assert lib.dsa_cache_insert(ctypes.byref(ic), ctypes.byref(lc), fake, 0, fake, fake, None, None) == P.OK
    # warm top-k: needs the latent pool, and only FP8 / NVFP4 latent formats
    r = rows(1, 4096, 64)
    assert lib.dsa_topk_slots_warm(fake, 4096, ctypes.byref(r), None, 16, fake, fake, None, None, 0,
                                   None) == P.ERR_INVALID_ARG
    assert lib.dsa_topk_slots_warm(fake, 4096, ctypes.byref(r), ctypes.byref(P._Cache(fake, 9, 64, 10, 0.01)), 16,
                                   fake, fake, None, None, 0, None) == P.ERR_UNSUPPORTED
    # the histogram top-k's workspace: none for short rows or many rows (or without a device)
    assert lib.dsa_topk_workspace_size(8, 8192, 2048) == 0
    assert lib.dsa_topk_workspace_size(65, 131072, 2048) == 0
    assert lib.dsa_topk_workspace_size(0, 131072, 2048) == 0
