"""The bench's byte accounting (the numerator of its roofline fraction and of the layer's GB/s),
checked on the CPU against the traffic of each query row written out term by term."""
import bench
from prefill_dsa_indexer_gb300 import inputs as I

H, K = 96, 2048


def _row_io(L):
    return (32 * 128 + 32 * 4          # indexer query (e4m3) and head weights (fp32)
            + H * 576 * 2              # MLA query (bf16)
            + H * 512 * 4 + H * 4)     # output and lse (fp32)


def _group_reads(L, key_b, lat_b):
    return (key_b * L                  # every visible index key, once per row group
            + 4 * -(-L // 64)          # its block-table entries
            + lat_b * min(L, K))       # the selected latents (the largest row's count)


def test_decode_layer_bytes_are_the_per_row_sum():
    for name in ("decode_b8_128k_fp8", "decode_b32_16k_64k", "decode_b8_128k_fp4"):
        wl = I.workload(name)
        assert wl.rows_per_group == 1
        kb, lb = I.INDEX_TOKEN_BYTES[wl.key_fmt], I.LATENT_TOKEN_BYTES[wl.lat_fmt]
        want = sum(_group_reads(int(L), kb, lb) + _row_io(int(L)) for L in wl.row_ctx())
        assert bench.layer_algorithmic_bytes(wl, kb, lb) == want, name


def test_rows_of_one_request_read_its_keys_once():
    for name in ("verify_b4_256k", "verify_b1_1m"):
        wl = I.workload(name)
        G = wl.rows_per_group
        rc = [int(x) for x in wl.row_ctx()]
        want = sum(_row_io(L) for L in rc)
        want += sum(_group_reads(max(rc[g:g + G]), 132, 576) for g in range(0, len(rc), G))
        assert bench.layer_algorithmic_bytes(wl, 132, 576) == want, name
        # the scan itself: keys and block table once per group, queries and weights and the
        # fp32 logits of every row
        scan = sum(132 * max(rc[g:g + G]) + 4 * -(-max(rc[g:g + G]) // 64) for g in range(0, len(rc), G))
        scan += len(rc) * (32 * 128 + 32 * 4) + 4 * sum(rc)
        assert bench.indexer_algorithmic_bytes(wl, 132) == scan, name


def test_headline_decode_counts():
    wl = I.workload("decode_b8_128k_fp8")
    # 8 rows of 131,072 visible tokens: 18,801,152 B per row for the layer
    assert bench.layer_algorithmic_bytes(wl, 132, 576) == 8 * 18_801_152
    assert bench.indexer_algorithmic_bytes(wl, 132) == 8 * (132 * 131072 + 4 * 2048 + 4096 + 128 + 4 * 131072)
    # MXFP4 keys (68 B) and NVFP4 latents (352 B): about 79.6 MB for the layer
    fp4 = I.workload("decode_b8_128k_fp4")
    assert bench.layer_algorithmic_bytes(fp4, 68, 352) == 79_630_336
