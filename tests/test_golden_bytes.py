"""The byte figures the pages print, checked against the cache layout the
generator writes and against the bytes accounting the benchmark uses."""
import json
import os

import numpy as np

from dsa_sparse_attention_index_gb300 import roofline, synth

G = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "kv_bytes_per_token.json")))


def test_per_token_kv_table():
    n = G["layers"]
    lat, key = G["latent_bytes"], G["index_key_bytes"]
    tab = G["per_token_bytes_24_layers"]
    assert n * lat["fp8"] == tab["k3_fp8_latent"]
    assert n * (lat["fp8"] + key["fp8"]) == tab["k31_fp8_latent_fp8_key"]
    assert n * (lat["nvfp4"] + key["mxfp4"]) == tab["k31_nvfp4_latent_mxfp4_key"]


def test_key_and_latent_bytes_match_the_cache_layout():
    assert synth.INDEX_PAGE[synth.KEY_FP8] // synth.BLOCK == G["index_key_bytes"]["fp8"] == 128 + 4
    assert synth.INDEX_PAGE[synth.KEY_MXFP4] // synth.BLOCK == G["index_key_bytes"]["mxfp4"] == 64 + 4
    assert synth.LATENT_PAGE // synth.BLOCK == G["latent_bytes"]["fp8"] == synth.LATENT
    assert (synth.IDX_HEADS, synth.IDX_DIM, synth.MLA_HEADS) == (G["indexer_heads"], G["indexer_dim"], G["mla_heads"])
    assert round(1 - 68 / 132, 3) == G["mxfp4_index_storage_reduction"]


def test_dsa_fraction_of_dense_mla_bytes():
    k = G["topk"]
    f = [roofline.pages_fraction(L, k) for L in (4096, 32768, 131072, 1 << 20)]
    assert round(f[-1], 2) == G["dsa_over_dense_fraction_long_context"]      # ~23% at 1M
    assert abs(f[0] - 0.729) < 1e-3 and abs(f[1] - 0.292) < 1e-3 and abs(f[2] - 0.245) < 1e-3
    assert abs(roofline.pages_fraction(10 ** 12, k) - 132 / 576) < 1e-6          # -> 22.9%
    assert abs(roofline.pages_fraction(1 << 20, k, 68) - 0.120) < 1e-3


def test_step_bytes_counts_each_sequence_key_once():
    b = roofline.step_bytes([1000, 3000], nq=4, topk=2048)
    assert b["keys"] == 132 * 4000
    vis = roofline.visible_lengths([1000, 3000], 4)
    assert list(vis) == [997, 998, 999, 1000, 2997, 2998, 2999, 3000]
    assert b["latents"] == 576 * int(np.minimum(vis, 2048).sum())
    assert roofline.mla_flops([4096]) == 2 * 96 * 2048 * (576 + 512)


def test_nvfp4_latent_record_and_the_420_byte_configuration():
    """352 B NVFP4 latents: the generator's record and page, and with MXFP4
    keys a pool row of 420 B a token (24 layers: the printed 10,080 B)."""
    rec = synth.LATENT_RECORD[synth.LATENT_NVFP4]
    assert rec == G["latent_bytes"]["nvfp4"] == 512 // 2 + 512 // 16 + 64
    c = synth.make_case("nvg", seq_lens=[130], key_format=synth.KEY_MXFP4, latent_format=synth.LATENT_NVFP4, seed=1)
    assert c.row_stride == synth.BLOCK * (rec + G["index_key_bytes"]["mxfp4"])
    assert G["layers"] * c.row_stride // synth.BLOCK == G["per_token_bytes_24_layers"]["k31_nvfp4_latent_mxfp4_key"]
    assert c.row_stride % 128 == 0 and c.index_off % 128 == 0
    b = roofline.step_bytes([1000], topk=2048, key_format=1, latent_format=1)
    assert b["keys"] == 68 * 1000 and b["latents"] == 352 * 1000
