"""NVFP4 latents (Day-0 post, packed-cache section: 352 B a token instead of
576, E2M1 with E4M3 block scales) in the sparse MLA, against the oracle:
decode rows with 2,048 and 100 selected tokens, a single token bit-exact
for every code and a spread of block scales, a fused step in the 420 B/token
configuration (MXFP4 keys), and the decode-context-parallel combine over
NVFP4 latents.  Tolerances as for E4M3 latents.
"""
import numpy as np
import pytest
import torch

import oracle
from dsa_sparse_attention_index_gb300 import synth
from test_gpu_dcp import _gpu_dcp_mla, check_dcp_mla
from test_gpu_parity import OUT_RTOL_EDGE, _gpu_mla, _run_step, check_mla, check_scores

pytestmark = pytest.mark.gpu

NV = synth.LATENT_NVFP4


@pytest.mark.parametrize("k", [2048, 100])
def test_sparse_mla_nvfp4_matches_oracle(k):
    case = synth.make_case("nvm", seq_lens=[6000, 2500, 900], nq=1, seed=41 + k, latent_format=NV)
    dc = synth.device_case(case)
    rng = np.random.default_rng(k)
    idx = np.full((3, k), -1, dtype=np.int32)
    for r, L in enumerate(case.row_lens()):
        n = min(k, int(L))
        idx[r, :n] = np.sort(rng.choice(int(L), n, replace=False))
    idx[0, 50:90] = -1
    o, l = _gpu_mla(case, dc, idx)
    check_mla(case, idx, o, l, rtol=0.0 if k == 2048 else OUT_RTOL_EDGE)


def test_sparse_mla_nvfp4_single_token_is_bit_exact():
    """One selected token: out = bf16(latent_scale * scale * e2m1) exactly,
    for every E2M1 code in both nibbles and scales from E4M3 subnormals to
    448, and the E4M3 tail codes feed only the logit."""
    case = synth.make_case("nv1", seq_lens=[700], nq=1, seed=43, latent_format=NV)
    rec = np.zeros(352, dtype=np.uint8)
    rec[:256] = [(i % 16) | (((5 * i + 2) % 16) << 4) for i in range(256)]
    rec[256:288] = [0x01, 0x02, 0x07, 0x08, 0x09, 0x30, 0x38, 0x3F, 0x40, 0x55, 0x6A, 0x7E,
                    0x81, 0x88, 0xB8, 0xFE, 0x00, 0x10, 0x20, 0x28, 0x44, 0x48, 0x50, 0x58,
                    0x60, 0x66, 0x70, 0x77, 0xC0, 0xD4, 0xE8, 0xF0]
    rec[288:] = [(3 * i + 5) % 0x7F for i in range(64)]
    r = case.block_table[0, 200 // 64]
    off = case.latent_off + (200 % 64) * 352
    case.pool[r, off:off + 352] = rec
    dc = synth.device_case(case)
    idx = np.full((1, 4), -1, dtype=np.int32)
    idx[0, 0] = 200
    o, l = _gpu_mla(case, dc, idx)
    codes = np.stack([rec[:256] & 0xF, rec[:256] >> 4], axis=1).reshape(-1)
    mag = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float32)
    e2m1 = np.where(codes & 8, np.float32(-1.0), np.float32(1.0)) * mag[codes & 7]
    scale = torch.from_numpy(rec[256:288].copy()).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    vals = torch.from_numpy((e2m1 * np.repeat(scale, 16)).astype(np.float32)) * np.float32(case.latent_scale)
    want = vals.to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(o[0], np.broadcast_to(want, (96, 512)))


@pytest.mark.parametrize("kw", [dict(seq_lens=[9000, 4100, 30000], heavy_tail=0.1),
                                dict(seq_lens=[5000, 2100], nq=4, key_format=synth.KEY_FP8)])
def test_decode_step_nvfp4_matches_oracle(kw):
    kw = dict(kw)
    kw.setdefault("key_format", synth.KEY_MXFP4)
    case = synth.make_case("nvs", seed=44, latent_format=NV, **kw)
    scores, idx, o, l = _run_step(case)
    check_scores(case, scores)
    s64 = scores.cpu().numpy().astype(np.float64)
    np.testing.assert_array_equal(idx, oracle.topk(s64, case.row_lens(), case.topk))
    check_mla(case, idx, o, l)


def test_dcp_sparse_mla_nvfp4():
    case = synth.make_case("nvd", seq_lens=[6000, 2500], nq=1, seed=45, latent_format=NV)
    dc = synth.device_case(case)
    rng = np.random.default_rng(45)
    idx = np.stack([np.sort(rng.choice(L, 2048, replace=False)) for L in (6000, 2500)]).astype(np.int32)
    o, l, po, pl = _gpu_dcp_mla(case, dc, idx, 8)
    check_dcp_mla(case, idx, 8, o, l, po, pl)
