"""GPU parity of the fused decode path's front end: the new tokens written into
the paged cache (latent and index key, FP8 or MXFP4) and the indexer query in
FP8 with its scale folded into the head weights, bit-exact against the oracle;
then a whole step (write, quantise, score, select, attend) against the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from dsa_sparse_attention_index_gb300 import binding, synth
from test_gpu_parity import _run_step, _status, check_mla, check_scores

pytestmark = pytest.mark.gpu


def _bf16_bits(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _new_rows(rows, seed, extreme_latents=True):
    rng = np.random.default_rng(seed)
    lat = rng.standard_normal((rows, 576)).astype(np.float32) * 2
    key = rng.standard_normal((rows, 128)).astype(np.float32) * np.exp(rng.uniform(-2, 2, (rows, 1)))
    if rows >= 4:
        key[1] = 0.0                                   # all-zero key: scale 1 / E8M0 byte 0
        key[2, 32:64] *= 1e-35                          # a block of subnormal-range values
        key[3, :3] = [-0.0, 1e30, -1e30]               # a negative zero and saturating values
        if extreme_latents:                             # saturating latent codes (+-448)
            lat[0, :4] = [1e30, -1e30, -0.0, 1e-38]
    return _bf16_bits(lat), _bf16_bits(key)


@pytest.mark.parametrize("fmt,lfmt", [(synth.KEY_FP8, synth.LATENT_FP8), (synth.KEY_MXFP4, synth.LATENT_FP8),
                                       (synth.KEY_MXFP4, synth.LATENT_NVFP4), (synth.KEY_FP8, synth.LATENT_NVFP4)])
@pytest.mark.parametrize("lens,nq", [([1000, 64, 777], 1), ([5000, 130], 4), ([3000], 64)])
def test_cache_append_matches_oracle(fmt, lfmt, lens, nq):
    case = synth.make_case("ap", seq_lens=lens, nq=nq, key_format=fmt, seed=nq + fmt, spare_blocks=2,
                           latent_format=lfmt)
    lat, key = _new_rows(case.rows, seed=len(lens) + nq)
    if lfmt == synth.LATENT_NVFP4 and case.rows >= 2:
        # NVFP4 blocks with a wide spread, an all-zero block and a tiny one
        rng = np.random.default_rng(nq)
        x = (rng.standard_normal((case.rows, 576)) * np.exp(rng.uniform(-6, 6, (case.rows, 36, 1))).repeat(16, 2)
             .reshape(case.rows, 576)).astype(np.float32)
        x[1, 32:48] = 0.0
        x[1, 48:64] *= 1e-30
        lat = _bf16_bits(x)
    ref = oracle.cache_append(case, lat, key)
    dc = synth.device_case(case)
    st = _status()
    binding.cache_append(dc.cache, dc.batch, torch.from_numpy(lat.view(np.int16)).cuda(),
                         torch.from_numpy(key.view(np.int16)).cuda(), st)
    torch.cuda.synchronize()
    assert st.item() == 0, binding.status_string(st.item())
    got = dc.cache.pool.cpu().numpy()
    bad = np.argwhere(got != ref)
    assert bad.size == 0, f"{len(bad)} bytes differ, first at (row, byte) {bad[:4].tolist()}"


def test_cache_append_reports_a_bad_block():
    case = synth.make_case("apb", seq_lens=[100], key_format=synth.KEY_FP8, seed=2)
    case.block_table[0, 1] = case.num_blocks + 5
    lat, key = _new_rows(1, seed=3)
    dc = synth.device_case(case)
    st = _status()
    binding.cache_append(dc.cache, dc.batch, torch.from_numpy(lat.view(np.int16)).cuda(),
                         torch.from_numpy(key.view(np.int16)).cuda(), st)
    torch.cuda.synchronize()
    assert st.item() == binding.ERR_BOUNDS


def test_quantize_index_query_matches_oracle():
    rng = np.random.default_rng(9)
    q = rng.standard_normal((37, 32, 128)).astype(np.float32) * np.exp(rng.uniform(-4, 4, (37, 32, 1)))
    q[0, 3] = 0.0
    q[1, 7, :2] = [1e30, -0.0]
    q_b = _bf16_bits(q)
    w = rng.standard_normal((37, 32)).astype(np.float32)
    codes_ref, w_ref = oracle.quantize_query(q_b, w)
    codes = torch.empty((37, 32, 128), dtype=torch.uint8, device="cuda")
    w_out = torch.empty((37, 32), dtype=torch.float32, device="cuda")
    binding.quantize_index_query(torch.from_numpy(q_b.view(np.int16)).cuda(), torch.from_numpy(w).cuda(), codes, w_out)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(codes.cpu().numpy(), codes_ref)
    np.testing.assert_array_equal(w_out.cpu().numpy(), w_ref)


@pytest.mark.parametrize("fmt,nq,lfmt", [(synth.KEY_FP8, 1, synth.LATENT_FP8), (synth.KEY_FP8, 4, synth.LATENT_FP8),
                                         (synth.KEY_MXFP4, 1, synth.LATENT_FP8),
                                         (synth.KEY_MXFP4, 1, synth.LATENT_NVFP4)])
def test_step_that_owns_its_cache_update(fmt, nq, lfmt):
    """Write the step's new tokens, quantise the indexer query, then run the
    fused step; every stage against the oracle on the updated cache."""
    case = synth.make_case("own", seq_lens=[9000, 4100], nq=nq, key_format=fmt, seed=31 + nq, latent_format=lfmt)
    rng = np.random.default_rng(7)
    # no saturating latents here: one selected +-448 code would make the MLA's
    # error scale with its value (the attended values' spread), not with 1e-2
    lat, key = _new_rows(case.rows, seed=12, extreme_latents=False)
    q_b = _bf16_bits(rng.standard_normal((case.rows, 32, 128)).astype(np.float32))
    w = (rng.standard_normal((case.rows, 32)) * 0.1).astype(np.float32)
    # the oracle's view: the updated pool and the quantised query
    case.pool = oracle.cache_append(case, lat, key)
    case.q_index, case.head_w = oracle.quantize_query(q_b, w)
    # the GPU's view: the original pool, updated and quantised on the device
    dc_pool = torch.from_numpy(synth.make_case("own", seq_lens=[9000, 4100], nq=nq, key_format=fmt,
                                               seed=31 + nq, latent_format=lfmt).pool).cuda()
    dc = synth.device_case(case)
    dc.cache.pool.copy_(dc_pool)
    st = _status()
    binding.cache_append(dc.cache, dc.batch, torch.from_numpy(lat.view(np.int16)).cuda(),
                         torch.from_numpy(key.view(np.int16)).cuda(), st)
    binding.quantize_index_query(torch.from_numpy(q_b.view(np.int16)).cuda(), torch.from_numpy(w).cuda(),
                                 dc.q_index, dc.head_w)
    torch.cuda.synchronize()
    assert st.item() == 0
    np.testing.assert_array_equal(dc.cache.pool.cpu().numpy(), case.pool)
    np.testing.assert_array_equal(dc.q_index.cpu().numpy(), case.q_index)
    np.testing.assert_array_equal(dc.head_w.cpu().numpy(), case.head_w)
    scores, idx, o, l = _run_step(case)
    check_scores(case, scores)
    s64 = scores.cpu().numpy().astype(np.float64)
    np.testing.assert_array_equal(idx, oracle.topk(s64, case.row_lens(), case.topk))
    check_mla(case, idx, o, l)
