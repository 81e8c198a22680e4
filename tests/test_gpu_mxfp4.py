"""GPU parity of the MXFP4 indexer path (68-byte keys: 64 bytes of packed
E2M1 codes plus four E8M0 block scales per token) against the fp64 oracle,
through the C ABI.  Same score tolerance as the FP8 path:
|gpu - ref| <= 1e-5 * max(|ref|, A_t).
"""
import numpy as np
import pytest
import torch

import oracle
from dsa_sparse_attention_index_gb300 import binding, synth
from test_gpu_parity import _run_step, _status, check_mla, check_scores, gpu_scores

pytestmark = pytest.mark.gpu

MX = synth.KEY_MXFP4


@pytest.mark.parametrize("lens", [
    [4096],
    [1, 63, 64, 65, 127, 128, 129, 200, 1000, 0],
    [70001, 3000],
])
def test_mxfp4_index_scores_match_oracle(lens):
    case = synth.make_case("mx", seq_lens=lens, key_format=MX, seed=len(lens) + 40, spare_blocks=2)
    check_scores(case, gpu_scores(case, synth.device_case(case)))


def _scale_byte_offset(case, token_page_slot, blk):
    # index page: 64 tokens x 64 packed bytes, then 64 tokens x 4 E8M0 bytes
    return case.index_off + synth.BLOCK * (synth.IDX_DIM // 2) + 4 * token_page_slot + blk


def test_mxfp4_special_block_scales():
    """E8M0 byte 0 (2^-127, a subnormal fp32 scale), large exponents and 255
    (NaN: the token's head logits are NaN, ReLU drops them, score 0).  Scales
    near 2^127 are left out: such keys have scores beyond the fp32 range."""
    case = synth.make_case("mxs", seq_lens=[700], key_format=MX, seed=3)
    pages = case.block_table[0]
    planted = {(0, 5, 0): 0, (0, 5, 3): 0, (1, 17, 2): 200, (2, 40, 1): 255, (3, 63, 0): 1, (10, 2, 3): 170}
    for (pg, slot, blk), e in planted.items():
        case.pool[pages[pg], _scale_byte_offset(case, slot, blk)] = e
    s = gpu_scores(case, synth.device_case(case))
    ref = check_scores(case, s)
    got = s.cpu().numpy()
    t_nan = 2 * 64 + 40
    assert ref[0, t_nan] == 0.0 and got[0, t_nan] == 0.0
    assert not np.isnan(got[0, :700]).any()


def test_mxfp4_several_queries_per_sequence_is_rejected():
    case = synth.make_case("mxq", seq_lens=[300], nq=2, key_format=MX, seed=1)
    dc = synth.device_case(case)
    s = torch.zeros((2, 304), dtype=torch.float32, device="cuda")
    with pytest.raises(binding.DsaError) as e:
        binding.index_scores(dc.cache, dc.batch, dc.q_index, dc.head_w, s, _status())
    assert e.value.code == binding.ERR_UNSUPPORTED


def test_mxfp4_identity_and_permuted_tables_agree():
    a = synth.make_case("mpa", seq_lens=[3000, 777], key_format=MX, permute_blocks=False, seed=9)
    b = synth.make_case("mpb", seq_lens=[3000, 777], key_format=MX, permute_blocks=True, seed=9)
    sa = gpu_scores(a, synth.device_case(a))
    sb = gpu_scores(b, synth.device_case(b))
    assert torch.equal(sa.view(torch.int32), sb.view(torch.int32))


@pytest.mark.parametrize("lens", [[50000, 20000], [2048, 2049, 100]])
def test_mxfp4_decode_step_matches_oracle(lens):
    case = synth.make_case("mxstep", seq_lens=lens, key_format=MX, heavy_tail=0.1, seed=23)
    scores, idx, o, l = _run_step(case)
    check_scores(case, scores)
    s64 = scores.cpu().numpy().astype(np.float64)
    np.testing.assert_array_equal(idx, oracle.topk(s64, case.row_lens(), case.topk))
    check_mla(case, idx, o, l)
