"""GPU parity of the native FP4 indexer: MXFP4 keys (64 bytes of packed E2M1
codes plus four E8M0 block scales a token) scored against an MXFP4 query by
the FP4 x FP4 block-scaled MMA (Day-0 post, MXFP4-indexer section: scoring
uses native FP4 matrix instructions with FP32 accumulation), against the fp64
oracle through the C ABI.  Same score tolerance as the other indexer paths:
|gpu - ref| <= 1e-5 * max(|ref|, A_t).  The products of E2M1 values and
power-of-two scales are exact, so the error is the fp32 accumulation alone.
"""
import numpy as np
import pytest
import torch

import oracle
from dsa_sparse_attention_index_gb300 import binding, synth
from test_gpu_parity import _run_step, _status, check_mla, check_scores, gpu_scores

pytestmark = pytest.mark.gpu

NAT = synth.KEY_MXFP4_NATIVE


@pytest.mark.parametrize("lens", [
    [4096],
    [1, 63, 64, 65, 127, 128, 129, 200, 1000, 0],
    [70001, 3000],
    [300000, 17],        # more units than the 11-stage ring, many times over
])
def test_native_index_scores_match_oracle(lens):
    case = synth.make_case("nat", seq_lens=lens, key_format=NAT, seed=len(lens) + 60, spare_blocks=2)
    check_scores(case, gpu_scores(case, synth.device_case(case)))


def _key_scale_offset(case, slot, blk):
    # index page: 64 tokens x 64 packed bytes, then 64 tokens x 4 E8M0 bytes
    return case.index_off + synth.BLOCK * (synth.IDX_DIM // 2) + 4 * slot + blk


def test_native_special_block_scales():
    """E8M0 byte 0 (2^-127), large exponents and 255 (NaN: that head's dot
    product is NaN, the ReLU drops it) on keys and on query heads.  Exponent
    pairs stay where q . k is inside the fp32 range."""
    case = synth.make_case("nats", seq_lens=[700], key_format=NAT, seed=3)
    pages = case.block_table[0]
    for (pg, slot, blk), e in {(0, 5, 0): 0, (0, 5, 3): 0, (1, 17, 2): 200, (2, 40, 1): 255, (3, 63, 0): 1,
                               (10, 2, 3): 170}.items():
        case.pool[pages[pg], _key_scale_offset(case, slot, blk)] = e
    rows = case.rows
    qe = case.q_index[rows * 32 * 64:].reshape(rows, 32, 4)   # a view into the query buffer
    qe[0, 7, 0] = 0
    qe[0, 11, 2] = 180
    check_scores(case, gpu_scores(case, synth.device_case(case)))
    # one query head's block NaN: that head drops out of every score on both
    # sides; the rounding scale A_t is that of the other heads (the NaN head's
    # bound is NaN), taken from the same query with the head's block at 2^-127
    qe[0, 3, 1] = 0
    bound = oracle.index_score_bounds(case, 704)
    qe[0, 3, 1] = 255
    s = gpu_scores(case, synth.device_case(case)).cpu().numpy()[0, :700].astype(np.float64)
    ref = oracle.index_scores(case, 704)[0, :700]
    assert not np.isnan(s).any() and not np.isnan(ref).any()
    assert (np.abs(s - ref) <= 1e-5 * np.fmax(np.abs(ref), bound[0, :700])).all()


def test_native_identity_and_permuted_tables_agree():
    a = synth.make_case("npa", seq_lens=[3000, 777], key_format=NAT, permute_blocks=False, seed=9)
    b = synth.make_case("npb", seq_lens=[3000, 777], key_format=NAT, permute_blocks=True, seed=9)
    sa = gpu_scores(a, synth.device_case(a))
    sb = gpu_scores(b, synth.device_case(b))
    assert torch.equal(sa.view(torch.int32), sb.view(torch.int32))


def test_native_several_queries_per_sequence_is_rejected():
    case = synth.make_case("natq", seq_lens=[300], nq=2, key_format=NAT, seed=1)
    dc = synth.device_case(case)
    s = torch.zeros((2, 304), dtype=torch.float32, device="cuda")
    with pytest.raises(binding.DsaError) as e:
        binding.index_scores(dc.cache, dc.batch, dc.q_index, dc.head_w, s, _status())
    assert e.value.code == binding.ERR_UNSUPPORTED


@pytest.mark.parametrize("lens", [[50000, 20000], [2048, 2049, 100]])
def test_native_decode_step_matches_oracle(lens):
    case = synth.make_case("natstep", seq_lens=lens, key_format=NAT, heavy_tail=0.1, seed=23)
    scores, idx, o, l = _run_step(case)
    check_scores(case, scores)
    s64 = scores.cpu().numpy().astype(np.float64)
    np.testing.assert_array_equal(idx, oracle.topk(s64, case.row_lens(), case.topk))
    check_mla(case, idx, o, l)
