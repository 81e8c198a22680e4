"""GPU parity of the prefill rows: a chunk of causal query rows per sequence
(row j of a sequence with context L and nq rows sees L - (nq - 1) + j tokens),
through the prefill indexer (8-row query groups against 512-key blocks on
the tensor cores), the top-k and the sparse MLA, against the fp64 oracle on
the same seeded inputs.  Tolerances as for decode.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from dsa_sparse_attention_index_gb300 import binding, synth
from test_gpu_bf16_scores import check_scores_bf16, gpu_scores_bf16
from test_gpu_parity import OUT_RTOL_EDGE, _run_step, check_mla, check_scores, gpu_scores

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("lens,nq", [
    ([5000], 64),            # 8 groups, a ragged last key block
    ([3000, 700], 8),        # one group per sequence
    ([300, 4100, 9], 12),    # a half group; rows of the 9-token sequence that see nothing
    ([1025, 513, 2048, 77, 6000], 24),   # several sequences, groups split across CTAs
])
def test_prefill_index_scores_match_oracle(lens, nq):
    case = synth.make_case("pf", seq_lens=lens, nq=nq, seed=nq + len(lens), spare_blocks=2)
    check_scores(case, gpu_scores(case, synth.device_case(case)))


def _fp8_scale_offset(case, slot):
    # FP8 index page: 64 tokens x 128 code bytes, then 64 fp32 scales
    return case.index_off + synth.BLOCK * synth.IDX_DIM + 4 * slot


def test_prefill_special_key_scales():
    """Negative, zero, -0 and NaN key scales on visible tokens: the scale is
    applied inside the ReLU there (max(0, c x) = c max(0, x) holds only for
    c >= 0), as the oracle defines; a NaN scale gives 0 for every head."""
    case = synth.make_case("pfx", seq_lens=[3000], nq=16, seed=11)
    pages = case.block_table[0]
    planted = {5: -1.5, 200: 0.0, 201: -0.0, 777: -0.25, 1500: float("nan"), 2990: -3.0}
    for t, v in planted.items():
        o = _fp8_scale_offset(case, t % synth.BLOCK)
        case.pool[pages[t // synth.BLOCK], o:o + 4] = np.array([v], dtype=np.float32).view(np.uint8)
    s = gpu_scores(case, synth.device_case(case))
    ref = check_scores(case, s)
    got = s.cpu().numpy()
    assert (got[:, 1500] == 0.0).all() and (ref[:, 1500] == 0.0).all()
    assert (got[:, 200] == 0.0).all()


def test_prefill_bf16_scores_match_oracle():
    case = synth.make_case("pfb", seq_lens=[2500, 600], nq=16, seed=8)
    check_scores_bf16(case, gpu_scores_bf16(case, synth.device_case(case)))


def test_prefill_decode_step_matches_oracle():
    case = synth.make_case("pfs", seq_lens=[6000, 2500], nq=16, topk=512, seed=5)
    scores, idx, o, l = _run_step(case)
    check_scores(case, scores)
    s64 = scores.cpu().numpy().astype(np.float64)
    np.testing.assert_array_equal(idx, oracle.topk(s64, case.row_lens(), case.topk))
    # k = 512: a more peaked softmax than k = 2048 gives |O| where the bf16
    # output half-ulp alone exceeds 1e-2 (the edge-case bound of the decode tests)
    check_mla(case, idx, o, l, rtol=OUT_RTOL_EDGE)


def _row_case(case, j):
    """Row j of sequence 0 of a prefill case, as a one-row decode of the
    tokens that row sees (same pool, table, queries and weights)."""
    L = int(case.seq_lens[0]) - (case.nq - 1) + j
    return dataclasses.replace(case, batch=1, nq=1, seq_lens=np.array([L], dtype=np.int32),
                               block_table=case.block_table[:1], q_index=case.q_index[j:j + 1],
                               head_w=case.head_w[j:j + 1], q_mla=case.q_mla[j:j + 1])


def test_prefill_full_size_sampled_rows():
    """The 2048-row chunk on a 153,600-token context, in one fused call;
    sampled rows checked one by one against the oracle."""
    case = synth.workload("prefill_q2048_l153600", seed=0)
    scores, idx, o, l = _run_step(case)
    for j in (0, 1, 777, 2046, 2047):
        rc = _row_case(case, j)
        check_scores(rc, scores[j:j + 1])
        s64 = scores[j:j + 1].cpu().numpy().astype(np.float64)
        np.testing.assert_array_equal(idx[j:j + 1], oracle.topk(s64, rc.row_lens(), case.topk))
        check_mla(rc, idx[j:j + 1], o[j:j + 1], l[j:j + 1])
