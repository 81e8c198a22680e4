"""GPU parity of the prefill rows: a chunk of causal query rows per sequence
(row j of a sequence with context L and nq rows sees L - (nq - 1) + j tokens),
through the indexer (rows in groups of four), the top-k and the sparse MLA,
against the fp64 oracle on the same seeded inputs.  Tolerances as for decode.
"""
import dataclasses

import numpy as np
import pytest

import oracle
from dsa_sparse_attention_index_gb300 import synth
from test_gpu_parity import OUT_RTOL_EDGE, _run_step, check_mla, check_scores, gpu_scores

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("lens,nq", [([5000], 64), ([3000, 700], 8), ([300, 4100, 9], 12)])
def test_prefill_index_scores_match_oracle(lens, nq):
    case = synth.make_case("pf", seq_lens=lens, nq=nq, seed=nq + len(lens), spare_blocks=2)
    check_scores(case, gpu_scores(case, synth.device_case(case)))


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
