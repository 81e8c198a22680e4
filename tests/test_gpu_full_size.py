"""Full-size parity: the decode workloads at their full sizes, in the launch
configuration the benchmark times (one fused dsa_decode_step over the whole
batch), checked on sampled rows against the oracle one row at a time; and
the decode-context-parallel merge and LSE combine of 8 shards on the
long-context batch's own scores.  Tolerances as in the small-case tests.

Workloads (seeded as the benchmark seeds them):
  speculative decode   8 sequences x 4 causal draft rows, 32,768 tokens each
  long-context batch   32 sequences, 64K-160K tokens, heavy-tailed keys
  1M-token decode      4 sequences of 1,048,576 tokens, MXFP4 index keys (E4M3
                       query, and MXFP4 query on the native FP4 path)
  420 B/token batch    the long-context batch with NVFP4 latents and MXFP4 keys
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from dsa_sparse_attention_index_gb300 import binding, synth
from test_gpu_dcp import _gpu_dcp_mla, check_dcp_mla
from test_gpu_parity import _run_step, _status, check_mla, check_scores

pytestmark = pytest.mark.gpu

SAMPLES = {
    "specdecode_b8x4_l32768": (0, 3, 13, 30),   # first and last draft rows of several sequences
    "longctx_b32_l64k-160k": (0, 11, 31),
    "mxfp4_b4_l1m": (0, 3),
    "mxfp4n_b4_l1m": (1, 2),
    "longctx_b32_l64k-160k_nvfp4": (5, 31),
}


def _row_case(case, r):
    """Query row r as a one-row decode over the tokens it sees (same pool,
    table, queries and weights)."""
    b, j = divmod(r, case.nq)
    L = int(case.seq_lens[b]) - (case.nq - 1) + j
    if case.key_format == synth.KEY_MXFP4_NATIVE:   # codes [rows][32][64], then E8M0 [rows][32][4]
        n = case.rows * 32 * 64
        q = np.concatenate([case.q_index[:n].reshape(case.rows, -1)[r], case.q_index[n:].reshape(case.rows, -1)[r]])
    else:
        q = case.q_index[r:r + 1]
    return dataclasses.replace(case, batch=1, nq=1, seq_lens=np.array([L], dtype=np.int32),
                               block_table=case.block_table[b:b + 1], q_index=q,
                               head_w=case.head_w[r:r + 1], q_mla=case.q_mla[r:r + 1])


@pytest.fixture(scope="module")
def longctx():
    case = synth.workload("longctx_b32_l64k-160k", seed=0)
    return case, _run_step(case)


def _check_rows(case, res, rows):
    scores, idx, o, l = res
    for r in rows:
        rc = _row_case(case, r)
        check_scores(rc, scores[r:r + 1])
        s64 = scores[r:r + 1].cpu().numpy().astype(np.float64)
        np.testing.assert_array_equal(idx[r:r + 1], oracle.topk(s64, rc.row_lens(), case.topk))
        check_mla(rc, idx[r:r + 1], o[r:r + 1], l[r:r + 1])


@pytest.mark.parametrize("name", ["specdecode_b8x4_l32768", "mxfp4_b4_l1m", "mxfp4n_b4_l1m",
                                  "longctx_b32_l64k-160k_nvfp4"])
def test_full_size_decode_step_sampled_rows(name):
    case = synth.workload(name, seed=0)
    _check_rows(case, _run_step(case), SAMPLES[name])


def test_full_size_long_context_sampled_rows(longctx):
    case, res = longctx
    _check_rows(case, res, SAMPLES["longctx_b32_l64k-160k"])


def test_full_size_dcp_merge_and_combine(longctx):
    """8 shards over the step's scores of the 32-row long-context batch (up to
    162K tokens a row, so up to 20K a shard): the merged top-k of every row
    bit-exact against the oracle's merge, and the partial attention plus LSE
    combine of sampled rows against the oracle's."""
    case, (scores, _, _, _) = longctx
    rows, k, shards = case.rows, case.topk, 8
    dc = synth.device_case(case)
    idx = torch.empty((rows, k), dtype=torch.int32, device="cuda")
    stats = torch.empty((rows, 3), dtype=torch.int32, device="cuda")
    ws = binding.workspace(binding.dcp_topk_workspace_size(rows, k, shards))
    st = _status()
    binding.dcp_topk(scores, dc.row_lens, case.max_len, k, shards, idx, ws, st, stats_out=stats)
    torch.cuda.synchronize()
    assert st.item() == 0, binding.status_string(st.item())
    idx = idx.cpu().numpy()
    ref, ref_stats = oracle.dcp_topk(scores.cpu().numpy(), case.row_lens(), k, shards)
    np.testing.assert_array_equal(idx, ref)
    np.testing.assert_array_equal(stats.cpu().numpy(), ref_stats.astype(np.int32))
    o, l, po, pl = _gpu_dcp_mla(case, dc, idx, shards)
    for r in SAMPLES["longctx_b32_l64k-160k"]:
        check_dcp_mla(_row_case(case, r), idx[r:r + 1], shards, o[r:r + 1], l[r:r + 1], po[:, r:r + 1],
                      pl[:, r:r + 1])
