"""Batch invariance (Day-0 post, section "day 0 的零失配 RL", zero-mismatch
RL: a token's log-prob must not depend on the batch it is computed in).
With the batch-invariant mode on, every row of a batch gets bitwise the same
scores, indices, output and LSE as when it is decoded alone; with it off, the
sparse MLA's split into chunks follows the number of rows and the outputs
differ in the last bits.
"""
import dataclasses

import numpy as np
import pytest

from dsa_sparse_attention_index_gb300 import binding, synth
from test_gpu_parity import _run_step

pytestmark = pytest.mark.gpu


def _seq_case(case, b):
    """Sequence b of a case alone (all of its query rows)."""
    r0, r1 = b * case.nq, (b + 1) * case.nq
    return dataclasses.replace(case, batch=1, seq_lens=case.seq_lens[b:b + 1].copy(),
                               block_table=case.block_table[b:b + 1], q_index=case.q_index[r0:r1],
                               head_w=case.head_w[r0:r1], q_mla=case.q_mla[r0:r1])


def _differences(case, seqs):
    """Element counts where the batched and the alone results differ:
    (scores, indices, outputs, LSE) summed over the sequences `seqs`."""
    s, idx, o, l = _run_step(case)
    s = s.cpu().numpy()
    lens = case.row_lens()
    d = np.zeros(4, dtype=np.int64)
    for b in seqs:
        s1, i1, o1, l1 = _run_step(_seq_case(case, b))
        s1 = s1.cpu().numpy()
        for j in range(case.nq):
            r, vis = b * case.nq + j, lens[b * case.nq + j]
            d[0] += np.count_nonzero(s[r, :vis].view(np.int32) != s1[j, :vis].view(np.int32))
            d[1] += np.count_nonzero(idx[r] != i1[j])
            d[2] += np.count_nonzero(o[r].view(np.int32) != o1[j].view(np.int32))
            d[3] += np.count_nonzero(l[r].view(np.int32) != l1[j].view(np.int32))
    return d


@pytest.mark.parametrize("nq,nseq", [(1, 40), (4, 10)])
def test_rows_decode_alike_alone_and_in_a_batch(nq, nseq):
    """40 query rows (one wave of chunks per row at most 3 wide) against the
    same sequences alone (up to 16 chunks): identical bits in the
    batch-invariant mode; without it only the attention output and LSE may
    move, and they do."""
    rng = np.random.default_rng(nq)
    lens = rng.integers(2500, 24000, nseq)
    case = synth.make_case("binv", seq_lens=lens, nq=nq, seed=90 + nq)
    seqs = (0, 3, nseq - 1)
    prev = binding.batch_invariant(True)
    try:
        assert np.all(_differences(case, seqs) == 0)
    finally:
        binding.batch_invariant(prev)
    binding.batch_invariant(False)
    try:
        d = _differences(case, seqs)
    finally:
        binding.batch_invariant(prev)
    assert d[0] == 0 and d[1] == 0          # the indexer and the top-k never depended on the batch
    assert d[2] > 0                         # the chunk split did
