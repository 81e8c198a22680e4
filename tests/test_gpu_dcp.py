"""GPU parity of the decode-context-parallel top-k merge (Day-0 post,
decode-context-parallelism section), emulated on one GPU: indices and the
words-sent statistics bit-exact against the oracle's shard-by-shard merge,
and equal to the plain top-k of the bf16-rounded scores.
"""
import numpy as np
import pytest
import torch

import oracle
from dsa_sparse_attention_index_gb300 import binding, synth
from test_gpu_parity import _status, gpu_scores

pytestmark = pytest.mark.gpu


def _gpu_dcp(m, lens, k, shards, max_row_len=None):
    rows = m.shape[0]
    max_row_len = int(max_row_len if max_row_len is not None else m.shape[1])
    scores = torch.from_numpy(np.ascontiguousarray(m, dtype=np.float32)).cuda()
    row_lens = torch.from_numpy(np.ascontiguousarray(lens, dtype=np.int32)).cuda()
    idx = torch.full((rows, k), -7, dtype=torch.int32, device="cuda")
    stats = torch.full((rows, 3), -7, dtype=torch.int32, device="cuda")
    ws = binding.workspace(binding.dcp_topk_workspace_size(rows, k, shards))
    st = _status()
    binding.dcp_topk(scores, row_lens, max_row_len, k, shards, idx, ws, st, stats_out=stats)
    torch.cuda.synchronize()
    assert st.item() == 0, binding.status_string(st.item())
    return idx.cpu().numpy(), stats.cpu().numpy()


def _check(m, lens, k, shards):
    got, stats = _gpu_dcp(m, lens, k, shards)
    ref, ref_stats = oracle.dcp_topk(m, lens, k, shards)
    np.testing.assert_array_equal(got, ref)
    np.testing.assert_array_equal(stats, ref_stats.astype(np.int32))
    return stats


@pytest.mark.parametrize("shards", [1, 2, 3, 5, 8])
def test_dcp_topk_matches_oracle(shards):
    rng = np.random.default_rng(40 + shards)
    n = 20_000
    m = np.zeros((7, n), dtype=np.float32)
    m[0] = rng.standard_normal(n)
    m[1] = rng.integers(0, 30, n)                        # heavy ties on the k-th key
    m[2] = rng.standard_normal(n) * 1e-3 + 1.0            # ties only after bf16 rounding
    m[3] = rng.standard_normal(n)
    m[3, [3, 500, 9000]] = [np.nan, -0.0, np.inf]
    m[3, 100:140] = 0.0
    m[4] = -rng.exponential(1.0, n)
    m[5] = 7.0                                            # all equal
    m[6] = rng.standard_normal(n)
    lens = np.array([n, n - 3, n - 1, 2048, 2049, n, 700], dtype=np.int32)
    _check(m, lens, 2048, shards)


@pytest.mark.parametrize("shards", [2, 4, 8])
def test_dcp_topk_resend(shards):
    """Every token of one shard outscores the rest: that shard's words are all
    taken and it resends its full local top-k; another row concentrates the
    top in two shards."""
    rng = np.random.default_rng(50 + shards)
    n = 60_000
    m = rng.standard_normal((3, n)).astype(np.float32)
    m[0, 1::shards] += 100.0
    m[1, 0::shards] += 50.0
    m[1, (shards - 1)::shards] += 50.0
    lens = np.array([n, n, n - 11], dtype=np.int32)
    stats = _check(m, lens, 2048, shards)
    assert stats[0, 1] >= 1 and stats[2, 1] == 0


@pytest.mark.parametrize("k", [64, 1])
def test_dcp_topk_small_k(k):
    rng = np.random.default_rng(k)
    m = rng.integers(0, 5, (3, 5000)).astype(np.float32)
    lens = np.array([5000, 10, 0], dtype=np.int32)
    _check(m, lens, k, 8)


def test_dcp_topk_on_indexer_scores():
    """8 shards over the indexer's own scores of a long-context batch, where
    the rows are up to 8 x 65,536 tokens."""
    case = synth.make_case("dcp", seq_lens=[150_000, 70_001, 4096, 300_000], nq=1, seed=6, heavy_tail=0.1)
    s = gpu_scores(case, synth.device_case(case), extra=0)
    m = s.cpu().numpy()
    _check(m, case.row_lens(), 2048, 8)
