"""GPU parity of decode context parallelism (Day-0 post,
decode-context-parallelism section), emulated on one GPU:

* the top-k merge: indices and the words-sent statistics bit-exact against
  the oracle's shard-by-shard merge, and equal to the plain top-k of the
  bf16-rounded scores;
* the LSE combine: per-shard partial attention (bf16 outputs, fp32 LSEs)
  and their log-sum-exp merge against the oracle's, and against the
  unsharded attention.
"""
import numpy as np
import pytest
import torch

import oracle
from dsa_sparse_attention_index_gb300 import binding, synth
from test_gpu_parity import LSE_ATOL, OUT_ATOL, _gpu_mla, _status, gpu_scores

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
    return got, stats


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
    _, stats = _check(m, lens, 2048, shards)
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


# ---------------------------------------------------------------- LSE combine
def _gpu_dcp_mla(case, dc, idx_np, shards):
    rows, k = idx_np.shape
    idx = torch.from_numpy(np.ascontiguousarray(idx_np, dtype=np.int32)).cuda()
    out = torch.empty((rows, 96, 512), dtype=torch.int16, device="cuda")
    lse = torch.empty((rows, 96), dtype=torch.float32, device="cuda")
    part_out = torch.empty((shards, rows, 96, 512), dtype=torch.int16, device="cuda")
    part_lse = torch.empty((shards, rows, 96), dtype=torch.float32, device="cuda")
    ws = binding.workspace(binding.dcp_sparse_mla_workspace_size(rows, k, shards))
    st = _status()
    n0 = binding.kernel_launches()
    binding.dcp_sparse_mla(dc.cache, dc.batch, dc.q_mla, idx, shards, case.sm_scale, out, lse, ws, st,
                           part_out=part_out, part_lse=part_lse)
    torch.cuda.synchronize()
    assert st.item() == 0, binding.status_string(st.item())
    assert binding.kernel_launches() - n0 == 3
    f = lambda t: t.view(torch.bfloat16).float().cpu().numpy()
    return f(out), lse.cpu().numpy(), f(part_out), part_lse.cpu().numpy()


def _check_lse(got, ref):
    fin = np.isfinite(ref)
    assert np.array_equal(fin, np.isfinite(got)) and np.all(np.isneginf(got[~fin]))
    if fin.any():
        assert np.abs(got[fin] - ref[fin]).max() <= LSE_ATOL


def check_dcp_mla(case, idx, shards, o, l, po, pl):
    """Tolerances: each shard's output is the sparse MLA over its tokens, so
    within the MLA bound (1e-2) of the oracle's before both sides round it to
    bf16; rounding two nearby values can land one bf16 step (2^-7 |O_w|)
    apart, so the partials and the merged output are held to
    1e-2 + 2^-7 max_w |O_w|.  The merged output is also held to that bound
    against the unsharded fp64 attention (the invariant of the scheme)."""
    ro, rl, rpo, rpl = oracle.dcp_sparse_mla(case, idx, shards)
    step = 2.0 ** -7 * np.abs(rpo).max(axis=0)
    for w in range(shards):
        excess = np.abs(po[w] - rpo[w]) - (OUT_ATOL + 2.0 ** -7 * np.abs(rpo[w]))
        assert excess.max() <= 0, f"shard {w}: max |O_w - ref| = {np.abs(po[w] - rpo[w]).max()}"
        _check_lse(pl[w], rpl[w])
        assert np.all(po[w][~np.isfinite(rpl[w])] == 0)
    excess = np.abs(o - ro) - (OUT_ATOL + step)
    assert excess.max() <= 0, f"max |out - ref| = {np.abs(o - ro).max()}"
    _check_lse(l, rl)
    plain, plain_lse = oracle.sparse_mla(case, idx)
    assert (np.abs(o - plain) - (OUT_ATOL + step)).max() <= 0
    _check_lse(l, plain_lse)


@pytest.mark.parametrize("shards", [1, 2, 3, 8])
def test_dcp_sparse_mla_matches_oracle(shards):
    """k = 2048 over rows of 6,000, 2,500 and 900 tokens (the last padded
    with -1): two pieces per shard, ragged tiles, a partly masked row."""
    case = synth.make_case("dcpm", seq_lens=[6000, 2500, 900], nq=1, seed=60 + shards)
    dc = synth.device_case(case)
    rng = np.random.default_rng(shards)
    k = 2048
    idx = np.full((3, k), -1, dtype=np.int32)
    for r, L in enumerate(case.row_lens()):
        n = min(k, int(L))
        idx[r, :n] = np.sort(rng.choice(int(L), n, replace=False))
    idx[0, 300:420] = -1
    o, l, po, pl = _gpu_dcp_mla(case, dc, idx, shards)
    check_dcp_mla(case, idx, shards, o, l, po, pl)
    # the invariant on the GPU too: the sharded and the unsharded kernels agree
    o1, l1 = _gpu_mla(case, dc, idx)
    assert np.abs(o - o1).max() <= 2 * OUT_ATOL + 2.0 ** -7 * np.abs(o1).max()
    assert np.abs(l - l1)[np.isfinite(l1)].max() <= 2 * LSE_ATOL


def test_dcp_sparse_mla_one_shard_holds_every_token():
    """All 2,048 selected tokens in shard 0 of 4: its group fills both of its
    pieces (1,024 tokens each), the other shards send LSE = -inf and
    nothing of theirs reaches the output."""
    case = synth.make_case("dcp1", seq_lens=[9000, 8300], nq=1, seed=70)
    dc = synth.device_case(case)
    rng = np.random.default_rng(70)
    idx = np.stack([np.sort(rng.choice(np.arange(0, L, 4), 2048, replace=False)) for L in (9000, 8300)])
    idx = idx.astype(np.int32)
    o, l, po, pl = _gpu_dcp_mla(case, dc, idx, 4)
    check_dcp_mla(case, idx, 4, o, l, po, pl)
    assert np.all(np.isneginf(pl[1:])) and np.all(po[1:] == 0)
    assert np.array_equal(o, po[0]) and np.array_equal(l, pl[0])   # weight exactly 1


@pytest.mark.parametrize("k", [100, 1])
def test_dcp_sparse_mla_small_k_and_empty_rows(k):
    """One piece per shard; a fully masked row (out 0, LSE -inf), a row with
    a single token, and five shards (some empty)."""
    case = synth.make_case("dcps", seq_lens=[700, 300, 50], nq=1, seed=80 + k)
    dc = synth.device_case(case)
    rng = np.random.default_rng(k)
    idx = np.full((3, k), -1, dtype=np.int32)
    idx[0] = np.sort(rng.choice(700, k, replace=False))
    idx[2, 0] = 33
    o, l, po, pl = _gpu_dcp_mla(case, dc, idx, 5)
    check_dcp_mla(case, idx, 5, o, l, po, pl)
    assert np.all(o[1] == 0) and np.all(np.isneginf(l[1]))


def test_dcp_merge_then_combine_on_speculative_rows():
    """Draft rows (4 per sequence, each seeing one more token): the merged
    top-k of 3 shards from the indexer's scores, then the shards' partial
    attention and LSE combine, each against the oracle."""
    case = synth.make_case("dcpspec", seq_lens=[9000, 4100], nq=4, seed=77)
    dc = synth.device_case(case)
    s = gpu_scores(case, dc, extra=0)
    m = s.cpu().numpy()
    idx, _ = _check(m, case.row_lens(), 2048, 3)
    o, l, po, pl = _gpu_dcp_mla(case, dc, idx, 3)
    check_dcp_mla(case, idx, 3, o, l, po, pl)
