"""The top-k entry point that allocates nothing (dsa_topk_noalloc).

Some callers cannot call cudaMalloc: a host framework that owns the whole
device memory pool, or a serving loop where an allocation could block or
synchronise the device.  This variant keeps its scratch in a device array
built into the library, so it takes no workspace argument.

The scratch is only touched by the four-kernel top-k (histograms, counters,
selected and candidate lists), which runs for rows too long to hold on chip
when the streaming cluster is not used.  The tests therefore force that path
with dsa_topk_force_multipass and use rows longer than 245,760 tokens, and
call the entry point twice in a row on different inputs: the first call
leaves its histograms, counters and candidates behind, so a second call that
read stale scratch (a missed clear, a wrong offset) would select differently.
Each call is checked bit for bit against the oracle and against dsa_topk with
a caller-owned workspace.  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import oracle
from dsa_sparse_attention_index_gb300 import binding

pytestmark = pytest.mark.gpu

K = 2048


def _long_rows(seed, rows=6, n=300_000):
    """Rows past the on-chip limit: ties on the k-th key, an all-equal row
    (its candidates overflow the candidate list), a row shorter than k, and
    rows of mixed lengths."""
    rng = np.random.default_rng(seed)
    m = rng.standard_normal((rows, n)).astype(np.float32)
    m[0] = rng.integers(0, 40, n)                  # ties on the k-th key
    m[1] = 3.0 + seed                              # all equal: the lowest k indices
    m[2, ::5] = 0.25                               # a tied run inside a normal row
    lens = np.array([n, n, n - 7, 100, 260_001, n - 2], dtype=np.int32)[:rows]
    return m, lens


def _workspace_topk(scores, lens, max_len):
    rows = scores.shape[0]
    ws = binding.workspace(binding.topk_workspace_size(rows, max_len, K))
    out = torch.empty((rows, K), dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.topk(scores, lens, max_len, K, out, ws, st)
    torch.cuda.synchronize()
    assert st.item() == 0, binding.status_string(st.item())
    return out.cpu().numpy()


def _noalloc_topk(scores, lens, max_len):
    rows = scores.shape[0]
    out = torch.full((rows, K), -7, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.topk_noalloc(scores, lens, max_len, K, out, st)
    torch.cuda.synchronize()
    assert st.item() == 0, binding.status_string(st.item())
    return out.cpu().numpy()


def test_topk_noalloc_uses_its_scratch_correctly_on_two_calls():
    prev = binding.topk_force_multipass(True)
    try:
        for call, seed in enumerate((5, 6)):
            m, lens = _long_rows(seed)
            scores, d_lens = torch.from_numpy(m).cuda(), torch.from_numpy(lens).cuda()
            n0 = binding.kernel_launches()
            got = _noalloc_topk(scores, d_lens, m.shape[1])
            assert binding.kernel_launches() - n0 == 4, "the four-kernel path (the one with scratch) must run"
            want = oracle.topk(m.astype(np.float64), lens, K)
            np.testing.assert_array_equal(got, want, err_msg=f"call {call}: differs from the oracle")
            np.testing.assert_array_equal(got, _workspace_topk(scores, d_lens, m.shape[1]),
                                          err_msg=f"call {call}: differs from dsa_topk")
    finally:
        binding.topk_force_multipass(prev)


def test_topk_noalloc_rows_no_longer_than_k():
    """Every row fits in k: the entry point still goes through its scratch
    set-up, and the final kernel writes 0..len-1 with -1 padding."""
    rng = np.random.default_rng(3)
    m = rng.standard_normal((5, K)).astype(np.float32)
    lens = np.array([K, 1, 0, 777, K - 1], dtype=np.int32)
    got = _noalloc_topk(torch.from_numpy(m).cuda(), torch.from_numpy(lens).cuda(), K)
    np.testing.assert_array_equal(got, oracle.topk(m.astype(np.float64), lens, K))


def test_topk_noalloc_rejects_more_rows_than_its_scratch_holds():
    scores = torch.zeros((65, 4096), dtype=torch.float32, device="cuda")
    lens = torch.full((65,), 4096, dtype=torch.int32, device="cuda")
    out = torch.empty((65, K), dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(binding.DsaError) as e:
        binding.topk_noalloc(scores, lens, 4096, K, out, st)
    assert e.value.code == binding.ERR_UNSUPPORTED
