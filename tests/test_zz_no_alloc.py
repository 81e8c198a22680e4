"""The top-k entry point that allocates nothing (dsa_topk_noalloc).

Some callers cannot call cudaMalloc (a framework that owns the device memory
pool, or a loop where allocation could block or synchronise the device); this
variant keeps its scratch in a device array built into the library.  The test
calls it through the C ABI twice in a row, on different inputs, and checks
each result against the workspace-taking dsa_topk (top-k is bit-exact), so a
second call that saw stale scratch from the first would fail.  This file is
collected last on purpose.
"""
import numpy as np
import pytest
import torch

from dsa_sparse_attention_index_gb300 import binding

pytestmark = pytest.mark.gpu


def _inputs(seed, rows, L):
    rng = np.random.default_rng(seed)
    m = rng.standard_normal((rows, L)).astype(np.float32)
    m[1, ::5] = 0.25                      # heavy ties in one row
    m[2] = 3.0                            # all equal (candidate overflow path)
    lens = rng.integers(1, L + 1, rows).astype(np.int32)
    lens[0], lens[3] = L, 100             # a full row and a row shorter than k
    return torch.from_numpy(m).cuda(), torch.from_numpy(lens).cuda()


def _with_workspace(scores, lens, L, k):
    rows = scores.shape[0]
    ws = binding.workspace(binding.topk_workspace_size(rows, L, k))
    out = torch.empty((rows, k), dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.topk(scores, lens, L, k, out, ws, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    return out


def test_topk_noalloc_matches_workspace_entry_point_on_two_calls():
    rows, L, k = 48, 20000, 2048
    for call, seed in enumerate((5, 6)):
        scores, lens = _inputs(seed, rows, L)
        want = _with_workspace(scores, lens, L, k)
        got = torch.full((rows, k), -7, dtype=torch.int32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        binding.topk_noalloc(scores, lens, L, k, got, st)
        torch.cuda.synchronize()
        assert st.item() == 0, f"call {call}: {binding.status_string(st.item())}"
        assert torch.equal(got, want), f"call {call}: differs from dsa_topk"


def test_topk_noalloc_rejects_more_rows_than_its_scratch_holds():
    scores = torch.zeros((65, 4096), dtype=torch.float32, device="cuda")
    lens = torch.full((65,), 4096, dtype=torch.int32, device="cuda")
    out = torch.empty((65, 2048), dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(binding.DsaError) as e:
        binding.topk_noalloc(scores, lens, 4096, 2048, out, st)
    assert e.value.code == binding.ERR_UNSUPPORTED
