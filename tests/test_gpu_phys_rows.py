"""GPU parity of the physical KV rows the top-k outputs beside its token
indices (Day-0 post, fused-decode section: the fused indexer outputs the
physical KV rows that attention reads): dsa_topk_paged and the fused step's
phys_out, bit for bit against the oracle's translation through the block
table, on every top-k path; and the step's attention, which reads those rows
instead of translating the indices again, bit for bit the same as the
attention on the indices alone."""
import numpy as np
import pytest
import torch

import oracle
from dsa_sparse_attention_index_gb300 import binding, synth
from test_gpu_parity import _gpu_mla, _status, gpu_scores

pytestmark = pytest.mark.gpu


def _topk_paged(case, dc, scores, k=2048, with_phys=True):
    rows = case.rows
    idx = torch.empty((rows, k), dtype=torch.int32, device="cuda")
    phys = torch.full((rows, k), -7, dtype=torch.int32, device="cuda") if with_phys else None
    ws = binding.workspace(binding.topk_workspace_size(rows, case.max_len, k))
    st = _status()
    binding.topk_paged(dc.cache, dc.batch, scores, k, idx, ws, st, phys_out=phys)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), (phys.cpu().numpy() if with_phys else None), st.item()


@pytest.mark.parametrize("lens,nq,multipass", [
    ([6000, 2500, 900, 40], 1, False),        # cluster top-k; a row shorter than k
    ([9000, 3000], 4, False),                 # draft rows share their sequence's table row
    ([260_000, 3000], 1, False),              # the two-level cluster form
    ([200_000, 340_000], 2, False),           # two levels with draft rows (2 segments and 3)
    ([260_000, 3000], 1, True),               # the four-kernel path
    ([50_000, 30_000], 160, False),           # many rows: one CTA per row
])
def test_topk_paged_rows_match_the_oracle(lens, nq, multipass):
    case = synth.make_case("ph", seq_lens=lens, nq=nq, seed=len(lens) + nq)
    dc = synth.device_case(case)
    scores = gpu_scores(case, dc)
    prev = binding.topk_force_multipass(multipass)
    try:
        idx, phys, st = _topk_paged(case, dc, scores)
    finally:
        binding.topk_force_multipass(prev)
    assert st == 0, binding.status_string(st)
    s64 = scores.cpu().numpy().astype(np.float64)
    np.testing.assert_array_equal(idx, oracle.topk(s64, case.row_lens(), 2048))
    np.testing.assert_array_equal(phys, oracle.phys_rows(case, idx))


def test_topk_paged_reports_a_bad_block_entry():
    case = synth.make_case("phb", seq_lens=[5000], seed=3)
    dc = synth.device_case(case)
    scores = gpu_scores(case, dc)
    idx, _, st = _topk_paged(case, dc, scores, with_phys=False)
    assert st == 0
    # an entry the selection uses, set outside the pool on the device only
    blk = int(idx[0, 0]) // 64
    dc.batch.block_table[0, blk] = case.num_blocks + 1
    idx2, phys, st = _topk_paged(case, dc, scores)
    assert st == binding.ERR_BOUNDS
    np.testing.assert_array_equal(idx2, idx)
    assert (phys[0][idx[0] // 64 == blk] == -1).all()


@pytest.mark.parametrize("fmt", [synth.KEY_FP8, synth.KEY_MXFP4])
def test_decode_step_phys_out_and_attention_on_rows(fmt):
    """The step's phys_out equals the oracle's translation of its idx_out, and
    its attention (reading the rows) equals sparse_mla_decode on the indices
    (translating them) bit for bit."""
    case = synth.make_case("phs", seq_lens=[7000, 3300, 2049], nq=1, key_format=fmt, seed=12)
    dc = synth.device_case(case)
    k, rows = case.topk, case.rows
    out = torch.empty((rows, 96, 512), dtype=torch.int16, device="cuda")
    lse = torch.empty((rows, 96), dtype=torch.float32, device="cuda")
    idx = torch.empty((rows, k), dtype=torch.int32, device="cuda")
    phys = torch.empty((rows, k), dtype=torch.int32, device="cuda")
    ws = binding.workspace(binding.workspace_size(dc.batch, k))
    st = _status()
    binding.decode_step(dc.cache, dc.batch, dc.q_index, dc.head_w, dc.q_mla, k, case.sm_scale, out, lse, ws, st,
                        idx_out=idx, phys_out=phys)
    torch.cuda.synchronize()
    assert st.item() == 0, binding.status_string(st.item())
    idx_np = idx.cpu().numpy()
    np.testing.assert_array_equal(phys.cpu().numpy(), oracle.phys_rows(case, idx_np))
    o2, l2 = _gpu_mla(case, dc, idx_np)
    np.testing.assert_array_equal(out.view(torch.bfloat16).float().cpu().numpy(), o2)
    np.testing.assert_array_equal(lse.cpu().numpy(), l2)
