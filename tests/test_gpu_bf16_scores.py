"""BF16 scores between the indexer and the top-k (Day-0 post,
decode-context-parallelism section: candidates picked straight from BF16
scores).  The indexer's bf16 scores are its fp32 scores rounded to nearest
even; the top-k over bf16 scores is bit-exact against the oracle's top-k of
the same values; the fused step with bf16 scores against the oracle; and
the documented consequence: the bf16 selection differs from the fp32 one only
among tokens whose bf16 score equals the k-th bf16 score.
"""
import numpy as np
import pytest
import torch

import oracle
from dsa_sparse_attention_index_gb300 import binding, synth
from test_gpu_parity import SCORE_RTOL, _status, check_mla, gpu_scores

pytestmark = pytest.mark.gpu

SENTINEL16 = 0x7FDE  # a NaN pattern marking never-written bf16 entries


def _ld8(n):
    return (max(n, 1) + 7) // 8 * 8


def gpu_scores_bf16(case, dc, extra=8):
    ld = _ld8(case.max_len) + extra
    s = torch.full((case.rows, ld), SENTINEL16, dtype=torch.int16, device="cuda")
    st = _status()
    binding.index_scores_bf16(dc.cache, dc.batch, dc.q_index, dc.head_w, s, st)
    torch.cuda.synchronize()
    assert st.item() == 0, binding.status_string(st.item())
    return s


def _values(bits):
    """bf16 bits (torch int16, any device) -> fp64 numpy, exactly."""
    return bits.view(torch.bfloat16).to(torch.float64).cpu().numpy()


def check_scores_bf16(case, bits):
    """Within the fp32 score tolerance plus one bf16 rounding (2^-9 |s|,
    taken as 2^-8 |ref|) of the fp64 oracle; never written past the visible
    length."""
    ld = bits.shape[1]
    ref = oracle.index_scores(case, ld)
    ref16 = oracle.index_scores_bf16(case, ld)
    bound = oracle.index_score_bounds(case, ld)
    got = _values(bits)
    raw = bits.cpu().numpy()
    for r, vis in enumerate(case.row_lens()):
        a, g, b16 = ref[r, :vis], got[r, :vis], ref16[r, :vis]
        slack = SCORE_RTOL * np.fmax(np.abs(a), bound[r, :vis])
        bad = np.nonzero(~(np.abs(g - a) <= slack + 2.0 ** -8 * np.abs(a)))[0]
        assert bad.size == 0, f"row {r}: {bad.size} bf16 scores out of tolerance, first t={bad[:5]}"
        # against the oracle's own rounding: equal unless the fp32 error crossed
        # a rounding boundary, then one bf16 step apart
        step = np.ldexp(1.0, np.frexp(np.fmax(np.abs(a), np.abs(g)))[1] - 8)
        bad = np.nonzero(~((g == b16) | (np.abs(g - b16) <= step + slack)))[0]
        assert bad.size == 0, f"row {r}: {bad.size} bf16 scores off the rounded oracle, first t={bad[:5]}"
        assert np.all(raw[r, vis:] == SENTINEL16), f"row {r}: wrote past its visible length"


@pytest.mark.parametrize("lens,nq,fmt", [
    ([4096], 1, synth.KEY_FP8),
    ([1, 63, 64, 65, 127, 128, 129, 200, 1000, 0], 1, synth.KEY_FP8),
    ([300, 1031], 2, synth.KEY_FP8),
    ([5000, 700], 8, synth.KEY_FP8),
    ([3000, 130], 1, synth.KEY_MXFP4),
])
def test_index_scores_bf16(lens, nq, fmt):
    case = synth.make_case("ib", seq_lens=lens, nq=nq, key_format=fmt, seed=len(lens) + nq, spare_blocks=2)
    dc = synth.device_case(case)
    bits = gpu_scores_bf16(case, dc)
    check_scores_bf16(case, bits)
    # the same fp32 values as dsa_index_scores, rounded to nearest even
    f32 = gpu_scores(case, dc, extra=0)
    want = f32.to(torch.bfloat16).view(torch.int16).cpu().numpy()
    got = bits.cpu().numpy()
    for r, vis in enumerate(case.row_lens()):
        np.testing.assert_array_equal(got[r, :vis], want[r, :vis])


def _gpu_topk_bf16(bits_np, lens, k, max_row_len=None):
    rows, n = bits_np.shape
    ld = _ld8(n)
    buf = np.zeros((rows, ld), dtype=np.int16)
    buf[:, :n] = bits_np
    s = torch.from_numpy(buf).cuda()
    row_lens = torch.from_numpy(np.ascontiguousarray(lens, dtype=np.int32)).cuda()
    idx = torch.full((rows, k), -7, dtype=torch.int32, device="cuda")
    st = _status()
    binding.topk_bf16(s, row_lens, int(max_row_len if max_row_len is not None else n), k, idx, st)
    torch.cuda.synchronize()
    assert st.item() == 0, binding.status_string(st.item())
    return idx.cpu().numpy()


def _bf16_bits(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy()


def _ref_topk(bits_np, lens, k):
    vals = torch.from_numpy(bits_np).view(torch.bfloat16).to(torch.float64).numpy()
    return oracle.topk(vals, lens, k)


@pytest.mark.parametrize("n", [2048, 2049, 30_000, 70_001, 245_760, 245_761, 400_000])
def test_topk_bf16_matches_oracle(n):
    """Row lengths across the paths (no selection, resident clusters of 1-8
    CTAs, the streaming clusters past 245,760), with rows of heavy ties,
    ties that exist only in bf16, and special values."""
    rng = np.random.default_rng(n)
    m = np.zeros((4, n), dtype=np.float32)
    m[0] = rng.standard_normal(n)
    m[1] = rng.integers(0, 50, n)
    m[2] = 1.0 + rng.standard_normal(n) * 1e-3
    m[3] = rng.standard_normal(n)
    m[3, [0, 7, n // 2, n - 1]] = [np.nan, -0.0, np.inf, -np.inf]
    m[3, 10:40] = 0.0
    bits = _bf16_bits(m)
    lens = np.array([n, n - 1, max(0, n - 5), n], dtype=np.int32)
    for k in (2048, 100):
        np.testing.assert_array_equal(_gpu_topk_bf16(bits, lens, k), _ref_topk(bits, lens, k))


def test_topk_bf16_short_rows_and_k():
    rng = np.random.default_rng(3)
    m = rng.standard_normal((4, 600)).astype(np.float32)
    bits = _bf16_bits(m)
    lens = np.array([600, 10, 0, 599], dtype=np.int32)
    for k in (1, 64, 600, 2048):
        np.testing.assert_array_equal(_gpu_topk_bf16(bits, lens, k), _ref_topk(bits, lens, k))


def _run_step_bf16(case):
    dc = synth.device_case(case)
    k, rows = case.topk, case.rows
    ld = _ld8(case.max_len)
    scores = torch.full((rows, ld), SENTINEL16, dtype=torch.int16, device="cuda")
    idx = torch.empty((rows, k), dtype=torch.int32, device="cuda")
    out = torch.empty((rows, 96, 512), dtype=torch.int16, device="cuda")
    lse = torch.empty((rows, 96), dtype=torch.float32, device="cuda")
    ws = binding.workspace(binding.workspace_size(dc.batch, k))
    st = _status()
    binding.decode_step_bf16(dc.cache, dc.batch, dc.q_index, dc.head_w, dc.q_mla, k, case.sm_scale, out, lse, ws,
                             st, scores_out=scores, idx_out=idx)
    torch.cuda.synchronize()
    assert st.item() == 0, binding.status_string(st.item())
    return dc, scores, idx.cpu().numpy(), out.view(torch.bfloat16).float().cpu().numpy(), lse.cpu().numpy()


@pytest.mark.parametrize("name,kw", [
    ("decode_b1_l4096", dict(seq_lens=[4096], permute_blocks=False)),
    ("spec_b2x4", dict(seq_lens=[5000, 2100], nq=4)),
    ("ragged_b3", dict(seq_lens=[70001, 1500, 2047])),
    ("long_b2", dict(seq_lens=[300_000, 9000], heavy_tail=0.1)),
])
def test_decode_step_bf16_matches_oracle(name, kw):
    case = synth.make_case(name, seed=27, **kw)
    dc, scores, idx, o, l = _run_step_bf16(case)
    check_scores_bf16(case, scores)
    vals = _values(scores)
    np.testing.assert_array_equal(idx, oracle.topk(vals, case.row_lens(), case.topk))
    check_mla(case, idx, o, l)
    # the tie consequence: against the fp32 selection of the same indexer, the
    # sets differ only among tokens whose bf16 score equals the k-th bf16 score
    f32 = gpu_scores(case, dc, extra=0)
    idx32 = oracle.topk(f32.cpu().numpy().astype(np.float64), case.row_lens(), case.topk)
    for r, vis in enumerate(case.row_lens()):
        if vis <= case.topk:
            assert np.array_equal(idx[r], idx32[r])
            continue
        kth = np.sort(vals[r, :vis])[::-1][case.topk - 1]
        diff = set(idx[r][idx[r] >= 0]) ^ set(idx32[r][idx32[r] >= 0])
        assert all(vals[r, t] == kth for t in diff), r


def test_decode_step_bf16_in_the_420_byte_configuration():
    """BF16 scores with MXFP4 keys and NVFP4 latents."""
    case = synth.make_case("b16nv", seq_lens=[20000, 3000], seed=29, key_format=synth.KEY_MXFP4,
                           latent_format=synth.LATENT_NVFP4, heavy_tail=0.1)
    dc, scores, idx, o, l = _run_step_bf16(case)
    check_scores_bf16(case, scores)
    np.testing.assert_array_equal(idx, oracle.topk(_values(scores), case.row_lens(), case.topk))
    check_mla(case, idx, o, l)
