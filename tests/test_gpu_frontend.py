"""GPU parity of the fused indexer front end (dsa_index_frontend) and of the
decode step that owns its cache update (dsa_decode_step_frontend).

Protocol (as for the top-k on the GPU's scores): the projected query q that
the kernel accumulates in fp32 is checked against the oracle's fp64
projection of the oracle's normalised query within a derived tolerance; the
FP8 codes and folded head weights are checked bit for bit against the
oracle's quantisation of the kernel's own q (the same fp32 decision on both
sides); the cache bytes are checked bit for bit against the oracle's write.

Tolerance of q[r][o] = sum_i W[o][i] xn[r][i] (D terms):
  * fp32 accumulation: one rounding of at most 2^-24 per K = 16 MMA step, D/16
    steps (96 for D = 1,536) -> under 6e-6 A, doubled for the products'
    alignment inside a step and rounded up: 2e-5 A, A = sum_i |W[o][i] xn[r][i]|;
  * the norm: the kernel's RMS factor is fp32 (relative error a few 1e-6), so
    an xn element whose exact value lies within 3e-5 (relative) of a bf16
    rounding boundary may round the other way: each such element adds
    |W[o][i]| times its bf16 spacing.
"""
import numpy as np
import pytest
import torch

import oracle
from dsa_sparse_attention_index_gb300 import binding, synth
from test_gpu_parity import _scores_buf, _status, check_mla, check_scores

pytestmark = pytest.mark.gpu


def _t(a, dtype=None):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


def _bf16_value(bits):
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def _q_tolerance(fe, xn_bits):
    """Per (row, output) tolerance of the fp32 projection (module docstring)."""
    W = _bf16_value(fe.w_iq)
    xn = _bf16_value(xn_bits)
    A = np.abs(xn) @ np.abs(W).T
    c = _bf16_value(fe.c_q)
    g = _bf16_value(fe.gamma)
    inv = 1.0 / np.sqrt((c * c).mean(axis=1, keepdims=True) + fe.eps)
    x64 = c * inv * g
    lo = oracle.round_bf16(x64 * (1.0 - 3e-5))
    hi = oracle.round_bf16(x64 * (1.0 + 3e-5))
    near = lo != hi
    _, e = np.frexp(np.abs(x64))
    ulp = np.ldexp(1.0, e - 8)
    flips = np.where(near, ulp, 0.0)
    return 2e-5 * A + flips @ np.abs(W).T


def _run_frontend(case, fe):
    dc = synth.device_case(case)
    rows = case.rows
    if case.key_format == synth.KEY_MXFP4_NATIVE:   # codes [rows][32][64], then E8M0 [rows][32][4]
        q_index = torch.empty(rows * 32 * 68, dtype=torch.uint8, device="cuda")
    else:
        q_index = torch.empty((rows, 32, 128), dtype=torch.uint8, device="cuda")
    w_out = torch.empty((rows, 32), dtype=torch.float32, device="cuda")
    q_proj = torch.empty((rows, 4096), dtype=torch.float32, device="cuda")
    st = _status()
    n0 = binding.kernel_launches()
    binding.index_frontend(dc.cache, dc.batch, _t(fe.c_q), _t(fe.gamma), fe.eps, _t(fe.w_iq), _t(fe.head_w),
                           _t(fe.new_latent), _t(fe.new_key), q_index, w_out, st, q_proj=q_proj)
    torch.cuda.synchronize()
    assert binding.kernel_launches() - n0 == 1
    assert st.item() == 0, binding.status_string(st.item())
    return dc, q_index.cpu().numpy(), w_out.cpu().numpy(), q_proj.cpu().numpy()


@pytest.mark.parametrize("lens,nq,dim,fmt,lfmt", [
    ([3000, 700, 1500], 1, 1536, synth.KEY_FP8, synth.LATENT_FP8),        # 3 rows, N padded to 16
    ([9000] * 16, 4, 1536, synth.KEY_FP8, synth.LATENT_FP8),             # 64 rows: one full row group
    ([5000] * 65, 1, 512, synth.KEY_MXFP4, synth.LATENT_FP8),            # 65 rows: a second group of 1
    ([4000] * 35, 4, 64, synth.KEY_FP8, synth.LATENT_NVFP4),             # 140 rows, one K stage
    ([300], 1, 2048, synth.KEY_MXFP4, synth.LATENT_NVFP4),               # 1 row, more stages than the ring
    ([5000] * 65, 1, 512, synth.KEY_MXFP4_NATIVE, synth.LATENT_FP8),     # the query in MXFP4
    ([700, 64, 65], 4, 1536, synth.KEY_MXFP4_NATIVE, synth.LATENT_NVFP4),
])
def test_frontend_matches_oracle(lens, nq, dim, fmt, lfmt):
    case = synth.make_case("fe", seq_lens=lens, nq=nq, key_format=fmt, seed=len(lens) + dim, latent_format=lfmt)
    fe = synth.make_frontend(case.rows, dim=dim, seed=dim + nq)
    pool_ref = oracle.cache_append(case, fe.new_latent, fe.new_key)
    dc, codes, w_out, q_proj = _run_frontend(case, fe)
    # the projection against the oracle's fp64 one
    xn = oracle.rms_norm_bf16(fe.c_q, fe.gamma, fe.eps)
    q_ref = oracle.index_query_proj(xn, fe.w_iq)
    tol = _q_tolerance(fe, xn)
    err = np.abs(q_proj.astype(np.float64) - q_ref)
    assert (err <= tol).all(), f"max excess {np.max(err - tol)} at {np.unravel_index(np.argmax(err - tol), err.shape)}"
    # codes and folded weights: the oracle's quantisation of the kernel's own q, bit for bit
    if fmt == synth.KEY_MXFP4_NATIVE:
        codes_ref, w_ref = oracle.quantize_query_mxfp4(q_proj.reshape(-1, 32, 128), fe.head_w)
    else:
        codes_ref, w_ref = oracle.quantize_query_f32(q_proj.reshape(-1, 32, 128), fe.head_w)
    np.testing.assert_array_equal(codes, codes_ref)
    np.testing.assert_array_equal(w_out, w_ref)
    # the new tokens in the cache, bit for bit
    got_pool = dc.cache.pool.cpu().numpy()
    bad = np.argwhere(got_pool != pool_ref)
    assert bad.size == 0, f"{len(bad)} cache bytes differ, first at {bad[:4].tolist()}"


def test_frontend_reports_a_bad_block():
    case = synth.make_case("feb", seq_lens=[100, 200], key_format=synth.KEY_FP8, seed=2)
    case.block_table[1, 3] = case.num_blocks + 3          # token 199 of sequence 1 (block 3)
    fe = synth.make_frontend(case.rows, dim=256, seed=1)
    dc = synth.device_case(case)
    q_index = torch.empty((2, 32, 128), dtype=torch.uint8, device="cuda")
    w_out = torch.empty((2, 32), dtype=torch.float32, device="cuda")
    st = _status()
    binding.index_frontend(dc.cache, dc.batch, _t(fe.c_q), _t(fe.gamma), fe.eps, _t(fe.w_iq), _t(fe.head_w),
                           _t(fe.new_latent), _t(fe.new_key), q_index, w_out, st)
    torch.cuda.synchronize()
    assert st.item() == binding.ERR_BOUNDS


@pytest.mark.parametrize("fmt,nq", [(synth.KEY_FP8, 1), (synth.KEY_FP8, 4), (synth.KEY_MXFP4, 1),
                                    (synth.KEY_MXFP4_NATIVE, 1)])
def test_step_that_owns_its_cache_update_in_one_call(fmt, nq):
    """dsa_decode_step_frontend: the front end then the fused step, one call,
    one launch more than the step; its outputs equal dsa_decode_step's on the front end's
    query and updated cache bit for bit, and every stage matches the oracle
    on the updated cache."""
    lens = [9000, 4100, 2600]
    case = synth.make_case("feo", seq_lens=lens, nq=nq, key_format=fmt, seed=40 + nq)
    fe = synth.make_frontend(case.rows, dim=1536, seed=7 + nq)
    k, rows = case.topk, case.rows
    ld = (case.max_len + 3) // 4 * 4
    # the one-call step
    dc = synth.device_case(case)
    out = torch.empty((rows, 96, 512), dtype=torch.int16, device="cuda")
    lse = torch.empty((rows, 96), dtype=torch.float32, device="cuda")
    scores = _scores_buf(rows, ld)
    idx = torch.empty((rows, k), dtype=torch.int32, device="cuda")
    ws = binding.workspace(binding.frontend_workspace_size(dc.batch, k))
    st = _status()
    n0 = binding.kernel_launches()
    binding.decode_step_frontend(dc.cache, dc.batch, _t(fe.c_q), _t(fe.gamma), fe.eps, _t(fe.w_iq), _t(fe.head_w),
                                 _t(fe.new_latent), _t(fe.new_key), dc.q_mla, k, case.sm_scale, out, lse, ws, st,
                                 scores_out=scores, idx_out=idx)
    torch.cuda.synchronize()
    launches = binding.kernel_launches() - n0
    assert st.item() == 0, binding.status_string(st.item())
    # the same through the two calls: front end, then dsa_decode_step on its outputs
    dc2, codes, w_out, _ = _run_frontend(case, fe)
    np.testing.assert_array_equal(dc.cache.pool.cpu().numpy(), dc2.cache.pool.cpu().numpy())
    out2 = torch.empty_like(out)
    lse2 = torch.empty_like(lse)
    ws2 = binding.workspace(binding.workspace_size(dc2.batch, k))
    n0 = binding.kernel_launches()
    binding.decode_step(dc2.cache, dc2.batch, _t(codes), _t(w_out), dc2.q_mla, k, case.sm_scale, out2, lse2, ws2, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert launches == binding.kernel_launches() - n0 + 1     # the step's launches and the front end
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
    # every stage against the oracle on the updated cache and the front end's query
    case.pool = oracle.cache_append(case, fe.new_latent, fe.new_key)
    case.q_index, case.head_w = codes, w_out
    check_scores(case, scores)
    s64 = scores.cpu().numpy().astype(np.float64)
    idx_np = idx.cpu().numpy()
    np.testing.assert_array_equal(idx_np, oracle.topk(s64, case.row_lens(), k))
    check_mla(case, idx_np, out.view(torch.bfloat16).float().cpu().numpy(), lse.cpu().numpy())
