"""Pins for the fp64 oracle: each test ties an oracle function to something
other than itself (a library decoder, exact integer arithmetic, a closed
form, a brute-force property, or a library softmax), chosen so that a
plausible mistake (dropped term, wrong sign, wrong index, swapped operand)
fails at least one of them.  CPU only."""
import copy
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from dsa_sparse_attention_index_gb300 import synth


# --------------------------------------------------------------- formats
def test_e4m3_decode_matches_torch_for_all_codes():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_to_double(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert nan.sum() == 2  # 0x7F and 0xFF
    assert np.array_equal(ref[~nan], got[~nan])
    assert np.nanmax(got) == 448.0 and oracle.e4m3_to_double(0x01) == 2.0 ** -9


def test_e2m1_decode_is_the_ocp_mx_table():
    # OCP MX v1.0, FP4 E2M1: exponent bias 1, one mantissa bit, no inf/NaN.
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for c in range(16):
        want = mags[c & 7] * (-1.0 if c & 8 else 1.0)
        assert oracle.e2m1_to_double(c) == want
    # torch's own E2M1 container, when present, agrees on the packed nibbles
    if hasattr(torch, "float4_e2m1fn_x2"):
        try:
            packed = torch.arange(256, dtype=torch.uint8).view(torch.float4_e2m1fn_x2)
            _ = packed.to(torch.float32)  # conversion may be unsupported
        except Exception:
            pass


def test_e8m0_decode_is_power_of_two():
    for c in range(255):
        assert oracle.e8m0_to_double(c) == math.ldexp(1.0, c - 127)
    assert math.isnan(oracle.e8m0_to_double(255))


def test_bf16_decode_matches_torch():
    rng = np.random.default_rng(5)
    bits = rng.integers(0, 1 << 16, size=4000, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.bf16_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])


def test_mxfp4_round_trip_is_nearest_representable():
    rng = np.random.default_rng(11)
    x = rng.standard_normal((200, 128))
    packed, e8 = synth.mxfp4_encode(x)
    for i in range(0, 200, 17):
        for d in range(128):
            nib = packed[i, d // 2] & 0xF if d % 2 == 0 else packed[i, d // 2] >> 4
            v = oracle.e8m0_to_double(int(e8[i, d // 32])) * oracle.e2m1_to_double(int(nib))
            scale = oracle.e8m0_to_double(int(e8[i, d // 32]))
            # quantisation error at most half a grid step (largest step 2 x scale), or clamp
            assert abs(v - x[i, d]) <= scale * 1.0 + 1e-12 or abs(x[i, d]) > 6 * scale


# --------------------------------------------------------------- indexer
def _decode_key_fp8(case, b, t):
    r = case.block_table[b, t // 64]
    page = case.pool[r, case.index_off:]
    codes = page[(t % 64) * 128:(t % 64) * 128 + 128]
    scale = page[64 * 128 + (t % 64) * 4:64 * 128 + (t % 64) * 4 + 4].view(np.float32)[0]
    return codes, float(scale)


def _e4m3_int(codes):
    """E4M3 values times 2^9 as exact Python ints (via torch's decoder)."""
    v = torch.from_numpy(np.asarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return [int(round(x * 512)) for x in v]


@pytest.fixture(scope="module")
def small_case():
    return synth.make_case("pin", seq_lens=[200, 75], nq=1, topk=16, seed=3, spare_blocks=2)


def test_index_scores_exact_integer_dot(small_case):
    """With w = e_h the score is max(0, scale * q_h.k_t): check it against an
    exact integer dot product for every head and several tokens."""
    c = copy.deepcopy(small_case)
    for h in (0, 7, 31):
        c.head_w = np.zeros_like(c.head_w)
        c.head_w[:, h] = 1.0
        s = oracle.index_scores(c)
        for b in range(c.batch):
            qi = _e4m3_int(c.q_index[b, h])
            for t in (0, 1, 63, 64, int(c.seq_lens[b]) - 1):
                codes, scale = _decode_key_fp8(c, b, t)
                dot = Fraction(sum(a * k for a, k in zip(qi, _e4m3_int(codes))), 512 * 512)
                want = max(Fraction(0), Fraction(scale) * dot)
                assert s[b, t] == float(want)


def test_index_score_bounds_are_the_absolute_sums(small_case):
    """A_t = sum_h |w_h| |scale_t| sum_d |q_hd k_td| (the tolerances' scale):
    exact integer sums of absolute products, and never below |s_t|."""
    c = small_case
    bnd = oracle.index_score_bounds(c)
    s = oracle.index_scores(c)
    for b in range(c.batch):
        for t in (0, 5, 64, int(c.seq_lens[b]) - 1):
            codes, scale = _decode_key_fp8(c, b, t)
            k = _e4m3_int(codes)
            want = Fraction(0)
            for h in range(32):
                qi = _e4m3_int(c.q_index[b, h])
                want += abs(Fraction(float(c.head_w[b, h]))) * abs(Fraction(scale)) * Fraction(
                    sum(abs(a * x) for a, x in zip(qi, k)), 512 * 512)
            assert bnd[b, t] == pytest.approx(float(want), rel=1e-14)
            assert abs(s[b, t]) <= bnd[b, t] * (1 + 1e-14)


def test_index_scores_one_hot_closed_form(small_case):
    c = copy.deepcopy(small_case)
    h, d = 5, 77
    c.q_index = np.zeros_like(c.q_index)
    c.q_index[:, h, d] = 0x38  # E4M3 code of 1.0
    c.head_w = np.zeros_like(c.head_w)
    c.head_w[:, h] = -2.0      # a negative weight keeps the ReLU inside the sum
    s = oracle.index_scores(c)
    for b in range(c.batch):
        for t in range(int(c.seq_lens[b])):
            codes, scale = _decode_key_fp8(c, b, t)
            kd = _e4m3_int(codes[d:d + 1])[0] / 512.0
            assert s[b, t] == -2.0 * max(0.0, scale * kd)


def test_index_scores_zero_weights_and_head_permutation(small_case):
    c = copy.deepcopy(small_case)
    c.head_w = np.zeros_like(c.head_w)
    s = oracle.index_scores(c)
    assert np.all(s[0, :200] == 0) and np.all(s[1, :75] == 0)
    base = oracle.index_scores(small_case)
    perm = np.random.default_rng(1).permutation(32)
    c = copy.deepcopy(small_case)
    c.q_index = c.q_index[:, perm]
    c.head_w = c.head_w[:, perm]
    s = oracle.index_scores(c)
    np.testing.assert_allclose(s[0, :200], base[0, :200], rtol=1e-14, atol=1e-12)
    # pairing q_h with a different head's weight would change the scores
    c.head_w = c.head_w[:, ::-1].copy()
    assert not np.allclose(oracle.index_scores(c)[0, :200], base[0, :200])


def test_index_scores_block_table_permutation_invariance():
    a = synth.make_case("pa", seq_lens=[300, 130], permute_blocks=False, seed=9)
    b = synth.make_case("pb", seq_lens=[300, 130], permute_blocks=True, seed=9)
    # same logical contents, different physical rows
    sa, sb = oracle.index_scores(a), oracle.index_scores(b)
    assert np.array_equal(sa[0, :300], sb[0, :300]) and np.array_equal(sa[1, :130], sb[1, :130])
    assert not np.array_equal(a.block_table, b.block_table)


def test_index_scores_visibility_and_scale_sign():
    c = synth.make_case("vis", seq_lens=[100], nq=4, seed=2)
    s = oracle.index_scores(c)
    for j in range(4):
        n = 100 - 3 + j
        assert np.all(np.isfinite(s[j, :n])) and np.all(np.isnan(s[j, n:]))
    # scale inside the ReLU: a negative per-token scale flips which heads pass
    c1 = copy.deepcopy(c)
    r = c1.block_table[0, 0]
    off = c1.index_off + 64 * 128
    sc = c1.pool[r, off:off + 4].view(np.float32).copy()
    c1.pool[r, off:off + 4] = (-sc).view(np.uint8)
    s1 = oracle.index_scores(c1)
    c1.head_w = np.zeros_like(c1.head_w)
    c1.head_w[:, 3] = 1.0
    c2 = copy.deepcopy(c1)
    c2.pool[r, off:off + 4] = sc.view(np.uint8)
    one_neg, one_pos = oracle.index_scores(c1)[0, 0], oracle.index_scores(c2)[0, 0]
    assert (one_neg == 0.0) != (one_pos == 0.0) or (one_neg == 0.0 and one_pos == 0.0)
    assert s1[0, 1] == s[0, 1]  # other tokens unaffected


def test_index_scores_mxfp4_exact_rational():
    c = synth.make_case("mx", seq_lens=[130], key_format=synth.KEY_MXFP4, seed=4)
    c.head_w = np.zeros_like(c.head_w)
    c.head_w[:, 9] = 1.0
    s = oracle.index_scores(c)
    bnd = oracle.index_score_bounds(c)
    qi = _e4m3_int(c.q_index[0, 9])
    for t in (0, 5, 64, 129):
        r = c.block_table[0, t // 64]
        page = c.pool[r, c.index_off:]
        packed = page[(t % 64) * 64:(t % 64) * 64 + 64]
        e8 = page[64 * 64 + (t % 64) * 4:64 * 64 + (t % 64) * 4 + 4]
        two_k = []
        for d in range(128):
            nib = packed[d // 2] & 0xF if d % 2 == 0 else packed[d // 2] >> 4
            mag = [0, 1, 2, 3, 4, 6, 8, 12][nib & 7] * (-1 if nib & 8 else 1)  # 2 x E2M1
            two_k.append(Fraction(mag, 2) * Fraction(2) ** (int(e8[d // 32]) - 127))
        dot = sum(Fraction(a, 512) * k for a, k in zip(qi, two_k))
        assert s[0, t] == float(max(Fraction(0), dot))
        # the tolerance scale: the sum of absolute products (scale_t = 1)
        assert bnd[0, t] == pytest.approx(float(sum(abs(Fraction(a, 512) * k) for a, k in zip(qi, two_k))), rel=1e-14)


# --------------------------------------------------------------- top-k
def _is_valid_topk(scores, n, k, out):
    sel = [int(i) for i in out if i >= 0]
    assert len(sel) == min(k, n)
    assert sel == sorted(sel) and len(set(sel)) == len(sel)
    assert all(i == -1 for i in out[len(sel):])

    def key(t):
        v = scores[t]
        return (0 if np.isnan(v) else 1, 0.0 if np.isnan(v) else v, -t)

    rest = set(range(n)) - set(sel)
    if sel and rest:
        assert min(key(t) for t in sel) > max(key(t) for t in rest)


def test_topk_brute_force_property_with_ties():
    rng = np.random.default_rng(0)
    for trial in range(300):
        n = int(rng.integers(0, 14))
        k = int(rng.integers(1, 7))
        vals = rng.choice([-1.0, 0.0, -0.0, 0.5, 2.0, np.nan], size=n)
        row = np.full((1, 16), 7.0)
        row[0, :n] = vals
        out = oracle.topk(row, np.array([n]), k)[0]
        _is_valid_topk(row[0], n, k, out)


def test_topk_special_cases():
    s = np.zeros((1, 5000))
    assert list(oracle.topk(s, np.array([5000]), 2048)[0]) == list(range(2048))
    s = np.random.default_rng(1).standard_normal((1, 100))
    out = oracle.topk(s, np.array([100]), 128)[0]
    assert list(out[:100]) == list(range(100)) and np.all(out[100:] == -1)
    assert np.all(oracle.topk(s, np.array([0]), 4)[0] == -1)
    s = np.array([[np.nan, -np.inf, -0.0, 0.0, 1.0]])
    assert list(oracle.topk(s, np.array([5]), 3)[0]) == [2, 3, 4]
    assert list(oracle.topk(s, np.array([5]), 4)[0]) == [1, 2, 3, 4]


def test_topk_matches_python_sort_on_random_rows():
    rng = np.random.default_rng(2)
    s = rng.standard_normal((4, 3000)).astype(np.float32).astype(np.float64)
    s[:, ::7] = s[:, 3:4]  # heavy duplicates around arbitrary values
    lens = np.array([3000, 2500, 17, 2049])
    got = oracle.topk(s, lens, 2048)
    for r in range(4):
        n = int(lens[r])
        want = sorted(sorted(range(n), key=lambda t: (-s[r, t], t))[:2048])
        assert list(got[r, :len(want)]) == want
        _is_valid_topk(s[r], n, 2048, got[r])


@pytest.mark.parametrize("seg", [97, 500, 2048])
def test_topk_of_segment_topks_is_the_topk(seg):
    """The decomposition the two-level selection of long rows rests on: the
    top-k of a row equals the top-k over the union of its segments' top-k,
    with the union kept in token order so that ties still go to the lower
    index (ties within and across segments, NaN, a short last segment)."""
    rng = np.random.default_rng(seg)
    k = 64
    for trial in range(20):
        n = int(rng.integers(1, 4000))
        row = rng.choice([0.0, 1.0, 2.0, np.nan, -1.0], size=n) + (rng.random(n) < 0.5) * rng.standard_normal(n)
        s = row[None, :]
        want = oracle.topk(s, np.array([n]), k)[0]
        cand = []
        for p0 in range(0, n, seg):
            part = row[p0:p0 + seg]
            sel = oracle.topk(part[None, :], np.array([part.size]), k)[0]
            cand += [p0 + int(t) for t in sel if t >= 0]
        cand = np.array(cand)                        # ascending: segments in order, each ascending
        assert np.all(np.diff(cand) > 0)
        sub = oracle.topk(row[cand][None, :], np.array([cand.size]), k)[0]
        got = np.array([cand[t] if t >= 0 else -1 for t in sub])
        np.testing.assert_array_equal(got, want)


# --------------------------------------------------------------- sparse MLA
def _latent(case, b, t):
    r = case.block_table[b, t // 64]
    row = case.pool[r, case.latent_off + (t % 64) * 576:case.latent_off + (t % 64) * 576 + 576]
    return torch.from_numpy(row.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy() * case.latent_scale


def _q(case, row):
    return torch.from_numpy(case.q_mla[row].view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()


@pytest.fixture(scope="module")
def mla_case():
    return synth.make_case("mla", seq_lens=[300, 90], nq=1, topk=64, seed=6)


def test_sparse_mla_matches_library_softmax(mla_case):
    c = mla_case
    rng = np.random.default_rng(3)
    idx = np.full((2, 64), -1, dtype=np.int32)
    idx[0] = np.sort(rng.choice(300, 64, replace=False))
    idx[1, :40] = np.sort(rng.choice(90, 40, replace=False))
    out, lse = oracle.sparse_mla(c, idx)
    for row in range(2):
        sel = [t for t in idx[row] if t >= 0]
        C = torch.from_numpy(np.stack([_latent(c, row, t) for t in sel]))
        Q = torch.from_numpy(_q(c, row))
        logits = (Q @ C.T) * c.sm_scale
        ref = torch.softmax(logits, dim=-1) @ C[:, :512]
        np.testing.assert_allclose(out[row], ref.numpy(), rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(lse[row], torch.logsumexp(logits, dim=-1).numpy(), rtol=1e-12)


def test_sparse_mla_closed_forms(mla_case):
    c = copy.deepcopy(mla_case)
    idx = np.full((2, 64), -1, dtype=np.int32)
    idx[0, 0] = 17          # one selected token: O = its value row, LSE = its logit
    out, lse = oracle.sparse_mla(c, idx)
    v = _latent(c, 0, 17)
    q = _q(c, 0)
    np.testing.assert_array_equal(out[0], np.broadcast_to(v[:512], (96, 512)))
    np.testing.assert_allclose(lse[0], c.sm_scale * (q @ v), rtol=1e-13,
                               atol=1e-14 * c.sm_scale * float(np.max(np.abs(q) @ np.abs(v))))
    assert np.all(out[1] == 0) and np.all(np.isneginf(lse[1]))   # no valid entry
    c.q_mla = np.zeros_like(c.q_mla)   # q = 0: uniform weights
    idx[1, :10] = np.arange(10) * 9
    out, lse = oracle.sparse_mla(c, idx)
    mean = np.mean([_latent(c, 1, t)[:512] for t in idx[1, :10]], axis=0)
    np.testing.assert_allclose(out[1], np.broadcast_to(mean, (96, 512)), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse[1], math.log(10), rtol=1e-14)


def test_sparse_mla_rejects_invisible_token(mla_case):
    idx = np.full((2, 64), -1, dtype=np.int32)
    idx[1, 0] = 95  # sequence 1 has 90 tokens
    with pytest.raises(oracle.OracleError):
        oracle.sparse_mla(mla_case, idx)


def test_decode_step_composes_the_three_stages():
    c = synth.make_case("step", seq_lens=[700], nq=2, topk=128, seed=8)
    s, idx, out, lse = oracle.decode_step(c)
    assert idx.shape == (2, 128)
    # row 0 sees 699 tokens, row 1 sees 700
    assert np.isnan(s[0, 699]) and np.isfinite(s[1, 699])
    for r in range(2):
        _is_valid_topk(s[r], int(c.row_lens()[r]), 128, idx[r])
    o2, l2 = oracle.sparse_mla(c, idx)
    assert np.array_equal(o2, out) and np.array_equal(l2, lse)


# ---------------------------------------------------------------- new-token write and FP8 query
def _bf16_bits(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _bf16_value(bits):
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32)


def _torch_e4m3(x):
    t = torch.from_numpy(np.clip(np.asarray(x, dtype=np.float32), -448.0, 448.0))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


_E2M1_MAG = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _e2m1_brute(x):
    """Nearest E2M1 code by search, ties to the even code, saturating at 6."""
    a = min(abs(x), 6.0)
    d = np.abs(_E2M1_MAG - a)
    best = [c for c in range(8) if d[c] == d.min()]
    c = min(best, key=lambda c: (c % 2, c))
    return c | (8 if np.signbit(x) else 0)


def test_e4m3_encode_matches_torch():
    rng = np.random.default_rng(11)
    x = np.concatenate([
        rng.standard_normal(4000) * np.exp(rng.uniform(-14, 7, 4000)),
        [0.0, -0.0, 448.0, 449.0, 464.0, 1e6, -1e6, 2.0 ** -9, 2.0 ** -10, 3 * 2.0 ** -11],
        # exact midpoints between neighbouring codes (ties to even)
        [(oracle.e4m3_to_double(c) + oracle.e4m3_to_double(c + 1)) / 2 for c in range(0, 0x7E)],
    ]).astype(np.float32)
    got = np.array([oracle.e4m3_encode(float(v)) for v in x], dtype=np.uint8)
    np.testing.assert_array_equal(got, _torch_e4m3(x))


def test_e2m1_encode_is_nearest_ties_even():
    vals = list(np.arange(-9, 9, 1 / 64)) + [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.0, 6.0, 7.0, 100.0]
    for v in vals:
        assert oracle.e2m1_encode(float(v)) == _e2m1_brute(float(v)), v


@pytest.mark.parametrize("fmt", [synth.KEY_FP8, synth.KEY_MXFP4])
def test_cache_append_writes_nearest_codes(fmt):
    case = synth.make_case("app", seq_lens=[130, 64], nq=3, key_format=fmt, seed=4)
    rng = np.random.default_rng(5)
    lat = rng.standard_normal((case.rows, 576)).astype(np.float32) * 3
    key = rng.standard_normal((case.rows, 128)).astype(np.float32)
    key[1] = 0.0                               # an all-zero key
    key[2, :32] *= 1e-30                       # a block of tiny values
    lat[0, :5] = [1e6, -1e6, 0.0, -0.0, 1e-30]
    lat_b, key_b = _bf16_bits(lat), _bf16_bits(key)
    lat, key = _bf16_value(lat_b), _bf16_value(key_b)
    pool = oracle.cache_append(case, lat_b, key_b)
    changed = np.zeros_like(pool, dtype=bool)
    for b in range(case.batch):
        for j in range(case.nq):
            nr = b * case.nq + j
            t = int(case.seq_lens[b]) - case.nq + j
            r = case.block_table[b, t // 64]
            slot = t % 64
            lat_codes = pool[r, case.latent_off + slot * 576:case.latent_off + (slot + 1) * 576]
            np.testing.assert_array_equal(lat_codes, _torch_e4m3(lat[nr] / np.float32(case.latent_scale)))
            changed[r, case.latent_off + slot * 576:case.latent_off + (slot + 1) * 576] = True
            page = pool[r, case.index_off:]
            if fmt == synth.KEY_FP8:
                amax = np.float32(np.abs(key[nr]).max())
                s = amax / np.float32(448.0) if amax > 0 else np.float32(1.0)
                np.testing.assert_array_equal(page[slot * 128:(slot + 1) * 128], _torch_e4m3(key[nr] / s))
                assert page[64 * 128 + 4 * slot:64 * 128 + 4 * slot + 4].view(np.float32)[0] == s
                changed[r, case.index_off + slot * 128:case.index_off + (slot + 1) * 128] = True
                changed[r, case.index_off + 64 * 128 + 4 * slot:case.index_off + 64 * 128 + 4 * slot + 4] = True
            else:
                for blk in range(4):
                    xs = key[nr, 32 * blk:32 * blk + 32].astype(np.float64)
                    amax = np.abs(xs).max()
                    e = -127 if amax == 0 else max(-127, min(127, int(np.floor(np.log2(amax))) - 2))
                    assert page[64 * 64 + 4 * slot + blk] == e + 127
                    packed = page[slot * 64 + 16 * blk:slot * 64 + 16 * blk + 16]
                    codes = np.stack([packed & 0xF, packed >> 4], axis=1).reshape(-1)
                    assert [int(c) for c in codes] == [_e2m1_brute(float(v) * 2.0 ** -e) for v in xs]
                changed[r, case.index_off + slot * 64:case.index_off + (slot + 1) * 64] = True
                changed[r, case.index_off + 64 * 64 + 4 * slot:case.index_off + 64 * 64 + 4 * slot + 4] = True
    np.testing.assert_array_equal(pool[~changed], case.pool[~changed])  # nothing else is touched


def test_quantize_query_folds_the_scale():
    rng = np.random.default_rng(8)
    q = rng.standard_normal((3, 32, 128)).astype(np.float32) * np.exp(rng.uniform(-3, 3, (3, 32, 1)))
    q[0, 5] = 0.0
    q_b = _bf16_bits(q)
    q = _bf16_value(q_b)
    w = rng.standard_normal((3, 32)).astype(np.float32)
    codes, w_out = oracle.quantize_query(q_b, w)
    amax = np.abs(q).max(axis=2)
    s = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    np.testing.assert_array_equal(codes, _torch_e4m3(q / s[..., None]))
    np.testing.assert_array_equal(w_out, (w * s).astype(np.float32))


# ---------------------------------------------------------------- DCP top-k merge
def _bf16_round(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).to(torch.float32).numpy()


@pytest.mark.parametrize("shards", [1, 2, 3, 5, 8])
def test_dcp_topk_is_the_topk_of_bf16_scores(shards):
    """The shard-wise candidates, the merge and the resends give exactly the
    top-k of the bf16-rounded scores with ties to the lower index (a full
    sort, the plain top-k)."""
    rng = np.random.default_rng(shards)
    n = 7000
    s = np.zeros((6, n), dtype=np.float32)
    s[0] = rng.standard_normal(n)
    s[1] = rng.integers(0, 40, n)                      # heavy ties
    s[2] = rng.standard_normal(n) * 1e-3 + 1.0          # ties only after bf16 rounding
    s[3] = rng.standard_normal(n)
    s[3, [5, 77, 900]] = [np.nan, -0.0, np.inf]
    s[3, 1000:1010] = 0.0
    s[4] = -rng.exponential(1.0, n)
    s[5] = rng.standard_normal(n)
    lens = np.array([n, n - 1, n - 7, 2048, 2049, 1000], dtype=np.int32)
    got, _ = oracle.dcp_topk(s, lens, 2048, shards)
    ref = oracle.topk(_bf16_round(s).astype(np.float64), lens, 2048)
    np.testing.assert_array_equal(got, ref)


@pytest.mark.parametrize("shards", [2, 4, 8])
def test_dcp_topk_resend_when_one_shard_holds_the_top(shards):
    """Every token of shard 0 outscores the rest: shard 0's candidates are all
    taken, so it resends its full local top-k and the result stays exact."""
    rng = np.random.default_rng(10 + shards)
    n = 40_000
    s = rng.standard_normal((2, n)).astype(np.float32)
    s[0, ::shards] += 100.0
    lens = np.array([n, n], dtype=np.int32)
    got, stats = oracle.dcp_topk(s, lens, 2048, shards)
    np.testing.assert_array_equal(got, oracle.topk(_bf16_round(s).astype(np.float64), lens, 2048))
    c = -(-3 * 2048 // (2 * shards))
    assert stats[0, 1] == 1 and stats[0, 2] == 2048      # shard 0 resent its full local top-k
    assert stats[1, 1] == 0 and stats[0, 0] == stats[1, 0] == shards * c


def test_dcp_candidate_bytes_ten_times_fewer():
    """W = 8, k = 2048: each shard sends ceil(1.5 * 2048 / 8) = 384 words of
    4 bytes, against its full local top-k as (fp32 score, token id) pairs:
    16,384 B / 1,536 B = 10.7."""
    rng = np.random.default_rng(3)
    s = rng.standard_normal((1, 100_000)).astype(np.float32)
    _, stats = oracle.dcp_topk(s, np.array([100_000], dtype=np.int32), 2048, 8)
    per_shard = stats[0, 0] // 8 * 4
    assert per_shard == 1536 and stats[0, 1] == 0
    assert (2048 * 8) / per_shard > 10


# ---------------------------------------------------------------- DCP LSE combine
def _bf16_bits_round(x):
    """fp64 -> nearest bf16 by integer rounding of the IEEE bits (keep the top
    16 of 64 bits' worth of significand: drop 45 bits, ties to even); valid
    for normal values, an independent route to the oracle's rounding."""
    b = np.ascontiguousarray(x, dtype=np.float64).view(np.uint64)
    lsb = (b >> np.uint64(45)) & np.uint64(1)
    b = (b + np.uint64((1 << 44) - 1) + lsb) & ~np.uint64((1 << 45) - 1)
    return b.view(np.float64)


def test_round_bf16_matches_torch_and_bit_rounding():
    ties = np.array([1.0 + 2.0**-8, 1.0 + 3 * 2.0**-8, -(1.0 + 2.0**-8), 3.0 * 2.0**-9 + 1.0])
    np.testing.assert_array_equal(oracle.round_bf16(ties), [1.0, 1.0 + 2.0**-6, -1.0, 1.0 + 2.0**-7])
    rng = np.random.default_rng(5)
    x32 = (rng.standard_normal(200_000) * np.exp(rng.uniform(-20, 20, 200_000))).astype(np.float32)
    ref = torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(oracle.round_bf16(x32.astype(np.float64)), ref)
    x64 = rng.standard_normal(200_000) * np.exp(rng.uniform(-20, 20, 200_000))
    np.testing.assert_array_equal(oracle.round_bf16(x64), _bf16_bits_round(x64))


@pytest.fixture(scope="module")
def dcp_case():
    c = synth.make_case("dcpmla", seq_lens=[300, 90], nq=1, topk=64, seed=11)
    rng = np.random.default_rng(12)
    idx = np.full((2, 64), -1, dtype=np.int32)
    idx[0] = np.sort(rng.choice(300, 64, replace=False))
    idx[1, :37] = np.sort(rng.choice(90, 37, replace=False))
    return c, idx


@pytest.mark.parametrize("shards", [1, 2, 3, 8])
def test_dcp_sparse_mla_exact_partials_give_the_unsharded_softmax(dcp_case, shards):
    """With unrounded partials the LSE combine is an identity: the merged
    output and LSE are the softmax attention over all selected tokens
    (torch's softmax and logsumexp in fp64), and shard w's LSE is the
    logsumexp over the selected tokens t with t mod W = w."""
    c, idx = dcp_case
    out, lse, O, L = oracle.dcp_sparse_mla(c, idx, shards, partial="f64")
    for row in range(2):
        sel = np.array([t for t in idx[row] if t >= 0])
        C = torch.from_numpy(np.stack([_latent(c, row, t) for t in sel]))
        Q = torch.from_numpy(_q(c, row))
        logits = (Q @ C.T) * c.sm_scale
        np.testing.assert_allclose(out[row], (torch.softmax(logits, dim=-1) @ C[:, :512]).numpy(),
                                   rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(lse[row], torch.logsumexp(logits, dim=-1).numpy(), rtol=1e-12)
        for w in range(shards):
            own = torch.from_numpy(sel % shards == w)
            if own.any():
                np.testing.assert_allclose(L[w, row], torch.logsumexp(logits[:, own], dim=-1).numpy(), rtol=1e-12)
            else:
                assert np.all(np.isneginf(L[w, row])) and np.all(O[w, row] == 0)


def test_dcp_sparse_mla_bf16_partials(dcp_case):
    """W = 1: the one partial is the whole output, so the result is the
    unsharded output rounded to bf16.  A shard that holds no selected token
    sends LSE = -inf and weighs nothing: with every selected token in shard
    0 the result is shard 0's rounded output."""
    c, idx = dcp_case
    ref_out, ref_lse = oracle.sparse_mla(c, idx)
    out, lse, _, _ = oracle.dcp_sparse_mla(c, idx, 1)
    np.testing.assert_array_equal(out, oracle.round_bf16(ref_out))
    np.testing.assert_array_equal(lse, ref_lse)
    only0 = np.where(idx % 4 == 0, idx, -1).astype(np.int32)
    out, lse, O, L = oracle.dcp_sparse_mla(c, only0, 4)
    o0, l0 = oracle.sparse_mla(c, only0)
    np.testing.assert_array_equal(out, oracle.round_bf16(o0))
    np.testing.assert_array_equal(lse, l0)
    assert np.all(np.isneginf(L[1:])) and np.all(O[1:] == 0)
    # the bf16 partials move the output by at most about one bf16 step of the largest |O_w|
    out8, _, O8, _ = oracle.dcp_sparse_mla(c, idx, 8)
    exact, _, _, _ = oracle.dcp_sparse_mla(c, idx, 8, partial="f64")
    assert np.all(np.abs(out8 - exact) <= 2.0**-8 * np.abs(O8).max(axis=0) + 1e-300)


# ---------------------------------------------------------------- NVFP4 latents
def _nvfp4_record_values(rec):
    """The 576 values (before latent_scale) of a 352-byte record, from torch's
    E4M3 decoder and the OCP E2M1 table: dims 0..511 scale x element, the
    rest E4M3 codes."""
    codes = np.stack([rec[:256] & 0xF, rec[:256] >> 4], axis=1).reshape(-1)
    e2m1 = np.where(codes & 8, -1.0, 1.0) * _E2M1_MAG[codes & 7]
    scale = torch.from_numpy(rec[256:288].copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    tail = torch.from_numpy(rec[288:352].copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return np.concatenate([e2m1 * np.repeat(scale, 16), tail])


def test_sparse_mla_nvfp4_single_token_closed_form():
    """One selected token: O is its value row exactly and LSE its logit;
    the record holds every E2M1 code in both nibbles, scales across the E4M3
    range (subnormal to 448) and E4M3 tail codes."""
    c = synth.make_case("nv1", seq_lens=[200, 90], nq=1, topk=8, seed=13, latent_format=synth.LATENT_NVFP4)
    rec = np.zeros(352, dtype=np.uint8)
    rec[:256] = [(i % 16) | (((7 * i + 3) % 16) << 4) for i in range(256)]
    rec[256:288] = [0x01, 0x07, 0x08, 0x30, 0x38, 0x40, 0x55, 0x7E, 0x81, 0xB8, 0xFE, 0x00, 0x02] + list(range(0x10, 0x80, 6))
    rec[288:352] = [(5 * i + 1) % 256 for i in range(64)]
    rec[288:352][rec[288:352] % 128 == 0x7F] = 0x11       # no NaN codes
    r = c.block_table[0, 17 // 64]
    off = c.latent_off + (17 % 64) * 352
    c.pool[r, off:off + 352] = rec
    idx = np.full((2, 8), -1, dtype=np.int32)
    idx[0, 0] = 17
    out, lse = oracle.sparse_mla(c, idx)
    v = _nvfp4_record_values(rec) * c.latent_scale
    np.testing.assert_array_equal(out[0], np.broadcast_to(v[:512], (96, 512)))
    q = _q(c, 0)
    np.testing.assert_allclose(lse[0], c.sm_scale * (q @ v), rtol=1e-13,
                               atol=1e-14 * c.sm_scale * float(np.max(np.abs(q) @ np.abs(v))))


def test_sparse_mla_nvfp4_matches_library_softmax():
    c = synth.make_case("nv2", seq_lens=[300, 90], nq=1, topk=64, seed=14, latent_format=synth.LATENT_NVFP4)
    rng = np.random.default_rng(4)
    idx = np.full((2, 64), -1, dtype=np.int32)
    idx[0] = np.sort(rng.choice(300, 64, replace=False))
    idx[1, :33] = np.sort(rng.choice(90, 33, replace=False))
    out, lse = oracle.sparse_mla(c, idx)
    for row in range(2):
        sel = [t for t in idx[row] if t >= 0]
        recs = []
        for t in sel:
            r = c.block_table[row, t // 64]
            o = c.latent_off + (t % 64) * 352
            recs.append(_nvfp4_record_values(c.pool[r, o:o + 352]) * c.latent_scale)
        C = torch.from_numpy(np.stack(recs))
        Q = torch.from_numpy(_q(c, row))
        logits = (Q @ C.T) * c.sm_scale
        np.testing.assert_allclose(out[row], (torch.softmax(logits, dim=-1) @ C[:, :512]).numpy(),
                                   rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(lse[row], torch.logsumexp(logits, dim=-1).numpy(), rtol=1e-12)


def test_cache_append_nvfp4_latents():
    """Block scale = torch's E4M3 of amax / (6 latent_scale) in fp32; codes =
    the brute-force nearest E2M1 of x / (latent_scale * scale); an all-zero
    block gets scale 0 and zero codes; the tail = torch's E4M3 of
    x / latent_scale; nothing else in the pool changes."""
    case = synth.make_case("appnv", seq_lens=[130, 64], nq=2, key_format=synth.KEY_MXFP4, seed=6,
                           latent_format=synth.LATENT_NVFP4)
    rng = np.random.default_rng(6)
    lat = rng.standard_normal((case.rows, 576)).astype(np.float32) * np.exp(rng.uniform(-4, 4, (case.rows, 36, 1))).repeat(16, axis=2).reshape(case.rows, 576).astype(np.float32)
    lat[0, 16:32] = 0.0                              # an all-zero block
    lat[1, :3] = [1e6, -1e6, 1e-30]                  # saturation and a tiny value
    key = rng.standard_normal((case.rows, 128)).astype(np.float32)
    lat_b, key_b = _bf16_bits(lat), _bf16_bits(key)
    lat = _bf16_value(lat_b)
    pool = oracle.cache_append(case, lat_b, key_b)
    ls = np.float32(case.latent_scale)
    changed = np.zeros_like(pool, dtype=bool)
    for b in range(case.batch):
        for j in range(case.nq):
            nr = b * case.nq + j
            t = int(case.seq_lens[b]) - case.nq + j
            r = case.block_table[b, t // 64]
            slot = t % 64
            o = case.latent_off + slot * 352
            rec = pool[r, o:o + 352]
            for blk in range(32):
                xs = lat[nr, 16 * blk:16 * blk + 16]
                sc = _torch_e4m3(np.array([np.abs(xs).max() / (np.float32(6.0) * ls)], dtype=np.float32))[0]
                assert rec[256 + blk] == sc
                sdec = np.float32(torch.from_numpy(np.array([sc], dtype=np.uint8)).view(torch.float8_e4m3fn).float().item())
                step = np.float32(ls * sdec)
                packed = rec[8 * blk:8 * blk + 8]
                codes = np.stack([packed & 0xF, packed >> 4], axis=1).reshape(-1)
                want = [_e2m1_brute(float(np.float32(v / step))) if sdec > 0 else 0 for v in xs]
                assert [int(c) for c in codes] == want, (nr, blk)
            np.testing.assert_array_equal(rec[288:], _torch_e4m3(lat[nr, 512:] / ls))
            changed[r, o:o + 352] = True
            changed[r, case.index_off + slot * 64:case.index_off + (slot + 1) * 64] = True
            changed[r, case.index_off + 64 * 64 + 4 * slot:case.index_off + 64 * 64 + 4 * slot + 4] = True
    np.testing.assert_array_equal(pool[~changed], case.pool[~changed])


def test_cache_append_nvfp4_agrees_with_the_input_generator():
    """The oracle's NVFP4 write (C, brute-force nearest codes) and the input
    generator's NVFP4 encoder (numpy/torch, midpoint search) implement the
    same rule independently: on bf16-valued latents they write the same
    352 bytes."""
    case = synth.make_case("nvx", seq_lens=[70], nq=1, key_format=synth.KEY_FP8, seed=9,
                           latent_format=synth.LATENT_NVFP4)
    rng = np.random.default_rng(9)
    lat = (rng.standard_normal((1, 576)) * np.exp(rng.uniform(-5, 5, (1, 36, 1))).repeat(16, 2).reshape(1, 576))
    lat_b = _bf16_bits(lat.astype(np.float32))
    key_b = _bf16_bits(rng.standard_normal((1, 128)).astype(np.float32))
    pool = oracle.cache_append(case, lat_b, key_b)
    t = 69
    r = case.block_table[0, t // 64]
    rec = pool[r, case.latent_off + (t % 64) * 352:case.latent_off + (t % 64 + 1) * 352]
    want = synth.nvfp4_latent_encode(_bf16_value(lat_b), case.latent_scale)[0]
    np.testing.assert_array_equal(rec, want)


# ---------------------------------------------------------------- fused indexer front end
def _bf16_from_f64_torch(x):
    """bf16 bits of fp64 values through torch's float64 -> bfloat16 rounding."""
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float64)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_rms_norm_matches_the_definition_through_torch():
    """xn = c / sqrt(mean(c^2) + eps) * gamma in fp64, rounded to bf16: the
    same values through torch's fp64 arithmetic and its bf16 rounding."""
    fe = synth.make_frontend(7, dim=256, seed=3)
    got = oracle.rms_norm_bf16(fe.c_q, fe.gamma, fe.eps)
    c = _bf16_value(fe.c_q).astype(np.float64)
    g = _bf16_value(fe.gamma).astype(np.float64)
    ct = torch.from_numpy(c)
    ref = ct / torch.sqrt((ct * ct).mean(dim=1, keepdim=True) + fe.eps) * torch.from_numpy(g)
    np.testing.assert_array_equal(got, _bf16_from_f64_torch(ref.numpy()))


def test_rms_norm_closed_forms():
    """A constant row a gives gamma * a / sqrt(a^2 + eps); eps = 0 makes the
    norm scale-invariant (rows c and 4c give the same xn); the sign of c
    carries through; gamma = 1, eps = 0 on a row of +-1 returns the row."""
    D = 64
    gamma = _bf16_bits(np.linspace(0.5, 1.5, D).astype(np.float32))
    g = _bf16_value(gamma).astype(np.float64)
    c = _bf16_bits(np.full((1, D), 3.0, dtype=np.float32))
    got = _bf16_value(oracle.rms_norm_bf16(c, gamma, 1e-6)[0]).astype(np.float64)
    want = _bf16_value(_bf16_from_f64_torch(g * 3.0 / math.sqrt(9.0 + 1e-6))).astype(np.float64)
    np.testing.assert_array_equal(got, want)
    rng = np.random.default_rng(5)
    x = rng.standard_normal((2, D)).astype(np.float32)
    c2 = _bf16_bits(np.stack([x[0], 4.0 * x[0], -x[1]]))
    out = oracle.rms_norm_bf16(c2, gamma, 0.0)
    np.testing.assert_array_equal(out[0], out[1])
    signs = np.sign(_bf16_value(out[2])) == np.sign(_bf16_value(c2[2]))   # gamma > 0: xn keeps c's sign
    assert signs[_bf16_value(c2[2]) != 0].all()
    ones = _bf16_bits(np.where(rng.random((1, D)) < 0.5, -1.0, 1.0).astype(np.float32))
    unit = _bf16_bits(np.ones(D, dtype=np.float32))
    np.testing.assert_array_equal(oracle.rms_norm_bf16(ones, unit, 0.0), ones)


def test_index_query_projection_exact_integers_and_one_hot_rows():
    """Small-integer operands make every dot product an exact integer (Python
    ints); a one-hot weight row copies one input; a row scaled by -2 flips the
    sign and doubles; against torch's fp64 matmul on random bf16 operands."""
    rng = np.random.default_rng(11)
    rows, D, outs = 3, 96, 40
    xi = rng.integers(-8, 9, (rows, D))
    wi = rng.integers(-8, 9, (outs, D))
    wi[5] = 0
    wi[5, 17] = 1                                          # one-hot: q[:, 5] = x[:, 17]
    wi[6] = -2 * wi[7]
    q = oracle.index_query_proj(_bf16_bits(xi.astype(np.float32)), _bf16_bits(wi.astype(np.float32)))
    want = [[sum(int(a) * int(b) for a, b in zip(xi[r], wi[o])) for o in range(outs)] for r in range(rows)]
    np.testing.assert_array_equal(q, np.array(want, dtype=np.float64))
    np.testing.assert_array_equal(q[:, 5], xi[:, 17].astype(np.float64))
    np.testing.assert_array_equal(q[:, 6], -2 * q[:, 7])
    fe = synth.make_frontend(4, dim=512, seed=9)
    xn = oracle.rms_norm_bf16(fe.c_q, fe.gamma, fe.eps)
    w = fe.w_iq[:200]
    got = oracle.index_query_proj(xn, w)
    ref = torch.from_numpy(_bf16_value(xn).astype(np.float64)) @ torch.from_numpy(_bf16_value(w).astype(np.float64)).T
    np.testing.assert_allclose(got, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_quantize_query_f32_folds_the_scale():
    """From fp32 query values: s = amax / 448 in fp32, codes = torch's E4M3 of
    q / s (fp32), w_out = w * s; an all-zero head takes s = 1; the bf16 entry
    point agrees on bf16-valued inputs."""
    rng = np.random.default_rng(13)
    q = (rng.standard_normal((4, 32, 128)) * np.exp(rng.uniform(-5, 5, (4, 32, 1)))).astype(np.float32)
    q[1, 2] = 0.0
    q[2, 3, :2] = [-0.0, 3.0e38]
    w = rng.standard_normal((4, 32)).astype(np.float32)
    codes, w_out = oracle.quantize_query_f32(q, w)
    amax = np.abs(q).max(axis=2)
    s = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    np.testing.assert_array_equal(codes, _torch_e4m3(q / s[..., None]))
    np.testing.assert_array_equal(w_out, (w * s).astype(np.float32))
    assert (codes[1, 2] == 0).all() and w_out[1, 2] == w[1, 2]
    qb = _bf16_bits(q)
    np.testing.assert_array_equal(oracle.quantize_query_f32(_bf16_value(qb), w)[0], oracle.quantize_query(qb, w)[0])


# ---------------------------------------------------------------- physical KV rows
def test_phys_rows_identity_table_and_permutation():
    """With the identity block table of one sequence the physical row of token
    t is t itself; with a permuted table it is perm[t // 64] * 64 + t % 64
    (checked against a Python loop over the same table), -1 stays -1, and
    rows of the same sequence (draft rows) share the sequence's table row."""
    ident = synth.make_case("pi", seq_lens=[3000], seed=1, permute_blocks=False)
    idx = np.array([[0, 1, 63, 64, 2999, -1]], dtype=np.int32)
    np.testing.assert_array_equal(oracle.phys_rows(ident, idx), idx)
    case = synth.make_case("pp", seq_lens=[700, 1300], nq=2, seed=4)
    rng = np.random.default_rng(2)
    idx = np.full((4, 50), -1, dtype=np.int32)
    for r, L in enumerate(case.row_lens()):
        idx[r, :40] = np.sort(rng.choice(int(L), 40, replace=False))
    got = oracle.phys_rows(case, idx)
    for r in range(4):
        for p in range(50):
            t = int(idx[r, p])
            want = -1 if t < 0 else int(case.block_table[r // 2, t // 64]) * 64 + t % 64
            assert got[r, p] == want
    case.block_table[1, 0] = case.num_blocks   # outside the pool
    idx2 = np.zeros((4, 1), dtype=np.int32)
    with pytest.raises(RuntimeError):
        oracle.phys_rows(case, idx2)


# --------------------------------------------------------------- native FP4 scoring
def _mx_values(packed, e8):
    """Exact values of MX-coded rows (codes [n, 64] packed, E8M0 [n, 4]) as Fractions."""
    out = []
    for p, e in zip(packed, e8):
        row = []
        for d in range(128):
            nib = p[d // 2] & 0xF if d % 2 == 0 else p[d // 2] >> 4
            mag = [0, 1, 2, 3, 4, 6, 8, 12][nib & 7] * (-1 if nib & 8 else 1)  # 2 x E2M1
            row.append(Fraction(mag, 2) * Fraction(2) ** (int(e[d // 32]) - 127))
        out.append(row)
    return out


def test_index_scores_native_fp4_exact_rational():
    """MXFP4 keys against an MXFP4 query (the native FP4 x FP4 product): with
    w = e_h the score is max(0, q_h . k_t), both sides decoded exactly from
    their E2M1 codes and E8M0 block scales."""
    c = synth.make_case("mxn", seq_lens=[130], key_format=synth.KEY_MXFP4_NATIVE, seed=4)
    rows = c.rows
    assert c.q_index.size == rows * 32 * 68
    qp = c.q_index[:rows * 32 * 64].reshape(rows * 32, 64)
    qe = c.q_index[rows * 32 * 64:].reshape(rows * 32, 4)
    for h in (0, 9, 31):
        c.head_w = np.zeros_like(c.head_w)
        c.head_w[:, h] = 1.0
        s = oracle.index_scores(c)
        bnd = oracle.index_score_bounds(c)
        qv = _mx_values(qp[h:h + 1], qe[h:h + 1])[0]
        for t in (0, 5, 64, 129):
            r = c.block_table[0, t // 64]
            page = c.pool[r, c.index_off:]
            kv = _mx_values([page[(t % 64) * 64:(t % 64) * 64 + 64]], [page[64 * 64 + (t % 64) * 4:64 * 64 + (t % 64) * 4 + 4]])[0]
            dot = sum(a * b for a, b in zip(qv, kv))
            assert s[0, t] == float(max(Fraction(0), dot))
            assert bnd[0, t] == pytest.approx(float(sum(abs(a * b) for a, b in zip(qv, kv))), rel=1e-14)


def test_index_scores_native_fp4_equals_fp8_query_when_the_query_is_exact():
    """When every query value is representable in both formats (E2M1 values
    times a power of two per block that E4M3 also holds exactly), the native
    and the FP8-query scores of the same keys are equal."""
    c8 = synth.make_case("mxe", seq_lens=[200, 70], key_format=synth.KEY_MXFP4, seed=9)
    rng = np.random.default_rng(2)
    rows = c8.rows
    vals = rng.choice([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], size=(rows, 32, 128)) * rng.choice([-1, 1], size=(rows, 32, 128))
    vals = vals * (2.0 ** rng.integers(-3, 3, size=(rows, 32, 4))).repeat(32, axis=2)
    c8.q_index = synth.e4m3_encode(vals.astype(np.float32))
    cn = synth.make_case("mxe", seq_lens=[200, 70], key_format=synth.KEY_MXFP4_NATIVE, seed=9)
    cn.q_index = synth.mxfp4_query_encode(vals.astype(np.float32))
    cn.head_w = c8.head_w
    np.testing.assert_array_equal(oracle.index_scores(cn), oracle.index_scores(c8))


def test_quantize_query_mxfp4_is_the_mx_encoding_per_head():
    """Per (row, head) and 32-dim block: E = floor(log2 amax) - 2 (clamped to
    [-127, 127]; byte 0 for an all-zero block), codes the nearest E2M1 of
    x 2^-E with ties to even (brute force), head weights unchanged."""
    rng = np.random.default_rng(13)
    q = rng.standard_normal((2, 32, 128)).astype(np.float32) * np.exp(rng.uniform(-4, 4, (2, 32, 1))).astype(np.float32)
    q[0, 3] = 0.0                      # an all-zero head
    q[1, 7, 32:64] *= np.float32(1e-38)  # a block of tiny values
    q[1, 8, :32] = 6.0 * 2.0 ** 5      # amax exactly 6 x 2^E: the top code
    q[1, 9, 64:96] = np.float32(2.0 ** 120)   # E clamps at 127
    w = rng.standard_normal((2, 32)).astype(np.float32)
    buf, w_out = oracle.quantize_query_mxfp4(q, w)
    np.testing.assert_array_equal(w_out, w)
    rows = 2
    packed = buf[:rows * 32 * 64].reshape(rows, 32, 64)
    e8 = buf[rows * 32 * 64:].reshape(rows, 32, 4)
    for r in range(rows):
        for h in range(32):
            for blk in range(4):
                xs = q[r, h, 32 * blk:32 * blk + 32].astype(np.float64)
                amax = np.abs(xs).max()
                e = -127 if amax == 0 else max(-127, min(127, math.frexp(amax)[1] - 1 - 2))
                assert e8[r, h, blk] == e + 127, (r, h, blk)
                p = packed[r, h, 16 * blk:16 * blk + 16]
                codes = np.stack([p & 0xF, p >> 4], axis=1).reshape(-1)
                assert [int(c) for c in codes] == [_e2m1_brute(float(v) * 2.0 ** -e) for v in xs], (r, h, blk)
    assert e8[0, 3].tolist() == [0, 0, 0, 0] and not packed[0, 3].any()
    assert (packed[1, 8, :16] == 0x77).all()          # +6 in both nibbles
    # the query generator's native layout is this encoding of its draws
    np.testing.assert_array_equal(synth.mxfp4_query_encode(q), buf)
