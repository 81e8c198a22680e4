"""fp64 CPU oracle for the DSA decode hot path — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The product path (``dsa_sparse_attention_index_gb300``
and its CUDA library) never does, and shares no code with it.

The arithmetic lives in ``dsa_oracle.c`` (plain C, double precision); this
module only compiles it with ``gcc`` and marshals numpy arrays through ctypes.
Each function's docstring names the passage of the source pages it follows;
the C file's header lists the pages and the readings taken where they are
silent.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dsa_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

IDX_HEADS, IDX_DIM = 32, 128
MLA_HEADS, LATENT, VALUE = 96, 576, 512


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/liboracle.so`` (gcc, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
        )
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
            lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_to_double.restype = f64
            lib.oracle_e2m1_to_double.argtypes = [ctypes.c_uint8]
            lib.oracle_e2m1_to_double.restype = f64
            lib.oracle_e8m0_to_double.argtypes = [ctypes.c_uint8]
            lib.oracle_e8m0_to_double.restype = f64
            lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_double.restype = f64
            lib.oracle_index_scores.argtypes = [P, i64, i64, i32, i32, P, i32, P, i32, i32, P, P, P, i64]
            lib.oracle_index_scores.restype = i32
            lib.oracle_index_score_bounds.argtypes = [P, i64, i64, i32, i32, P, i32, P, i32, i32, P, P, P, i64]
            lib.oracle_index_score_bounds.restype = i32
            lib.oracle_topk.argtypes = [P, i64, P, i32, i32, P]
            lib.oracle_topk.restype = i32
            lib.oracle_dcp_topk.argtypes = [P, i64, P, i32, i32, i32, P, P]
            lib.oracle_dcp_topk.restype = i32
            lib.oracle_sparse_mla.argtypes = [P, i64, i64, i32, f64, P, i32, P, i32, i32, P, P, i32, f64, P, P, i32]
            lib.oracle_sparse_mla.restype = i32
            lib.oracle_num_threads.argtypes = []
            lib.oracle_num_threads.restype = i32
            lib.oracle_e4m3_encode.argtypes = [f64]
            lib.oracle_e4m3_encode.restype = ctypes.c_uint8
            lib.oracle_e2m1_encode.argtypes = [f64]
            lib.oracle_e2m1_encode.restype = ctypes.c_uint8
            lib.oracle_cache_append.argtypes = [P, i64, i64, i64, i32, i32, ctypes.c_float, P, i32, P, i32, i32, P, P,
                                                i32]
            lib.oracle_cache_append.restype = i32
            lib.oracle_quantize_query.argtypes = [P, P, i32, P, P]
            lib.oracle_quantize_query.restype = i32
            lib.oracle_rms_norm_bf16.argtypes = [P, P, i32, i32, f64, P]
            lib.oracle_rms_norm_bf16.restype = i32
            lib.oracle_index_query_proj.argtypes = [P, P, i32, i32, i32, P]
            lib.oracle_index_query_proj.restype = i32
            lib.oracle_quantize_query_f32.argtypes = [P, P, i32, P, P]
            lib.oracle_quantize_query_f32.restype = i32
            lib.oracle_quantize_query_mxfp4.argtypes = [P, P, i32, P, P]
            lib.oracle_quantize_query_mxfp4.restype = i32
            lib.oracle_phys_rows.argtypes = [P, i32, i32, i32, P, i32, i32, P]
            lib.oracle_phys_rows.restype = i32
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


class OracleError(RuntimeError):
    pass


def _check(rc: int, what: str) -> None:
    if rc == 1:
        raise OracleError(f"{what}: invalid argument")
    if rc == 3:
        raise OracleError(f"{what}: block-table entry or token index outside the cache")
    if rc != 0:
        raise OracleError(f"{what}: error {rc}")


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def e4m3_to_double(code: int) -> float:
    """OCP E4M3 ('fn') decode from the format definition."""
    return float(_load().oracle_e4m3_to_double(code))


def e2m1_to_double(code: int) -> float:
    """OCP MX E2M1 decode from the format definition."""
    return float(_load().oracle_e2m1_to_double(code))


def e8m0_to_double(code: int) -> float:
    """OCP MX E8M0 scale decode: 2^(E-127)."""
    return float(_load().oracle_e8m0_to_double(code))


def bf16_to_double(bits: int) -> float:
    return float(_load().oracle_bf16_to_double(bits))


def _cache_args(case):
    return (
        _ptr(case.pool), int(case.row_stride), int(case.index_off), int(case.num_blocks),
        int(case.key_format), _ptr(case.block_table), int(case.block_table.shape[1]),
        _ptr(case.seq_lens), int(case.batch), int(case.nq),
    )


def index_scores(case, rows_ld: int | None = None) -> np.ndarray:
    """Lightning-indexer scores s[row, t] in fp64 for every visible token.

    Follows the Kimi K3.1 Pro Day-0 post, section on sparse attention (32
    light heads score every prior token with a 132-byte FP8 key) and its AMD
    MXFP4-indexer section (68-byte keys, FP32 accumulation, weighted head
    reduction; key_format 2: the MXFP4 keys against a native-FP4 query, whose
    buffer is codes [rows, 32, 64] then E8M0 scales [rows, 32, 4]).  Entries
    beyond a row's visible length are NaN.
    """
    ld = int(rows_ld or case.max_len)
    out = np.full((case.rows, ld), np.nan, dtype=np.float64)
    q = np.ascontiguousarray(case.q_index)
    w = np.ascontiguousarray(case.head_w)
    rc = _load().oracle_index_scores(*_cache_args(case), _ptr(q), _ptr(w), _ptr(out), ld)
    _check(rc, "index_scores")
    return out


def index_score_bounds(case, rows_ld: int | None = None) -> np.ndarray:
    """A_t = sum_h |w_h| |scale_t| sum_d |q_hd k_td| — the magnitude that any
    evaluation order's rounding error of the score is proportional to."""
    ld = int(rows_ld or case.max_len)
    out = np.full((case.rows, ld), np.nan, dtype=np.float64)
    rc = _load().oracle_index_score_bounds(
        *_cache_args(case), _ptr(np.ascontiguousarray(case.q_index)),
        _ptr(np.ascontiguousarray(case.head_w)), _ptr(out), ld)
    _check(rc, "index_score_bounds")
    return out


def topk(scores: np.ndarray, row_lens: np.ndarray, k: int) -> np.ndarray:
    """Top-k token indices per row: ties to the lower index, ascending output,
    -1 padding (the Day-0 post keeps the top 2,048 tokens per query)."""
    s = np.ascontiguousarray(scores, dtype=np.float64)
    lens = np.ascontiguousarray(row_lens, dtype=np.int32)
    rows = s.shape[0]
    out = np.empty((rows, k), dtype=np.int32)
    rc = _load().oracle_topk(_ptr(s), s.shape[1], _ptr(lens), rows, int(k), _ptr(out))
    _check(rc, "topk")
    return out


def dcp_topk(scores: np.ndarray, row_lens: np.ndarray, k: int, shards: int):
    """Top-k through the decode-context-parallel merge of W = `shards` shards
    (Day-0 post, decode-context-parallelism section): per shard the best
    ceil(1.5 k / W) bf16-keyed candidates as 32-bit words, a global selection,
    and a full local top-k resent by any shard that may hold more of it.
    Returns (indices [rows, k] ascending with -1 padding, stats [rows, 3]:
    words sent in the first round, shards that resent, words resent)."""
    s = np.ascontiguousarray(scores, dtype=np.float32)
    lens = np.ascontiguousarray(row_lens, dtype=np.int32)
    rows = s.shape[0]
    out = np.empty((rows, k), dtype=np.int32)
    stats = np.empty((rows, 3), dtype=np.int64)
    rc = _load().oracle_dcp_topk(_ptr(s), s.shape[1], _ptr(lens), rows, int(k), int(shards), _ptr(out), _ptr(stats))
    _check(rc, "dcp_topk")
    return out, stats


def sparse_mla(case, idx: np.ndarray, k: int | None = None):
    """Exact absorbed-MLA attention of 96 heads over the selected latents
    (Day-0 post, sparse-attention section: MLA runs exactly on the kept
    tokens).  Returns (out [rows, 96, 512] fp64, lse [rows, 96] fp64)."""
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    k = int(k or idx.shape[1])
    out = np.empty((case.rows, MLA_HEADS, VALUE), dtype=np.float64)
    lse = np.empty((case.rows, MLA_HEADS), dtype=np.float64)
    q = np.ascontiguousarray(case.q_mla, dtype=np.uint16)
    rc = _load().oracle_sparse_mla(
        _ptr(case.pool), int(case.row_stride), int(case.latent_off), int(case.num_blocks),
        float(case.latent_scale), _ptr(case.block_table), int(case.block_table.shape[1]),
        _ptr(case.seq_lens), int(case.batch), int(case.nq), _ptr(q), _ptr(idx), k,
        float(case.sm_scale), _ptr(out), _ptr(lse), int(getattr(case, "latent_format", 0)))
    _check(rc, "sparse_mla")
    return out, lse


def decode_step(case):
    """The whole decode hot path: scores -> top-k -> sparse MLA, in fp64.
    Returns (scores, idx, out, lse)."""
    s = index_scores(case)
    idx = topk(s, case.row_lens(), case.topk)
    out, lse = sparse_mla(case, idx, case.topk)
    return s, idx, out, lse


def e4m3_encode(x: float) -> int:
    """OCP E4M3 ('fn') encode: nearest code, ties to even, saturating at 448."""
    return int(_load().oracle_e4m3_encode(float(x)))


def e2m1_encode(x: float) -> int:
    """OCP MX E2M1 encode: nearest code, ties to even, saturating at 6."""
    return int(_load().oracle_e2m1_encode(float(x)))


def cache_append(case, new_latent: np.ndarray, new_key: np.ndarray) -> np.ndarray:
    """The pool after writing every sequence's nq new tokens (bf16 bits
    new_latent [rows, 576], new_key [rows, 128]) into their pages, following
    the Day-0 post's fused-decode section (the step writes the new token's
    index key and latent into the packed cache).  Returns a new pool array."""
    pool = np.array(case.pool, copy=True)
    lat = np.ascontiguousarray(new_latent, dtype=np.uint16)
    key = np.ascontiguousarray(new_key, dtype=np.uint16)
    rc = _load().oracle_cache_append(
        _ptr(pool), int(case.row_stride), int(case.latent_off), int(case.index_off), int(case.num_blocks),
        int(case.key_format), float(case.latent_scale), _ptr(case.block_table), int(case.block_table.shape[1]),
        _ptr(case.seq_lens), int(case.batch), int(case.nq), _ptr(lat), _ptr(key),
        int(getattr(case, "latent_format", 0)))
    _check(rc, "cache_append")
    return pool


def quantize_query(q_bf16: np.ndarray, head_w: np.ndarray):
    """FP8 indexer query per (row, head) with its scale folded into the head
    weight (Day-0 post, fused-decode section).  Returns (codes uint8
    [rows, 32, 128], w float32 [rows, 32])."""
    q = np.ascontiguousarray(q_bf16, dtype=np.uint16)
    w = np.ascontiguousarray(head_w, dtype=np.float32)
    rows = q.shape[0]
    codes = np.empty((rows, IDX_HEADS, IDX_DIM), dtype=np.uint8)
    w_out = np.empty((rows, IDX_HEADS), dtype=np.float32)
    _check(_load().oracle_quantize_query(_ptr(q), _ptr(w), rows, _ptr(codes), _ptr(w_out)), "quantize_query")
    return codes, w_out


def rms_norm_bf16(c_bf16: np.ndarray, gamma_bf16: np.ndarray, eps: float) -> np.ndarray:
    """The front end's query norm (Day-0 post, fused-decode section: "query
    norm"; read as RMSNorm with a learned weight): xn = c / sqrt(mean(c^2) +
    eps) * gamma per row, in fp64, rounded to bf16.  Inputs and result are
    bf16 bits [rows, D]."""
    c = np.ascontiguousarray(c_bf16, dtype=np.uint16)
    g = np.ascontiguousarray(gamma_bf16, dtype=np.uint16)
    rows, dim = c.shape
    out = np.empty_like(c)
    _check(_load().oracle_rms_norm_bf16(_ptr(c), _ptr(g), rows, dim, float(eps), _ptr(out)), "rms_norm_bf16")
    return out


def index_query_proj(xn_bf16: np.ndarray, w_bf16: np.ndarray) -> np.ndarray:
    """The indexer's query projection (Day-0 post, fused-decode section):
    q[r, o] = sum_i W[o, i] xn[r, i] in fp64 over bf16 operands, o = head *
    128 + dim.  xn [rows, D], W [outs, D] bf16 bits; returns float64 [rows, outs]."""
    xn = np.ascontiguousarray(xn_bf16, dtype=np.uint16)
    w = np.ascontiguousarray(w_bf16, dtype=np.uint16)
    rows, dim = xn.shape
    outs = w.shape[0]
    assert w.shape[1] == dim
    q = np.empty((rows, outs), dtype=np.float64)
    _check(_load().oracle_index_query_proj(_ptr(xn), _ptr(w), rows, dim, outs, _ptr(q)), "index_query_proj")
    return q


def quantize_query_f32(q_f32: np.ndarray, head_w: np.ndarray):
    """quantize_query from fp32 query values [rows, 32, 128] (the front end's
    projection accumulates in fp32): codes uint8 [rows, 32, 128] and the
    head weights times the scales, float32 [rows, 32]."""
    q = np.ascontiguousarray(q_f32, dtype=np.float32).reshape(-1, IDX_HEADS, IDX_DIM)
    w = np.ascontiguousarray(head_w, dtype=np.float32)
    rows = q.shape[0]
    codes = np.empty((rows, IDX_HEADS, IDX_DIM), dtype=np.uint8)
    w_out = np.empty((rows, IDX_HEADS), dtype=np.float32)
    _check(_load().oracle_quantize_query_f32(_ptr(q), _ptr(w), rows, _ptr(codes), _ptr(w_out)), "quantize_query_f32")
    return codes, w_out


def quantize_query_mxfp4(q_f32: np.ndarray, head_w: np.ndarray):
    """The indexer query in native FP4 (Day-0 post, fused-decode section: FP8
    or MXFP4 quantisation; MXFP4-indexer section: native FP4 scoring), from
    fp32 values [rows, 32, 128]: per 32-dim block the OCP MX shared exponent
    floor(log2 amax) - 2 and E2M1 codes, as the MXFP4 keys.  Returns the query
    buffer (uint8: codes [rows, 32, 64] then E8M0 scales [rows, 32, 4], flat)
    and the head weights, unchanged (float32 [rows, 32])."""
    q = np.ascontiguousarray(q_f32, dtype=np.float32).reshape(-1, IDX_HEADS, IDX_DIM)
    w = np.ascontiguousarray(head_w, dtype=np.float32)
    rows = q.shape[0]
    out = np.empty(rows * IDX_HEADS * (IDX_DIM // 2 + 4), dtype=np.uint8)
    w_out = np.empty((rows, IDX_HEADS), dtype=np.float32)
    _check(_load().oracle_quantize_query_mxfp4(_ptr(q), _ptr(w), rows, _ptr(out), _ptr(w_out)),
           "quantize_query_mxfp4")
    return out, w_out


def phys_rows(case, idx: np.ndarray) -> np.ndarray:
    """The physical KV rows (block row * 64 + slot) of the selected tokens idx
    [rows, k] through the case's block table, -1 beside -1 (Day-0 post,
    fused-decode section: the fused indexer outputs the physical KV rows that
    attention reads).  Raises on a table entry outside the pool."""
    ix = np.ascontiguousarray(idx, dtype=np.int32)
    rows, k = ix.shape
    out = np.empty_like(ix)
    bt = np.ascontiguousarray(case.block_table, dtype=np.int32)
    _check(_load().oracle_phys_rows(_ptr(bt), int(bt.shape[1]), int(case.num_blocks), int(case.nq), _ptr(ix), rows,
                                    int(k), _ptr(out)), "phys_rows")
    return out


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round fp64 values to the nearest bf16 value, ties to even, exactly (8
    significant bits; subnormal spacing 2^-133; no overflow handling, the
    values here are far from the bf16 range's end).  Zeros, infinities and
    NaN pass through."""
    x = np.asarray(x, dtype=np.float64)
    out = x.copy()
    fin = np.isfinite(x) & (x != 0.0)
    _, e = np.frexp(x[fin])                    # |x| = m 2^e, m in [0.5, 1)
    quantum = np.ldexp(1.0, np.maximum(e - 8, -133))
    out[fin] = np.rint(x[fin] / quantum) * quantum  # exact: a power-of-two scale, then round half to even
    return out


def dcp_sparse_mla(case, idx: np.ndarray, shards: int, k: int | None = None, partial: str = "bf16"):
    """Sparse MLA under decode context parallelism (Day-0 post,
    decode-context-parallelism section): shard w of W holds the tokens t
    with t mod W = w and attends over the selected tokens it holds; the
    partial outputs are merged through their log-sum-exp:
        lse = ln sum_w exp(LSE_w),  out = sum_w exp(LSE_w - lse) O_w.
    partial = "bf16": each O_w is rounded to bf16 before the merge (the
    exchanged format; the post's combine kernels move BF16 outputs);
    "f64": no rounding, so the result is the unsharded attention.
    Returns (out [rows, 96, 512], lse [rows, 96], O [W, rows, 96, 512],
    LSE [W, rows, 96]), all fp64."""
    if partial not in ("bf16", "f64"):
        raise ValueError("partial must be 'bf16' or 'f64'")
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    W = int(shards)
    parts_o, parts_l = [], []
    for w in range(W):
        own = np.where((idx >= 0) & (idx % W == w), idx, -1).astype(np.int32)
        o, l = sparse_mla(case, own, k)
        parts_o.append(round_bf16(o) if partial == "bf16" else o)
        parts_l.append(l)
    O = np.stack(parts_o)                      # [W, rows, 96, 512]
    L = np.stack(parts_l)                      # [W, rows, 96]
    m = L.max(axis=0)                          # -inf where no shard holds a token
    safe_m = np.where(np.isfinite(m), m, 0.0)
    wexp = np.where(np.isfinite(L), np.exp(L - safe_m), 0.0)
    tot = wexp.sum(axis=0)
    lse = np.where(tot > 0, safe_m + np.log(np.where(tot > 0, tot, 1.0)), -np.inf)
    wgt = np.where(tot > 0, wexp / np.where(tot > 0, tot, 1.0), 0.0)   # exp(LSE_w - lse)
    out = (wgt[..., None] * O).sum(axis=0)
    return out, lse, O, L


def index_scores_bf16(case, rows_ld: int | None = None) -> np.ndarray:
    """Indexer scores rounded to bf16, nearest with ties to even (Day-0 post,
    decode-context-parallelism section: the top-k candidates come straight
    from BF16 scores).  The fp64 scores of index_scores, rounded."""
    return round_bf16(index_scores(case, rows_ld))
