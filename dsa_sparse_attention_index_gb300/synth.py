"""Seeded synthetic workloads for the DSA decode path.

This module only *generates inputs*: random draws, their rounding into the
storage formats (E4M3 bytes, bf16 bits, MXFP4 codes) and their placement in
the packed paged cache.  It contains none of the method's arithmetic (no
scoring, selection or attention), and it is the only code that the CUDA path
and the fp64 oracle both consume.  Every array is produced on the host from
one ``numpy.random.Generator(PCG64(seed))`` in a fixed draw order.

Cache layout (per block row; the descriptor values below are passed to both
the library and the oracle, which each read the bytes on their own):

    FP8 index keys   [latent page 64 x 576 B][codes 64 x 128 B][scales 64 x fp32]
                     row = 36,864 + 8,448 = 45,312 B
    MXFP4 index keys [latent page 64 x 576 B][codes 64 x 64 B][E8M0 64 x 4 B]
                     row = 36,864 + 4,352 = 41,216 B

Both row sizes and both page offsets are multiples of 128 B.  The packed
block row (one contiguous row per cache block holding a layer's latent page
and index-key page) follows the Kimi K3.1 Pro Day-0 post, section on the KV
cache that serves three kinds of state; the split of the 132-byte FP8 key
into a 128-byte code row and a separate fp32 scale keeps every code row
16-byte aligned.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

BLOCK = 64
IDX_HEADS, IDX_DIM = 32, 128
MLA_HEADS, LATENT, VALUE = 96, 576, 512
KEY_FP8, KEY_MXFP4, KEY_MXFP4_NATIVE = 0, 1, 2   # native: MXFP4 keys and an MXFP4 query
LATENT_FP8, LATENT_NVFP4 = 0, 1

LATENT_RECORD = {LATENT_FP8: LATENT,              # 576 B: E4M3 codes
                 LATENT_NVFP4: VALUE // 2 + VALUE // 16 + (LATENT - VALUE)}  # 352 B: E2M1 + E4M3 scales + E4M3 tail
LATENT_PAGE = BLOCK * LATENT                      # 36,864 B (FP8 latents)
INDEX_PAGE = {KEY_FP8: BLOCK * (IDX_DIM + 4),     # 8,448 B
              KEY_MXFP4: BLOCK * (IDX_DIM // 2 + 4),  # 4,352 B
              KEY_MXFP4_NATIVE: BLOCK * (IDX_DIM // 2 + 4)}

_E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
_E2M1_MID = (_E2M1_GRID[1:] + _E2M1_GRID[:-1]) / 2   # 0.25 0.75 1.25 1.75 2.5 3.5 5


@dataclasses.dataclass
class Case:
    """One synthetic decode workload, laid out exactly as the cache expects."""

    name: str
    batch: int
    nq: int                     # query rows per sequence (speculative draft size)
    seq_lens: np.ndarray        # int32 [batch], context incl. the current token(s)
    key_format: int             # KEY_FP8, KEY_MXFP4 or KEY_MXFP4_NATIVE
    topk: int
    pool: np.ndarray            # uint8 [num_blocks, row_stride]
    row_stride: int
    latent_off: int
    index_off: int
    latent_scale: float
    block_table: np.ndarray     # int32 [batch, max_blocks]; -1 = unallocated
    q_index: np.ndarray         # uint8: E4M3 codes [rows, 32, 128]; native FP4: codes [rows, 32, 64] then E8M0 [rows, 32, 4], flat
    head_w: np.ndarray          # float32 [rows, 32]
    q_mla: np.ndarray           # uint16 (bf16 bits) [rows, 96, 576]
    sm_scale: float
    seed: int = 0
    latent_format: int = LATENT_FP8  # LATENT_FP8 or LATENT_NVFP4

    @property
    def rows(self) -> int:
        return self.batch * self.nq

    @property
    def num_blocks(self) -> int:
        return int(self.pool.shape[0])

    @property
    def max_len(self) -> int:
        return int(self.seq_lens.max()) if self.batch else 0

    def row_lens(self) -> np.ndarray:
        """Tokens visible to each query row: row j of a sequence with context L
        and nq draft rows sees L - (nq - 1) + j tokens (causal within the draft)."""
        L = np.repeat(self.seq_lens.astype(np.int64), self.nq)
        j = np.tile(np.arange(self.nq, dtype=np.int64), self.batch)
        return np.maximum(L - (self.nq - 1) + j, 0).astype(np.int32)

    def token_bytes(self) -> int:
        return 132 if self.key_format == KEY_FP8 else 68

    def latent_bytes(self) -> int:
        return LATENT_RECORD[self.latent_format]


# ---------------------------------------------------------------------------
# storage-format encoders (input rounding only)
# ---------------------------------------------------------------------------

def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """Round to OCP E4M3 ('fn') codes, nearest-even, saturating at +-448."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).clamp(-448.0, 448.0)
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def bf16_encode(x: np.ndarray) -> np.ndarray:
    """Round to bfloat16 (nearest-even); returns the raw 16-bit patterns."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def mxfp4_encode(x: np.ndarray):
    """OCP MX quantisation of rows of 128 values into E2M1 elements with one
    E8M0 scale per 32 elements.  Shared exponent floor(log2(amax)) - 2 (2 is
    E2M1's largest exponent), elements rounded to nearest-even and clamped
    to +-6.  Returns (packed codes uint8 [n, 64], e8m0 uint8 [n, 4]); element
    2i sits in the low nibble of byte i."""
    import torch

    x = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float64)).reshape(-1, IDX_DIM // 32, 32)
    amax = x.abs().amax(dim=2)
    _, ex = torch.frexp(amax)                    # amax = m * 2^ex, m in [0.5, 1): floor(log2 amax) = ex - 1
    e = torch.where(amax > 0, ex.to(torch.int64) - 1 - 2, torch.full_like(ex, -127, dtype=torch.int64))
    e = e.clamp(-127, 127)
    scaled = torch.ldexp(x, (-e).unsqueeze(-1).to(torch.float64))   # exact: a power-of-two scaling
    code = e2m1_codes(scaled).to(torch.uint8).reshape(-1, IDX_DIM).numpy()
    packed = (code[:, 0::2] | (code[:, 1::2] << 4)).astype(np.uint8)
    e = e.numpy()
    e8m0 = (e + 127).astype(np.uint8).reshape(-1, IDX_DIM // 32)
    return packed, e8m0


def mxfp4_query_encode(q: np.ndarray) -> np.ndarray:
    """An indexer query [rows, 32, 128] in the native-FP4 layout: each head's
    128 values quantised as one MXFP4 key (mxfp4_encode); the buffer holds the
    packed codes [rows, 32, 64] followed by the E8M0 scales [rows, 32, 4]."""
    rows = q.shape[0]
    packed, e8 = mxfp4_encode(np.asarray(q).reshape(rows * IDX_HEADS, IDX_DIM))
    return np.concatenate([packed.reshape(-1), e8.reshape(-1)]).astype(np.uint8)


def e2m1_codes(mag_signed: "torch.Tensor") -> "torch.Tensor":
    """Nearest E2M1 codes (ties to even, |x| >= 6 -> 6) of a float64 tensor,
    as int64 nibbles with the sign in bit 3."""
    import torch

    mag = mag_signed.abs()
    # count the midpoints below |x|; at an exact midpoint this picks the lower
    # code, so the three midpoints whose upper code is the even one move up
    # (round half to even); |x| >= 6 lands on code 7 (6.0)
    code = torch.bucketize(mag, torch.from_numpy(_E2M1_MID), right=False)
    code = code + ((mag == 0.75) | (mag == 1.75) | (mag == 3.5)).to(code.dtype)
    return code | torch.where(mag_signed < 0, 8, 0)


def nvfp4_latent_encode(x: np.ndarray, latent_scale: float) -> np.ndarray:
    """NVFP4 latent records [n, 352] of [n, 576] values: per 16 dims of
    0..511 a block scale e4m3(amax / (6 latent_scale)) and E2M1 codes of
    x / (latent_scale * scale) (element 2i in the low nibble of byte i); dims
    512..575 as e4m3(x / latent_scale)."""
    import torch

    x = np.ascontiguousarray(x, dtype=np.float32)
    n = x.shape[0]
    ls = np.float32(latent_scale)
    head = x[:, :VALUE].reshape(n, VALUE // 16, 16)
    amax = np.abs(head).max(axis=2)
    sc = e4m3_encode(amax / (np.float32(6.0) * ls))                       # [n, 32] codes
    sdec = torch.from_numpy(sc.copy()).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    step = (ls * sdec).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(sdec[..., None] > 0, head / step[..., None], np.float32(0.0)).astype(np.float32)
    codes = e2m1_codes(torch.from_numpy(q.astype(np.float64))).to(torch.uint8).numpy().reshape(n, VALUE)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    tail = e4m3_encode(x[:, VALUE:] / ls)
    return np.concatenate([packed, sc, tail], axis=1)


# ---------------------------------------------------------------------------
# workload construction
# ---------------------------------------------------------------------------

def make_case(name: str, seq_lens, nq: int = 1, key_format: int = KEY_FP8, topk: int = 2048,
              heavy_tail: float = 0.0, permute_blocks: bool = True, spare_blocks: int = 0,
              seed: int = 0, chunk_tokens: int = 1 << 16, latent_format: int = LATENT_FP8) -> Case:
    """Build a workload.  Draw order: block permutation, latent scale, then
    per sequence and per token chunk: index-key values, heavy-tail mask,
    per-token key scales (FP8 only), latent values; then tail/spare filler
    bytes; then indexer queries, head weights, MLA queries.

    Distributions: index keys and latents E4M3(N(0,1)); key scales U(0.5, 2);
    latent scale U(0.5, 2); indexer queries E4M3(N(0,1)) [32, 128]; head
    weights N(0, 0.1^2) fp32; MLA queries bf16(N(0,1)) [96, 576].  With
    ``heavy_tail`` = f, a fraction f of tokens have their key values x4 before
    rounding.  MXFP4 keys quantise the same N(0,1) draws per OCP MX (and, for
    KEY_MXFP4_NATIVE, the query draws likewise, per head); NVFP4
    latents quantise the same latent draws as ``nvfp4_latent_encode``.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    seq_lens = np.asarray(seq_lens, dtype=np.int32).reshape(-1)
    batch = int(seq_lens.shape[0])
    nblk = [max(1, math.ceil(int(L) / BLOCK)) for L in seq_lens]
    max_blocks = max(nblk) if nblk else 1
    used = sum(nblk)
    num_blocks = used + int(spare_blocks)
    perm = rng.permutation(num_blocks).astype(np.int32)   # drawn in every case: fixed draw order
    if not permute_blocks:
        perm = np.arange(num_blocks, dtype=np.int32)
    latent_scale = float(rng.uniform(0.5, 2.0))

    idx_page = INDEX_PAGE[key_format]
    rec = LATENT_RECORD[latent_format]
    lat_page = BLOCK * rec
    row_stride = lat_page + idx_page
    latent_off, index_off = 0, lat_page
    pool = np.zeros((num_blocks, row_stride), dtype=np.uint8)
    block_table = np.full((batch, max_blocks), -1, dtype=np.int32)

    cursor = 0
    for b in range(batch):
        rows_b = perm[cursor:cursor + nblk[b]]
        cursor += nblk[b]
        block_table[b, :nblk[b]] = rows_b
        L = int(seq_lens[b])
        for t0 in range(0, L, chunk_tokens):
            n = min(chunk_tokens, L - t0)
            kv = rng.standard_normal((n, IDX_DIM), dtype=np.float32)
            if heavy_tail > 0:
                kv *= np.where(rng.random(n) < heavy_tail, 4.0, 1.0).astype(np.float32)[:, None]
            if key_format == KEY_FP8:
                codes = e4m3_encode(kv)
                scales = rng.uniform(0.5, 2.0, size=n).astype(np.float32)
            else:
                codes, e8 = mxfp4_encode(kv)
            lat_x = rng.standard_normal((n, LATENT), dtype=np.float32)
            lat = e4m3_encode(lat_x) if latent_format == LATENT_FP8 else nvfp4_latent_encode(lat_x, latent_scale)
            t = np.arange(t0, t0 + n)
            r = rows_b[t // BLOCK]
            slot = t % BLOCK
            # scatter token rows into their pages
            lat_view = pool[:, latent_off:latent_off + lat_page].reshape(num_blocks, BLOCK, rec)
            lat_view[r, slot] = lat
            if key_format == KEY_FP8:
                cview = pool[:, index_off:index_off + BLOCK * IDX_DIM].reshape(num_blocks, BLOCK, IDX_DIM)
                cview[r, slot] = codes
                sview = pool[:, index_off + BLOCK * IDX_DIM:index_off + idx_page].reshape(num_blocks, BLOCK, 4)
                sview[r, slot] = scales.view(np.uint8).reshape(n, 4)
            else:
                cb = IDX_DIM // 2
                cview = pool[:, index_off:index_off + BLOCK * cb].reshape(num_blocks, BLOCK, cb)
                cview[r, slot] = codes
                eview = pool[:, index_off + BLOCK * cb:index_off + idx_page].reshape(num_blocks, BLOCK, 4)
                eview[r, slot] = e8
    # filler: unused tail slots of each last page, and spare rows, get random bytes
    for b in range(batch):
        L = int(seq_lens[b])
        tail = L % BLOCK if L > 0 else 0
        if tail or L == 0:
            r = block_table[b, nblk[b] - 1]
            s0 = tail
            fill = rng.integers(0, 256, size=(BLOCK - s0, rec), dtype=np.uint8)
            pool[r, latent_off:latent_off + lat_page].reshape(BLOCK, rec)[s0:] = fill
            per_tok = idx_page // BLOCK
            code_b = per_tok - 4
            codes_view = pool[r, index_off:index_off + BLOCK * code_b].reshape(BLOCK, code_b)
            codes_view[s0:] = rng.integers(0, 256, size=(BLOCK - s0, code_b), dtype=np.uint8)
            sc_view = pool[r, index_off + BLOCK * code_b:index_off + idx_page].reshape(BLOCK, 4)
            sc_view[s0:] = rng.integers(0, 256, size=(BLOCK - s0, 4), dtype=np.uint8)
    if spare_blocks:
        spare = perm[used:]
        pool[spare] = rng.integers(0, 256, size=(len(spare), row_stride), dtype=np.uint8)

    rows = batch * nq
    q_draw = rng.standard_normal((rows, IDX_HEADS, IDX_DIM), dtype=np.float32)
    q_index = e4m3_encode(q_draw) if key_format != KEY_MXFP4_NATIVE else mxfp4_query_encode(q_draw)
    head_w = (rng.standard_normal((rows, IDX_HEADS)) * 0.1).astype(np.float32)
    q_mla = bf16_encode(rng.standard_normal((rows, MLA_HEADS, LATENT), dtype=np.float32))
    return Case(name=name, batch=batch, nq=nq, seq_lens=seq_lens, key_format=key_format, topk=topk,
                pool=pool, row_stride=row_stride, latent_off=latent_off, index_off=index_off,
                latent_scale=latent_scale, block_table=block_table, q_index=q_index, head_w=head_w,
                q_mla=q_mla, sm_scale=1.0 / math.sqrt(LATENT), seed=seed, latent_format=latent_format)


# ---------------------------------------------------------------------------
# the named workloads
# ---------------------------------------------------------------------------

WORKLOADS = {
    # tiny single decode: batch 1, one query, L = 4096, identity block table
    "decode_b1_l4096": dict(seq_lens=[4096], nq=1, permute_blocks=False),
    # speculative verify: 8 sequences x 4 causal draft rows, L = 32,768 each
    "specdecode_b8x4_l32768": dict(seq_lens=[32768] * 8, nq=4),
    # long-context batch: 32 sequences, L ~ U(64K, 160K), 10% of keys x4
    "longctx_b32_l64k-160k": dict(seq_lens=None, nq=1, heavy_tail=0.10),
    # 1M-token decode with MXFP4 index keys: batch 4
    "mxfp4_b4_l1m": dict(seq_lens=[1 << 20] * 4, nq=1, key_format=KEY_MXFP4),
    # the same with the query in MXFP4 too, scored by the native FP4 x FP4 MMA
    "mxfp4n_b4_l1m": dict(seq_lens=[1 << 20] * 4, nq=1, key_format=KEY_MXFP4_NATIVE),
    # the long-context batch in the 10,080 B/token configuration: NVFP4
    # latents (352 B) and MXFP4 keys (68 B), 420 B a token and layer
    "longctx_b32_l64k-160k_nvfp4": dict(seq_lens=None, nq=1, heavy_tail=0.10, key_format=KEY_MXFP4,
                                        latent_format=LATENT_NVFP4),
    # smaller cases of the same shapes for profiler captures (inputs still larger than L2)
    "longctx_b32_l64k": dict(seq_lens=[65536] * 32, nq=1, heavy_tail=0.1),
    "mxfp4_b8_l256k": dict(seq_lens=[1 << 18] * 8, nq=1, key_format=KEY_MXFP4),
    "mxfp4n_b8_l256k": dict(seq_lens=[1 << 18] * 8, nq=1, key_format=KEY_MXFP4_NATIVE),
    "longctx_b32_l64k_nvfp4": dict(seq_lens=[65536] * 32, nq=1, heavy_tail=0.1, key_format=KEY_MXFP4,
                                   latent_format=LATENT_NVFP4),
    # chunked-prefill append: 2048 new query rows on a 151,552-token prefix
    "prefill_q2048_l153600": dict(seq_lens=[153600], nq=2048),
    # a smaller chunk of the same context for profiler captures (scores still larger than L2)
    "prefill_q256_l153600": dict(seq_lens=[153600], nq=256),
}


def longctx_lengths(seed: int = 0, batch: int = 32, lo: int = 65536, hi: int = 163840) -> np.ndarray:
    """Context lengths of the long-context batch: integers U[lo, hi], drawn
    from their own seeded generator so the workload is reproducible."""
    rng = np.random.Generator(np.random.PCG64(seed + 1000))
    return rng.integers(lo, hi + 1, size=batch).astype(np.int32)


def workload(name: str, seed: int = 0, **overrides) -> Case:
    spec = dict(WORKLOADS[name])
    spec.update(overrides)
    if spec.get("seq_lens") is None:
        spec["seq_lens"] = longctx_lengths(seed)
    return make_case(name, seed=seed, **spec)


# ---------------------------------------------------------------------------
# device copies (marshalling only)
# ---------------------------------------------------------------------------

@dataclasses.dataclass
class DeviceCase:
    cache: object        # binding.PagedCache
    batch: object        # binding.Batch
    q_index: object      # uint8, the case's query layout
    head_w: object       # float32 [rows, 32]
    q_mla: object        # int16 (bf16 bits) [rows, 96, 576]
    row_lens: object     # int32 [rows]


def device_case(case: Case, device="cuda") -> DeviceCase:
    """Copy a workload's arrays to the GPU in the layouts libdsa expects."""
    import torch

    from . import binding

    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)
    cache = binding.PagedCache(pool=t(case.pool), row_stride=case.row_stride, latent_off=case.latent_off,
                               index_off=case.index_off, key_format=case.key_format,
                               latent_scale=case.latent_scale, latent_format=case.latent_format)
    batch = binding.Batch(block_table=t(case.block_table), seq_lens=t(case.seq_lens.astype(np.int32)),
                          queries_per_seq=case.nq, max_seq_len=max(case.max_len, 0))
    return DeviceCase(cache=cache, batch=batch, q_index=t(case.q_index), head_w=t(case.head_w),
                      q_mla=t(case.q_mla.view(np.int16)), row_lens=t(case.row_lens()))


# ---------------------------------------------------------------------------
# the fused indexer front end's inputs
# ---------------------------------------------------------------------------

# Width of the compressed query that the indexer front end normalises and
# projects.  The pages do not give it; 1,536 is the compressed-query width of
# the DeepSeek-style MLA that DSA comes from.
QUERY_RANK = 1536
NORM_EPS = 1e-6
INDEX_Q_OUT = IDX_HEADS * IDX_DIM   # 4,096 projected query values per row


@dataclasses.dataclass
class FrontendInputs:
    """One step's inputs to the fused indexer front end, for `rows` query rows:
    what the packed input projection hands it (the compressed query, the raw
    head weights, the new token's index key and latent) and the layer's norm
    and projection weights.  bf16 tensors are stored as their 16-bit patterns."""

    c_q: np.ndarray         # uint16 [rows, D]      compressed query
    gamma: np.ndarray       # uint16 [D]            RMSNorm weight
    w_iq: np.ndarray        # uint16 [4096, D]      indexer query projection (row o = head * 128 + dim)
    head_w: np.ndarray      # float32 [rows, 32]    head weights before the query scale is folded in
    new_latent: np.ndarray  # uint16 [rows, 576]    the new token's latent
    new_key: np.ndarray     # uint16 [rows, 128]    the new token's index key
    eps: float = NORM_EPS


def make_frontend(rows: int, dim: int = QUERY_RANK, seed: int = 0) -> FrontendInputs:
    """Seeded front-end inputs.  Draw order: compressed queries N(0, 1), the
    norm weight U(0.5, 1.5), the projection N(0, 1/D) (unit-variance outputs),
    head weights N(0, 0.1), new latents N(0, 1), new index keys N(0, 1)."""
    rng = np.random.Generator(np.random.PCG64(seed + 2000))
    c_q = bf16_encode(rng.standard_normal((rows, dim)).astype(np.float32))
    gamma = bf16_encode(rng.uniform(0.5, 1.5, dim).astype(np.float32))
    w_iq = bf16_encode((rng.standard_normal((INDEX_Q_OUT, dim)) / math.sqrt(dim)).astype(np.float32))
    head_w = (rng.standard_normal((rows, IDX_HEADS)) * 0.1).astype(np.float32)
    new_latent = bf16_encode(rng.standard_normal((rows, LATENT)).astype(np.float32))
    new_key = bf16_encode(rng.standard_normal((rows, IDX_DIM)).astype(np.float32))
    return FrontendInputs(c_q=c_q, gamma=gamma, w_iq=w_iq, head_w=head_w, new_latent=new_latent, new_key=new_key)
