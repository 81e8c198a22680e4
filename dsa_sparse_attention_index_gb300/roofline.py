"""Algorithmic byte and FLOP accounting for the DSA decode step.

"Algorithmic" means the bytes the method cannot avoid moving between HBM and
the chip for one layer-step, independent of how the kernels are written:

* index keys: every visible token's key once per sequence — 132 B (128 E4M3
  codes + fp32 scale) or 68 B (128 E2M1 + 4 E8M0, with an E4M3 or a native
  MXFP4 query) — all draft rows of a sequence share one read;
* latents: 576 B (E4M3) or 352 B (NVFP4) for each selected token of each
  query row (up to top-k);
* queries and head weights in, attention output (bf16 [96, 512]) and LSE
  (fp32 [96]) out.

Score tensors, top-k workspaces, split-KV partials and the block table are
implementation overheads and are not counted.  The Kimi K3.1 Pro Day-0 post
(sparse-attention section) compares 132*L + 2048*576 key+latent bytes with
dense MLA's 576*L per layer: ``pages_fraction`` reproduces that ratio.
"""
from __future__ import annotations

import numpy as np

IDX_HEADS, IDX_DIM = 32, 128
MLA_HEADS, LATENT, VALUE = 96, 576, 512
KEY_BYTES = {0: 132, 1: 68, 2: 68}
# indexer query bytes per row: E4M3 [32][128], or native FP4 codes [32][64] and E8M0 [32][4]
QUERY_BYTES = {0: IDX_HEADS * IDX_DIM, 1: IDX_HEADS * IDX_DIM, 2: IDX_HEADS * (IDX_DIM // 2 + 4)}
LATENT_BYTES = {0: 576, 1: 352}


def visible_lengths(seq_lens, nq: int) -> np.ndarray:
    L = np.repeat(np.asarray(seq_lens, dtype=np.int64), nq)
    j = np.tile(np.arange(nq, dtype=np.int64), len(seq_lens))
    return np.maximum(L - (nq - 1) + j, 0)


def step_bytes(seq_lens, nq: int = 1, topk: int = 2048, key_format: int = 0, latent_format: int = 0) -> dict:
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    vis = visible_lengths(seq_lens, nq)
    rows = len(vis)
    keys = int(KEY_BYTES[key_format] * seq_lens.sum())
    latents = int(LATENT_BYTES[latent_format] * np.minimum(vis, topk).sum())
    q_in = rows * (QUERY_BYTES[key_format] + IDX_HEADS * 4 + MLA_HEADS * LATENT * 2)
    out = rows * (MLA_HEADS * VALUE * 2 + MLA_HEADS * 4)
    return dict(keys=keys, latents=latents, queries=q_in, outputs=out,
                total=keys + latents + q_in + out, rows=rows)


def indexer_bytes(seq_lens, nq: int = 1, key_format: int = 0) -> int:
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    rows = len(seq_lens) * nq
    return int(KEY_BYTES[key_format] * seq_lens.sum() + rows * (QUERY_BYTES[key_format] + IDX_HEADS * 4))


def mla_bytes(seq_lens, nq: int = 1, topk: int = 2048, latent_format: int = 0) -> int:
    vis = visible_lengths(seq_lens, nq)
    rows = len(vis)
    return int(LATENT_BYTES[latent_format] * np.minimum(vis, topk).sum()
               + rows * (MLA_HEADS * LATENT * 2 + MLA_HEADS * VALUE * 2 + MLA_HEADS * 4))


def indexer_flops(seq_lens, nq: int = 1) -> int:
    vis = visible_lengths(seq_lens, nq)
    return int(2 * IDX_HEADS * IDX_DIM * vis.sum())


def mla_flops(seq_lens, nq: int = 1, topk: int = 2048) -> int:
    vis = visible_lengths(seq_lens, nq)
    n = np.minimum(vis, topk).sum()
    return int(2 * MLA_HEADS * n * (LATENT + VALUE))


def pages_fraction(L: int, topk: int = 2048, key_bytes: int = 132) -> float:
    """(key bytes * L + topk * 576) / (576 * L): DSA vs dense-MLA bytes per layer."""
    return (key_bytes * L + min(topk, L) * LATENT) / (LATENT * L)
