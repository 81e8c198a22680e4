"""The decode-context-parallel top-k exchange (Day-0 post,
decode-context-parallelism section) across real processes: two gloo ranks,
each holding only its token shard (t mod 2), send their best ceil(1.5 k / W)
candidates as 32-bit words (bf16 order key above the local position), gather
everyone's words, select the same global top-k, detect a shard that may hold
more of it, let that shard resend its full local top-k, and select again.
The result and the words-sent statistics equal the oracle's single-process
model of the protocol (and the library's one-GPU emulation is tested against
that model).  The LSE combine likewise: each rank's partial attention over
the selected tokens it holds, gathered as bf16 outputs and LSEs and merged,
equals the oracle's.  Runs on CPU; the rendezvous is on 127.0.0.1."""
import multiprocessing as mp
import os
import socket
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
K = 2048


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _scores(n):
    rng = np.random.default_rng(123)
    m = np.zeros((3, n), dtype=np.float32)
    m[0] = rng.standard_normal(n)
    m[1] = rng.integers(0, 25, n)              # heavy ties
    m[2] = rng.standard_normal(n)
    m[2, 0::2] += 100.0                         # shard 0 holds the whole top-k: it must resend
    return m


def _order_keys(x):
    """16-bit order keys of bf16-rounded scores (torch's rounding), NaN lowest, -0 = +0."""
    import torch

    b = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16)
    b = b.numpy().astype(np.int64) & 0xFFFF
    b = np.where(np.isnan(x), -1, b)
    b = np.where(b == 0x8000, 0, b)
    key = np.where(b < 0, 0, np.where(b & 0x8000, (~b) & 0xFFFF, b | 0x8000))
    return key.astype(np.int64)


def _select(words_by_rank, W, k):
    """Global top-k of the gathered words by (key desc, global index asc)."""
    keys, glob = [], []
    for r, w in enumerate(words_by_rank):
        w = w[w >= 0]
        keys.append(w >> 16)
        glob.append((w & 0xFFFF) * W + r)
    keys, glob = np.concatenate(keys), np.concatenate(glob)
    order = np.lexsort((glob, -keys))[:k]
    return glob[order]


def _rank(rank, world, port, n, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch
    import torch.distributed as dist

    dist.init_process_group("gloo")
    m = _scores(n)
    c = -(-3 * K // (2 * world))
    out, stats = [], []
    for row in m:
        mine = row[rank::world]                      # this shard's tokens, local position = t // W
        key = _order_keys(mine)
        order = np.lexsort((np.arange(len(mine)), -key))
        words_all = (key[order] << 16) | order         # local top order, as words
        sent = min(len(mine), c)

        def gather(count, width):
            buf = torch.full((width,), -1, dtype=torch.int64)
            buf[:count] = torch.from_numpy(words_all[:count])
            parts = [torch.empty_like(buf) for _ in range(world)]
            dist.all_gather(parts, buf)
            return [p.numpy() for p in parts]

        got = gather(sent, K)
        sel = _select(got, world, K)
        counts = [int((g >= 0).sum()) for g in got]
        taken = [int((sel % world == r).sum()) for r in range(world)]
        n_local = [len(row[r::world]) for r in range(world)]
        flags = [taken[r] == counts[r] and counts[r] < min(n_local[r], K) for r in range(world)]
        words0 = sum(counts)
        if any(flags):
            resend = min(n_local[rank], K) if flags[rank] else sent
            got = gather(resend, K)
            sel = _select(got, world, K)
        res_words = sum(min(n_local[r], K) for r in range(world) if flags[r])
        idx = np.full(K, -1, dtype=np.int64)
        idx[:len(sel)] = np.sort(sel)
        out.append(idx)
        stats.append((words0, sum(flags), res_words))
    q.put((rank, np.stack(out), np.array(stats)))
    dist.destroy_process_group()


def test_dcp_exchange_over_two_gloo_ranks_matches_the_oracle():
    sys.path.insert(0, ROOT)
    import oracle

    n = 6000
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, n, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=180) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    m = _scores(n)
    ref, ref_stats = oracle.dcp_topk(m, np.full(3, n, dtype=np.int32), K, 2)
    for _, idx, stats in res:                        # every rank ends with the same selection
        np.testing.assert_array_equal(idx, ref.astype(np.int64))
        np.testing.assert_array_equal(stats, ref_stats)
    assert ref_stats[2, 1] == 1 and ref_stats[0, 1] == 0   # the dominated row made shard 0 resend


def _rank_combine(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    import oracle
    from dsa_sparse_attention_index_gb300 import synth

    dist.init_process_group("gloo")
    case, idx = _combine_case(synth)
    # this rank's partial attention over the selected tokens it holds, sent as
    # bf16 outputs and fp64 LSEs
    own = np.where((idx >= 0) & (idx % world == rank), idx, -1).astype(np.int32)
    o, l = oracle.sparse_mla(case, own)
    o16 = torch.from_numpy(oracle.round_bf16(o))
    parts_o = [torch.empty_like(o16) for _ in range(world)]
    parts_l = [torch.empty_like(torch.from_numpy(l)) for _ in range(world)]
    dist.all_gather(parts_o, o16)
    dist.all_gather(parts_l, torch.from_numpy(l))
    O = torch.stack(parts_o).numpy()
    L = torch.stack(parts_l).numpy()
    lse = np.logaddexp.reduce(L, axis=0)             # -inf where no rank holds a token
    with np.errstate(invalid="ignore"):
        w = np.where(np.isfinite(L), np.exp(L - np.where(np.isfinite(lse), lse, 0.0)), 0.0)
    out = (w[..., None] * O).sum(axis=0)
    q.put((rank, out, lse))
    dist.destroy_process_group()


def _combine_case(synth):
    case = synth.make_case("gloo_mla", seq_lens=[400, 90], nq=1, topk=64, seed=21)
    rng = np.random.default_rng(21)
    idx = np.full((2, 64), -1, dtype=np.int32)
    idx[0] = np.sort(rng.choice(400, 64, replace=False))
    idx[1, :30] = np.sort(rng.choice(90, 30, replace=False))
    return case, idx


def test_dcp_lse_combine_over_two_gloo_ranks_matches_the_oracle():
    sys.path.insert(0, ROOT)
    import oracle
    from dsa_sparse_attention_index_gb300 import synth

    oracle.build()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_combine, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=180) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    case, idx = _combine_case(synth)
    ref_out, ref_lse, _, _ = oracle.dcp_sparse_mla(case, idx, 2)
    for _, out, lse in res:
        np.testing.assert_allclose(out, ref_out, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(lse, ref_lse, rtol=1e-13)
