#!/usr/bin/env python3
"""DSA decode layer-step benchmark on GB300.

One step = one layer's full decode hot path over one batch: lightning-indexer
scores -> top-2048 -> exact sparse MLA, i.e. ``dsa_decode_step`` of libdsa.
Default workload: the long-context batch (32 sequences, context ~ U(64K,
160K), 10% heavy-tailed keys, FP8 keys and latents, random block table).

Prints ONE JSON line.  ``value`` is the whole-job algorithmic HBM throughput
(GB/s): the key bytes (132 B/token, once per sequence), the selected
latents (576 B/token/row, 352 with NVFP4 latents), queries and outputs, divided by the step time.
The inputs exceed L2 and L2 is also flushed (a 256 MB read) between timed
steps, outside the per-step CUDA-event pairs.  SM clocks are sampled with
nvidia-smi over a soak of identical steps that ends with the timed region.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the fp64 CPU oracle on a bounded sample
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from dsa_sparse_attention_index_gb300 import roofline, synth  # noqa: E402

METRIC = "DSA decode µs/layer-step & achieved HBM GB/s (fraction of 8 TB/s) at 1 GB300"
DEFAULT_WORKLOAD = "longctx_b32_l64k-160k"
NOMINAL_HBM_GBS = 8000.0
L2_FLUSH_BYTES = 256 << 20   # > 129 MB L2; flushed by READING it (clean lines, no write-back)
# The other configurations of the target statement, measured after the headline
# one with the same protocol (fewer steps) and reported in the line's
# "workloads" block: speculative verify, 1M-token MXFP4 keys, chunked prefill.
EXTRA_WORKLOADS = ("specdecode_b8x4_l32768", "mxfp4_b4_l1m", "mxfp4n_b4_l1m", "prefill_q2048_l153600")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--soak-s", type=float, default=1.5, help="seconds of identical steps before the timed region")
    ap.add_argument("--workloads", default=",".join(EXTRA_WORKLOADS),
                    help="other workloads measured after the headline one (comma-separated, 'none' for none)")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def tensor_peak():
    """Dense bf16 tensor TFLOP/s: the measured sustained figure (kernels timed inside
    long back-to-back sequences), else the fallback."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        if "bf16_tflops_sustained" in d:
            return float(d["bf16_tflops_sustained"]), "measured sustained"
        return float(d["bf16_tflops"]), "measured"
    return 1700.0, "fallback sustained"


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        busy = [s for s in sm if smax and s > 0.5 * smax] or sm
        return {"sm_mhz": statistics.median(busy) if busy else None, "sm_max_mhz": smax,
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------- CPU baseline
def cpu_sample(case, n_rows: int):
    """Sub-case of the workload: its first sequences (all their draft rows);
    for a chunk with more rows than n_rows, the last n_rows rows of the first
    sequence (they see the same tokens as in the full chunk)."""
    import copy

    sub = copy.copy(case)
    if case.nq > n_rows:
        sub.nq, sub.batch = n_rows, 1
        sub.seq_lens = case.seq_lens[:1].copy()
        sub.block_table = case.block_table[:1].copy()
        r0, r1 = case.nq - n_rows, case.nq
    else:
        nseq = max(1, min(case.batch, n_rows // case.nq))
        sub.seq_lens = case.seq_lens[:nseq].copy()
        sub.batch = nseq
        sub.block_table = case.block_table[:nseq].copy()
        r0, r1 = 0, nseq * case.nq
    sub.q_index, sub.head_w, sub.q_mla = case.q_index[r0:r1], case.head_w[r0:r1], case.q_mla[r0:r1]
    return sub


def run_oracle(sub):
    import oracle

    t0 = time.perf_counter()
    oracle.decode_step(sub)
    return time.perf_counter() - t0


def host_cpu() -> str:
    """The host's CPU model (x86 `model name`; on Arm the implementer and part
    numbers) and its logical core count."""
    model = ""
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read()
        for key in ("model name", "Model name", "CPU part"):
            for line in info.splitlines():
                if line.split(":")[0].strip() == key:
                    model = (key + " " if key == "CPU part" else "") + line.split(":", 1)[1].strip()
                    break
            if model:
                break
    except OSError:
        pass
    import platform

    return f"{model or platform.processor() or 'unknown'} ({platform.machine()}, {os.cpu_count()} logical cores)"


def l2_label(step_bytes: int, l2_bytes: int = 129 << 20) -> str:
    """How the timed steps treat L2: flushed between steps either way; says
    whether a step's inputs alone would fit in it."""
    side = "above" if step_bytes > l2_bytes else "below"
    return (f"L2 flushed by a 256 MB read between timed steps (outside the step events); a step's algorithmic "
            f"bytes {step_bytes / 1e6:.1f} MB, {side} the 129 MB L2")


def step_percentiles(step_ms) -> dict:
    """Median and p10/p90 of the per-step times (ms)."""
    a = np.asarray(step_ms, dtype=np.float64)
    return {"ms_p10": round(float(np.percentile(a, 10)), 5), "ms_p50": round(float(np.percentile(a, 50)), 5),
            "ms_p90": round(float(np.percentile(a, 90)), 5)}


def cpu_baseline(case, max_rows: int = 4, min_seconds: float = 10.0, max_runs: int = 50):
    """The oracle's decode step on a bounded sample of the workload, repeated
    until about min_seconds of CPU work (at most max_runs passes)."""
    import oracle

    sub = cpu_sample(case, max_rows)
    runs, dt = 0, 0.0
    while runs < max_runs and (runs == 0 or dt < min_seconds):
        dt += run_oracle(sub)
        runs += 1
    b = roofline.step_bytes(sub.seq_lens, sub.nq, sub.topk, sub.key_format, sub.latent_format)["total"]
    return {"value": b * runs / dt / 1e9, "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
            "cpu": host_cpu(),
            "sample": f"{sub.batch} of {case.batch} sequences ({sub.rows} query rows, "
                      f"{int(sub.seq_lens.sum())} context tokens) of the same workload, fp64 C oracle, "
                      f"{runs} passes in {dt:.1f} s"}


def stage_roofline(case, st_ms, traffic=None):
    """Per-stage figures and the dominant kernel's roofline for one workload
    from its median stage times (ms): a prefill chunk or a step whose MLA
    outlasts the indexer against the tensor peak (the indexer's fp8 at the
    measured bf16 peak x 2, the nominal ratio), else the indexer against the
    measured HBM copy bandwidth."""
    k = case.topk
    peak, peak_kind = peaks()
    bf16_peak, bf16_kind = tensor_peak()
    idx_bytes = roofline.indexer_bytes(case.seq_lens, case.nq, case.key_format)
    idx_gbs = idx_bytes / (st_ms["index"] * 1e-3) / 1e9
    idx_fl = roofline.indexer_flops(case.seq_lens, case.nq)
    mla_fl = roofline.mla_flops(case.seq_lens, case.nq, k)
    idx_tf = idx_fl / (st_ms["index"] * 1e-3) / 1e12
    mla_tf = mla_fl / (st_ms["mla"] * 1e-3) / 1e12
    mla_gbs = roofline.mla_bytes(case.seq_lens, case.nq, k, case.latent_format) / (st_ms["mla"] * 1e-3) / 1e9
    stages = {"index": {"us": round(st_ms["index"] * 1e3, 2), "GB/s": round(idx_gbs, 1), "TFLOP/s": round(idx_tf, 1)},
              "topk": {"us": round(st_ms["topk"] * 1e3, 2)},
              "mla": {"us": round(st_ms["mla"] * 1e3, 2), "GB/s": round(mla_gbs, 1), "TFLOP/s": round(mla_tf, 1)}}
    if case.nq > 4 and st_ms["index"] >= st_ms["mla"]:
        roof = {"kernel": "prefill_indexer_kernel (dsa_index_scores)", "bound": "tensor", "achieved": round(idx_tf, 1),
                "peak": 2 * bf16_peak, "peak_kind": bf16_kind + " bf16 x 2 (fp8)", "unit": "TFLOP/s",
                "frac": round(idx_tf / (2 * bf16_peak), 4), "traffic": None, "algorithmic_flops": idx_fl}
    elif st_ms["mla"] > st_ms["index"]:
        roof = {"kernel": "sparse_mla_kernel (sparse_mla_decode)", "bound": "tensor", "achieved": round(mla_tf, 1),
                "peak": bf16_peak, "peak_kind": bf16_kind + " bf16", "unit": "TFLOP/s",
                "frac": round(mla_tf / bf16_peak, 4), "traffic": None, "algorithmic_flops": mla_fl}
    else:
        roof = {"kernel": "indexer_kernel (dsa_index_scores)", "bound": "hbm", "achieved": round(idx_gbs, 1),
                "peak": peak, "peak_kind": peak_kind, "unit": "GB/s", "frac": round(idx_gbs / peak, 4),
                "traffic": traffic, "algorithmic_bytes": idx_bytes}
    return stages, roof


# ---------------------------------------------------------------- replicas
class Replicas:
    """This process among torchrun's ranks (RANK, LOCAL_RANK, WORLD_SIZE): one
    independent replica of the step per GPU.  The data path has no exchange;
    the ranks only meet at barriers around the timed region and in the max
    over ranks of the measured times."""

    def __init__(self, backend: str):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        if self.world > 1:
            import torch.distributed as dist

            dist.init_process_group(backend)

    def barrier(self):
        if self.world > 1:
            import torch.distributed as dist

            dist.barrier()

    def max(self, x: float, device="cpu") -> float:
        """The largest x over the ranks (every rank gets it)."""
        if self.world == 1:
            return float(x)
        import torch
        import torch.distributed as dist

        t = torch.tensor([float(x)], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()


# ---------------------------------------------------------------- GPU arm
def main_ours(args):
    import torch

    from dsa_sparse_attention_index_gb300 import binding

    reps = Replicas("nccl")
    world, rank, local = reps.world, reps.rank, reps.local
    torch.cuda.set_device(local)
    binding.lib()  # fail loudly if the CUDA library is missing

    case = synth.workload(args.workload, seed=args.seed)
    dc = synth.device_case(case)
    k = case.topk
    rows = case.rows
    ld = (case.max_len + 3) // 4 * 4
    dev = torch.device("cuda", local)
    out = torch.empty((rows, 96, 512), dtype=torch.int16, device=dev)
    lse = torch.empty((rows, 96), dtype=torch.float32, device=dev)
    scores = torch.empty((rows, ld), dtype=torch.float32, device=dev)
    idx = torch.empty((rows, k), dtype=torch.int32, device=dev)
    ws = binding.workspace(binding.workspace_size(dc.batch, k), dev)
    tk_ws = binding.workspace(binding.topk_workspace_size(rows, case.max_len, k), dev)
    mla_ws = binding.workspace(binding.sparse_mla_workspace_size(rows, k), dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flush_buf = torch.ones(L2_FLUSH_BYTES // 8, dtype=torch.int64, device=dev)
    flush_sink = torch.empty((), dtype=torch.int64, device=dev)

    class _Flush:
        @staticmethod
        def zero_():  # read 256 MB: evicts L2 with clean lines, outside the step events
            flush_sink.copy_(flush_buf.sum())

    flush = _Flush()
    stream = torch.cuda.current_stream()

    def step():
        binding.decode_step(dc.cache, dc.batch, dc.q_index, dc.head_w, dc.q_mla, k, case.sm_scale, out, lse, ws,
                            status, stream=stream)

    def barrier():
        reps.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        flush.zero_()
        step()
    barrier()
    assert status.item() == 0, binding.status_string(status.item())

    # ---- headline: K fused steps, each bracketed by its own events, L2 flushed in between
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        t_soak = time.perf_counter()
        while time.perf_counter() - t_soak < args.soak_s:
            for _ in range(20):
                flush.zero_()
                step()
            torch.cuda.synchronize()
        barrier()
        t_wall = time.perf_counter()
        n_launch0 = binding.kernel_launches()
        for e0, e1 in ev:
            flush.zero_()
            e0.record(stream)
            step()
            e1.record(stream)
        n_launches = binding.kernel_launches() - n_launch0
        barrier()
        t_wall = time.perf_counter() - t_wall
    clocks = clk.summary()
    step_ms = [e0.elapsed_time(e1) for e0, e1 in ev]
    ms = reps.max(statistics.mean(step_ms), dev)
    assert status.item() == 0, binding.status_string(status.item())

    # ---- per-stage attribution (same kernels through the three stage entry points)
    stage = {"index": [], "topk": [], "mla": []}
    n_att = max(5, args.steps)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n_att)]
    for e in evs:  # enqueued back to back: the GPU never waits for the host inside an event pair
        flush.zero_()
        e[0].record(stream)
        binding.index_scores(dc.cache, dc.batch, dc.q_index, dc.head_w, scores, status, stream)
        e[1].record(stream)
        binding.topk(scores, dc.row_lens, case.max_len, k, idx, tk_ws, status, stream)
        e[2].record(stream)
        binding.sparse_mla_decode(dc.cache, dc.batch, dc.q_mla, idx, case.sm_scale, out, lse, mla_ws, status, stream)
        e[3].record(stream)
    torch.cuda.synchronize()
    for e in evs:
        stage["index"].append(e[0].elapsed_time(e[1]))
        stage["topk"].append(e[1].elapsed_time(e[2]))
        stage["mla"].append(e[2].elapsed_time(e[3]))
    assert status.item() == 0, binding.status_string(status.item())
    st_ms = {kk: statistics.median(v) for kk, v in stage.items()}

    # ---- the same step with bf16 scores between the indexer and the top-k: the
    #      fused call, its two first stages, and how often the selection moves
    b16 = None
    if rank == 0:
        ld16 = (case.max_len + 7) // 8 * 8
        s16 = torch.empty((rows, ld16), dtype=torch.int16, device=dev)
        idx16 = torch.empty((rows, k), dtype=torch.int32, device=dev)
        evf = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n_att)]
        for e in evf:
            flush.zero_()
            e[0].record(stream)
            binding.decode_step_bf16(dc.cache, dc.batch, dc.q_index, dc.head_w, dc.q_mla, k, case.sm_scale, out,
                                     lse, ws, status, stream=stream)
            e[1].record(stream)
        evb = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n_att)]
        for e in evb:
            flush.zero_()
            e[0].record(stream)
            binding.index_scores_bf16(dc.cache, dc.batch, dc.q_index, dc.head_w, s16, status, stream)
            e[1].record(stream)
            binding.topk_bf16(s16, dc.row_lens, case.max_len, k, idx16, status, stream)
            e[2].record(stream)
        torch.cuda.synchronize()
        assert status.item() == 0, binding.status_string(status.item())
        med = lambda evs, a, b_: round(statistics.median(e[a].elapsed_time(e[b_]) for e in evs) * 1e3, 2)
        same = int((idx16 == idx).all(dim=1).sum().item())  # `idx` holds the fp32 selection of the same step
        n_scores = int(case.row_lens().astype(np.int64).sum())
        b16 = {"step_us": med(evf, 0, 1), "index_us": med(evb, 0, 1), "topk_us": med(evb, 1, 2),
               "score_bytes_per_step": 2 * n_scores, "fp32_score_bytes_per_step": 4 * n_scores,
               "rows_with_the_fp32_selection": same, "rows": rows}

    # ---- the decode-context-parallel top-k merge of 8 shards on the step's scores
    #      (L2-resident after the indexer, as in a step): time and words sent
    dcp = None
    shards = 8
    if case.max_len <= 65536 * shards and rank == 0:
        dcp_ws = binding.workspace(binding.dcp_topk_workspace_size(rows, k, shards), dev)
        dcp_idx = torch.empty((rows, k), dtype=torch.int32, device=dev)
        dcp_stats = torch.empty((rows, 3), dtype=torch.int32, device=dev)
        dev_ = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n_att)]
        for e in dev_:
            flush.zero_()
            binding.index_scores(dc.cache, dc.batch, dc.q_index, dc.head_w, scores, status, stream)
            e[0].record(stream)
            binding.dcp_topk(scores, dc.row_lens, case.max_len, k, shards, dcp_idx, dcp_ws, status,
                             stats_out=dcp_stats, stream=stream)
            e[1].record(stream)
        torch.cuda.synchronize()
        assert status.item() == 0, binding.status_string(status.item())
        stt = dcp_stats.cpu().numpy()
        words = float(stt[:, 0].mean())
        per_shard = words / shards * 4
        dcp = {"shards": shards, "us": round(statistics.median(e[0].elapsed_time(e[1]) for e in dev_) * 1e3, 2),
               "launches": 4, "words_per_row": round(words, 1), "rows_with_resend": int((stt[:, 1] > 0).sum()),
               "bytes_per_shard_and_row": round(per_shard, 1),
               "vs_full_local_topk_pairs": round(k * 8 / per_shard, 2)}
        # the partial attention of the 8 shards over the merged selection and the
        # LSE combine of their bf16 outputs (L2 flushed before each call)
        cm_ws = binding.workspace(binding.dcp_sparse_mla_workspace_size(rows, k, shards), dev)
        cm_out = torch.empty_like(out)
        cm_lse = torch.empty_like(lse)
        evc = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n_att)]
        for e in evc:
            flush.zero_()
            e[0].record(stream)
            binding.dcp_sparse_mla(dc.cache, dc.batch, dc.q_mla, dcp_idx, shards, case.sm_scale, cm_out, cm_lse,
                                   cm_ws, status, stream=stream)
            e[1].record(stream)
        binding.sparse_mla_decode(dc.cache, dc.batch, dc.q_mla, dcp_idx, case.sm_scale, out, lse, mla_ws, status,
                                  stream)
        torch.cuda.synchronize()
        assert status.item() == 0, binding.status_string(status.item())
        diff = (cm_out.view(torch.bfloat16).float() - out.view(torch.bfloat16).float()).abs().max().item()
        dcp["lse_combine"] = {
            "us": round(statistics.median(e[0].elapsed_time(e[1]) for e in evc) * 1e3, 2), "launches": 3,
            "partial_bytes_per_shard_and_row": 96 * 512 * 2 + 96 * 4,
            "max_abs_vs_unsharded": round(diff, 5)}

    # ---- the fused indexer front end on this batch (RMSNorm, the 4096 x 1536 query projection,
    #      FP8 query, the new tokens into the cache) alone, and the step that owns its cache
    #      update (front end + step, one call); both write the cache, so they run on a copy
    fe_block = None
    if rank == 0:
        fe = synth.make_frontend(rows, seed=args.seed)
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if a.dtype == np.uint16
                                       else np.ascontiguousarray(a)).to(dev)
        f_cq, f_g, f_w, f_hw, f_lat, f_key = (t(fe.c_q), t(fe.gamma), t(fe.w_iq), t(fe.head_w), t(fe.new_latent),
                                              t(fe.new_key))
        pool_copy = dc.cache.pool.clone()
        f_cache = binding.PagedCache(pool=pool_copy, row_stride=dc.cache.row_stride, latent_off=dc.cache.latent_off,
                                     index_off=dc.cache.index_off, key_format=dc.cache.key_format,
                                     latent_scale=dc.cache.latent_scale, latent_format=dc.cache.latent_format)
        f_qi = torch.empty_like(dc.q_index)
        f_wo = torch.empty_like(dc.head_w)
        f_ws = binding.workspace(binding.frontend_workspace_size(dc.batch, k), dev)
        evf = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n_att)]
        for e in evf:
            flush.zero_()
            e[0].record(stream)
            binding.index_frontend(f_cache, dc.batch, f_cq, f_g, fe.eps, f_w, f_hw, f_lat, f_key, f_qi, f_wo, status,
                                   stream=stream)
            e[1].record(stream)
        evs2 = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n_att)]
        for e in evs2:
            flush.zero_()
            e[0].record(stream)
            binding.decode_step_frontend(f_cache, dc.batch, f_cq, f_g, fe.eps, f_w, f_hw, f_lat, f_key, dc.q_mla, k,
                                         case.sm_scale, out, lse, f_ws, status, stream=stream)
            e[1].record(stream)
        torch.cuda.synchronize()
        assert status.item() == 0, binding.status_string(status.item())
        fe_us = statistics.median(e[0].elapsed_time(e[1]) for e in evf) * 1e3
        # bytes the front end must move: the projection weights once, the queries, the
        # outputs and the new tokens' cache records
        fe_bytes = (fe.w_iq.nbytes + fe.gamma.nbytes + fe.c_q.nbytes + fe.head_w.nbytes + fe.new_latent.nbytes +
                    fe.new_key.nbytes + rows * (4096 + 128) + rows * (case.latent_bytes() + case.token_bytes()))
        fe_block = {"us": round(fe_us, 2), "algorithmic_bytes": int(fe_bytes), "GB/s": round(fe_bytes / fe_us / 1e3, 1),
                    "q_rank": int(fe.c_q.shape[1]), "launches": 1,
                    "step_with_frontend_us": round(statistics.median(e[0].elapsed_time(e[1]) for e in evs2) * 1e3, 2)}
        del pool_copy, f_cache

    # ---- end to end through the public call, host buffers, copies inside the timed region:
    #      the step's host inputs packed in one pinned buffer (one host->device copy into a
    #      device buffer whose views are the step's arguments), its outputs in one device
    #      buffer (one device->host copy into pinned memory)
    e2e_ms = []
    if not args.no_e2e:
        from dsa_sparse_attention_index_gb300 import binding as B

        srcs = [dc.q_index, dc.head_w, dc.q_mla, dc.batch.block_table, dc.batch.seq_lens]
        al = lambda n: (n + 255) // 256 * 256
        offs, tot = [], 0
        for t in srcs:
            offs.append(tot)
            tot += al(t.numel() * t.element_size())
        h_in = torch.empty(tot, dtype=torch.uint8).pin_memory()
        d_in = torch.empty(tot, dtype=torch.uint8, device=dev)
        views = []
        for t, o in zip(srcs, offs):
            n = t.numel() * t.element_size()
            h_in[o:o + n].copy_(t.contiguous().view(-1).view(torch.uint8).cpu())
            views.append(d_in[o:o + n].view(t.dtype).view(t.shape))
        e_qi, e_w, e_qm, e_bt, e_sl = views
        e_batch = B.Batch(block_table=e_bt, seq_lens=e_sl, queries_per_seq=case.nq, max_seq_len=max(case.max_len, 0))
        o_bytes = al(out.numel() * 2)
        d_out = torch.empty(o_bytes + lse.numel() * 4, dtype=torch.uint8, device=dev)
        e_out = d_out[:out.numel() * 2].view(torch.int16).view(out.shape)
        e_lse = d_out[o_bytes:].view(torch.float32).view(lse.shape)
        h_out = torch.empty(d_out.numel(), dtype=torch.uint8).pin_memory()
        bi, bo = tot, d_out.numel()
        for it in range(args.warmup + args.steps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            d_in.copy_(h_in, non_blocking=True)
            B.decode_step(dc.cache, e_batch, e_qi, e_w, e_qm, k, case.sm_scale, e_out, e_lse, ws, status,
                          stream=stream)
            h_out.copy_(d_out, non_blocking=True)
            e1.record(stream)
            torch.cuda.synchronize()
            if it >= args.warmup:
                e2e_ms.append(e0.elapsed_time(e1))
        step()  # the device-resident step once more: the e2e call computed the same outputs
        torch.cuda.synchronize()
        assert status.item() == 0, binding.status_string(status.item())
        assert torch.equal(e_out, out) and torch.equal(e_lse, lse)
        e2e_t = reps.max(statistics.mean(e2e_ms), dev)

    b = roofline.step_bytes(case.seq_lens, case.nq, k, case.key_format, case.latent_format)
    total_bytes = b["total"] * world
    value = total_bytes / (ms * 1e-3) / 1e9
    stages, roof = stage_roofline(case, st_ms, load_traffic(args.workload))
    roof["step_frac"] = round(value / world / peaks()[0], 4)
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 5),
        **step_percentiles(step_ms),
        "us_per_layer_step": round(ms * 1e3, 2),
        "tokens_per_s": round(rows * world / (ms * 1e-3), 1),
        "frac_of_8TBps": round(value / world / NOMINAL_HBM_GBS, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3 x e4m3 -> fp32 (indexer); bf16 x bf16 -> fp32 (MLA)",
        "data": "synthetic",
        "config": {
            "workload": args.workload, "batch": case.batch, "queries_per_seq": case.nq,
            "seq_len_mean": float(np.mean(case.seq_lens)), "seq_len_min": int(case.seq_lens.min()),
            "seq_len_max": int(case.seq_lens.max()), "topk": k, "key_bytes": case.token_bytes(),
            "latent_bytes": case.latent_bytes(), "heads": 96, "index_heads": 32, "block": 64,
            "algorithmic_bytes_per_step": b["total"], "parallelism": f"replicas x{world}",
            "l2": l2_label(b["total"]),
        },
        "stage_us": {kk: round(v * 1e3, 2) for kk, v in st_ms.items()},
        "stages": stages,
        "roofline": roof,
        "gpu_launches": n_launches,
        "dcp_topk": dcp,
        "frontend": fe_block,
        "bf16_scores": b16,
        "clocks": clocks,
        "wall_s_timed_region": round(t_wall, 4),
    }
    if e2e_ms:
        line["e2e"] = {"value": round(total_bytes / (e2e_t * 1e-3) / 1e9, 1), "unit": "GB/s",
                       "ms_per_step": round(e2e_t, 5), "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo}
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(case)
    extra = [w for w in args.workloads.split(",") if w and w != "none" and w != args.workload]
    if rank == 0 and extra:  # the headline's buffers stay: HBM holds both
        line["workloads"] = {w: measure_workload(w, args, dev, flush, stream, max(5, min(args.steps, 20)))
                             for w in extra}
    if rank == 0:
        print(json.dumps(line), flush=True)
    reps.close()


def measure_workload(name, args, dev, flush, stream, steps):
    """One more workload with the headline's protocol: warm-up steps, a soak
    under the clock sampler, `steps` fused steps each bracketed by its own
    events with L2 flushed in between, then the three stages enqueued back to
    back.  Returns its block of the JSON line; frees its buffers."""
    import torch

    from dsa_sparse_attention_index_gb300 import binding

    case = synth.workload(name, seed=args.seed)
    dc = synth.device_case(case, dev)
    k, rows = case.topk, case.rows
    ld = (case.max_len + 3) // 4 * 4
    out = torch.empty((rows, 96, 512), dtype=torch.int16, device=dev)
    lse = torch.empty((rows, 96), dtype=torch.float32, device=dev)
    scores = torch.empty((rows, ld), dtype=torch.float32, device=dev)
    idx = torch.empty((rows, k), dtype=torch.int32, device=dev)
    ws = binding.workspace(binding.workspace_size(dc.batch, k), dev)
    tk_ws = binding.workspace(binding.topk_workspace_size(rows, case.max_len, k), dev)
    mla_ws = binding.workspace(binding.sparse_mla_workspace_size(rows, k), dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def step():
        binding.decode_step(dc.cache, dc.batch, dc.q_index, dc.head_w, dc.q_mla, k, case.sm_scale, out, lse, ws,
                            status, stream=stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    assert status.item() == 0, binding.status_string(status.item())
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    with ClockSampler(torch.cuda.current_device()) as clk:
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < min(args.soak_s, 0.5):
            for _ in range(5):
                flush.zero_()
                step()
            torch.cuda.synchronize()
        n0 = binding.kernel_launches()
        for e0, e1 in ev:
            flush.zero_()
            e0.record(stream)
            step()
            e1.record(stream)
        n_launches = binding.kernel_launches() - n0
        torch.cuda.synchronize()
    step_ms = [e0.elapsed_time(e1) for e0, e1 in ev]
    assert status.item() == 0, binding.status_string(status.item())
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    for e in evs:
        flush.zero_()
        e[0].record(stream)
        binding.index_scores(dc.cache, dc.batch, dc.q_index, dc.head_w, scores, status, stream)
        e[1].record(stream)
        binding.topk(scores, dc.row_lens, case.max_len, k, idx, tk_ws, status, stream)
        e[2].record(stream)
        binding.sparse_mla_decode(dc.cache, dc.batch, dc.q_mla, idx, case.sm_scale, out, lse, mla_ws, status, stream)
        e[3].record(stream)
    torch.cuda.synchronize()
    assert status.item() == 0, binding.status_string(status.item())
    st_ms = {kk: statistics.median(e[j].elapsed_time(e[j + 1]) for e in evs)
             for j, kk in enumerate(("index", "topk", "mla"))}
    ms = statistics.mean(step_ms)
    b = roofline.step_bytes(case.seq_lens, case.nq, k, case.key_format, case.latent_format)["total"]
    stages, roof = stage_roofline(case, st_ms, load_traffic(name))
    roof["step_frac"] = round(b / (ms * 1e-3) / 1e9 / peaks()[0], 4)
    res = {"ms_per_step": round(ms, 5), **step_percentiles(step_ms), "us_per_layer_step": round(ms * 1e3, 2),
           "value": round(b / (ms * 1e-3) / 1e9, 1), "unit": "GB/s", "tokens_per_s": round(rows / (ms * 1e-3), 1),
           "steps": steps, "gpu_launches": n_launches,
           "config": {"batch": case.batch, "queries_per_seq": case.nq, "seq_len_mean": float(np.mean(case.seq_lens)),
                      "topk": k, "key_bytes": case.token_bytes(), "latent_bytes": case.latent_bytes(),
                      "algorithmic_bytes_per_step": b, "l2": l2_label(b)},
           "stage_us": {kk: round(v * 1e3, 2) for kk, v in st_ms.items()}, "stages": stages, "roofline": roof,
           "clocks": clk.summary()}
    del dc, out, lse, scores, idx, ws, tk_ws, mla_ws
    torch.cuda.empty_cache()
    return res


def load_traffic(workload):
    """DRAM bytes per indexer launch from the committed ncu summary, if any,
    and only while the indexer's source is the one the counters were taken
    from (its sha256 is recorded beside them)."""
    import hashlib

    p = os.path.join(ROOT, "profiles", "indexer_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    src = os.path.join(ROOT, "dsa_sparse_attention_index_gb300", "csrc", "indexer.cu")
    with open(src, "rb") as f:
        if hashlib.sha256(f.read()).hexdigest() != d.get("indexer_source_sha256"):
            return None
    return d.get(workload)


# ---------------------------------------------------------------- reference arm
def main_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle

    case = synth.workload(args.workload, seed=args.seed)
    sub = cpu_sample(case, 1)
    for _ in range(min(args.warmup, 1)):
        run_oracle(sub)
    times = [run_oracle(sub) for _ in range(args.steps)]
    dt = statistics.mean(times)
    b = roofline.step_bytes(sub.seq_lens, sub.nq, sub.topk, sub.key_format, sub.latent_format)["total"]
    v = b / dt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "sample": f"{sub.batch} sequence(s), {sub.rows} query row(s)"},
        "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
                         "cpu": host_cpu(),
                         "sample": f"first {sub.batch} sequence(s) of the workload per step"},
        "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    a = parse()
    if a.impl == "reference":
        main_reference(a)
    else:
        main_ours(a)
