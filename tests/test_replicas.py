"""The multi-GPU path of the benchmark, on CPU: the step shards by sequence
with no exchange, so N GPUs run N replicas that meet only at barriers and in
the max over ranks of the measured times.  Two gloo ranks (spawned
processes, rendezvous on 127.0.0.1) check that helper; the reference arm's
non-zero ranks exit at once without output."""
import multiprocessing as mp
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, values, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench

    reps = bench.Replicas("gloo")
    reps.barrier()
    got = [reps.max(v) for v in values[rank]]
    reps.barrier()
    q.put((rank, reps.world, reps.rank, got))
    reps.close()


def test_two_gloo_replicas_take_the_max_of_their_times():
    values = {0: [1.25, 7.0, -3.0], 1: [2.5, 0.5, -1.0]}
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, values, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert sorted((r, w, rr) for r, w, rr, _ in out) == [(0, 2, 0), (1, 2, 1)]
    for _, _, _, got in out:
        assert got == [2.5, 7.0, -1.0]


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    env = dict(os.environ)
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        os.environ.pop(k, None)
    try:
        reps = bench.Replicas("gloo")
        assert (reps.world, reps.rank) == (1, 0) and reps.max(4.5) == 4.5
        reps.barrier()
        reps.close()
    finally:
        os.environ.clear()
        os.environ.update(env)


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` times the oracle on the host and prints one
    JSON line with the contract's keys (small workload, one step)."""
    import json

    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "decode_b1_l4096", "--steps", "1", "--warmup", "3"], capture_output=True, text=True,
                       env=env, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["config"]["workload"] == "decode_b1_l4096" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1 and d["cpu_baseline"]["cpu"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]


def test_step_percentiles_and_host_cpu():
    sys.path.insert(0, ROOT)
    import bench

    p = bench.step_percentiles([0.2, 0.1, 0.4, 0.3, 0.5])
    assert p == {"ms_p10": 0.14, "ms_p50": 0.3, "ms_p90": 0.46}
    assert "logical cores" in bench.host_cpu()


def test_cpu_baseline_line():
    sys.path.insert(0, ROOT)
    import bench
    from dsa_sparse_attention_index_gb300 import synth

    d = bench.cpu_baseline(synth.make_case("cb", seq_lens=[3000, 700], seed=1), min_seconds=0.0)
    assert d["kind"] == "oracle" and d["value"] > 0 and d["cores"] >= 1 and d["cpu"]
    assert "1 passes" in d["sample"] and "2 of 2 sequences" in d["sample"]


def test_l2_label_says_which_side_of_l2_a_step_is():
    sys.path.insert(0, ROOT)
    import bench

    assert "above the 129 MB L2" in bench.l2_label(522_000_000)
    assert "below the 129 MB L2" in bench.l2_label(1_720_000)
