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
