"""Multi-process host logic of the bench on the CPU (gloo, world size 2).

The product path does not shard: under torchrun every rank runs an independent
replica on its own GPU, the ranks meet only at barriers, and the job's time is
the slowest rank's.  These tests run that host logic with two gloo ranks and
no GPU, and check the reference arm's rule that only rank 0 does work."""
import os
import socket
import subprocess
import sys
import textwrap

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


RANK_SCRIPT = textwrap.dedent("""
    import os, sys
    sys.path.insert(0, sys.argv[1])
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo")
    rank, world = dist.get_rank(), dist.get_world_size()
    dist.barrier()
    ms = bench.max_over_ranks(1.5 * (rank + 1), "cpu")        # rank 1 is the slower one
    gbs = bench.job_throughput(3_000_000, world, ms)
    dist.barrier()
    dist.destroy_process_group()
    print("rank %d ms %.3f gbs %.6f" % (rank, ms, gbs))
""")


def test_slowest_rank_and_job_bytes(tmp_path):
    script = tmp_path / "rank.py"
    script.write_text(RANK_SCRIPT)
    port = str(_free_port())
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=port)
        procs.append(subprocess.Popen([sys.executable, str(script), ROOT], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=120)
        assert p.returncode == 0, err
        outs.append(out.strip())
    # both ranks see the slower rank's 3.0 ms; the job moved 2 x 3 MB in it
    for rank, out in enumerate(outs):
        assert out == "rank %d ms 3.000 gbs 2.000000" % rank, outs


def test_single_process_keeps_its_time():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.5, "cpu") == 2.5
    assert abs(bench.job_throughput(5_000_000, 1, 2.5) - 2.0) < 1e-12


def test_reference_arm_other_ranks_do_no_work():
    # Under torchrun the reference arm runs on rank 0 only; rank 1 prints nothing
    # and exits 0 without timing the oracle.
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "0"], env=env, cwd=ROOT, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
