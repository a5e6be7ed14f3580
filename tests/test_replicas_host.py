"""The multi-GPU form of bench.py is replicas only: every rank runs its own seeded batch
on its own GPU and the ranks share nothing but a barrier around the timed region and
the maximum of their timings. This covers that host-side path with two gloo ranks on
the CPU (no GPU, no collective on the data path)."""
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_RANK_SCRIPT = r"""
import sys
sys.path.insert(0, sys.argv[1])
import bench
r = bench.Ranks()
r.barrier()
m = r.max(float(r.rank + 1) * 1.5)
r.barrier()
print(f"rank={r.rank} world={r.world} max={m}", flush=True)
r.close()
"""


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_share_the_barrier_and_the_max_timing():
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2", MASTER_ADDR="127.0.0.1",
                   MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, "-c", _RANK_SCRIPT, ROOT], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=120)
        assert p.returncode == 0, err[-2000:]
        outs.append(out.strip().splitlines()[-1])
    assert outs == ["rank=0 world=2 max=3.0", "rank=1 world=2 max=3.0"]


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    old = {k: os.environ.pop(k, None) for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    try:
        r = bench.Ranks()
        assert (r.rank, r.world, r.local) == (0, 1, 0)
        r.barrier()
        assert r.max(2.5) == 2.5
        r.close()
    finally:
        for k, v in old.items():
            if v is not None:
                os.environ[k] = v
