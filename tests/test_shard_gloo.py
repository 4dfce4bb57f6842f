"""Multi-rank host logic on CPU (gloo, world size 2): each rank selects over
its own contiguous row block; the concatenation of the blocks equals the
selection over the whole matrix. The bench's reference arm also runs under
torchrun with two ranks (rank 0 reports, rank 1 exits without work)."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

from maxk_sparse_activations_gb300.shard import row_range

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_row_range_partitions():
    for N in (0, 1, 7, 1000, 1 << 20):
        for world in (1, 2, 3, 8):
            spans = [row_range(N, r, world) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == N
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
            sizes = [b - a for a, b in spans]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        row_range(10, 2, 2)


def _worker(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    from maxk_sparse_activations_gb300 import synth
    x = synth.normal_f32(1001, 256, seed=0)
    a, b = row_range(x.shape[0], rank, world)
    _, idx, it = oracle.replay(x[a:b], 32, 3, 0.0)
    got = [None] * world
    dist.all_gather_object(got, (a, b, idx, it))
    if rank == 0:
        idx_all = np.concatenate([g[2] for g in got])
        it_all = np.concatenate([g[3] for g in got])
        _, ref_idx, ref_it = oracle.replay(x, 32, 3, 0.0)
        ok = bool(np.array_equal(idx_all, ref_idx) and np.array_equal(it_all, ref_it))
        with open(os.path.join(out_dir, "ok"), "w") as f:
            f.write("1" if ok else "0")
    dist.barrier()
    dist.destroy_process_group()


def test_sharded_rows_equal_whole(tmp_path, oracle_mod):
    port = 29500 + (os.getpid() % 1000)
    mp.spawn(_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    assert (tmp_path / "ok").read_text() == "1"


def _one_json_line(p):
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, p.stdout[-2000:]
    return json.loads(lines[0])


def test_bench_reference_arm_two_ranks_under_torchrun(oracle_mod):
    port = 30500 + (os.getpid() % 1000)
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "2", "--warmup", "0", "--rows", "65536", "--ref-seconds", "2"]
    d = _one_json_line(subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600))
    assert d["impl"] == "reference" and d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["n_gpus"] == 2 and d["e2e"]["h2d_bytes_per_step"] == 0


def test_bench_gpus_flag_launches_the_ranks_itself(oracle_mod):
    """`bench.py --gpus 2` without an outer torchrun starts two ranks itself;
    rank 0 alone prints the line and reports both ranks."""
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0",
           "--rows", "65536", "--ref-seconds", "2"]
    d = _one_json_line(subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600))
    assert d["impl"] == "reference" and d["n_gpus"] == 2


def test_bench_rejects_a_world_size_that_differs_from_gpus():
    env = dict(os.environ, WORLD_SIZE="1", RANK="0")
    p = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--gpus", "2"], cwd=ROOT,
                       capture_output=True, text=True, timeout=120, env=env)
    assert p.returncode != 0 and "WORLD_SIZE" in p.stderr
