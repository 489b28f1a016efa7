"""The N > 1 host paths on CPU (gloo, world size 2): the bench's rendezvous,
max-over-ranks timing and barrier, the reference arm under torchrun (rank 0
alone runs and prints; the other rank exits 0 without work), and the spatially
sharded GroupNorm's exchange: each rank's partial results gathered in rank
order (bwd_gn3d_stats_gb300.shard.all_gather_rank_order) and combined into the
whole volume's.  On CPU the partial results and their combination come from
the fp64 oracle; the library's own kernels for them run in the GPU tests."""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE="2",
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist

    r, ws, local = bench.dist_setup("gloo")
    v = bench.max_over_ranks(float(10 * (r + 1)), ws)
    bench.barrier(ws)
    out.put((r, ws, local, v))
    dist.destroy_process_group()


def test_max_over_ranks_and_barrier_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == [(0, 2, 0, 20.0), (1, 2, 1, 20.0)]


def test_reference_arm_under_torchrun_two_ranks():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2", "--master-addr",
           "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"), "--impl", "reference",
           "--workload", "fp32_2x16x16^3_G4", "--steps", "1", "--warmup", "3", "--gpus", "2"]
    res = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, res.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def _shard_main(rank, port, out):
    """Rank r holds D-slab r of one volume: it computes its slab's moments and
    row sums with the oracle, exchanges them over gloo in rank order, combines,
    and reports what it got."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE="2",
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import numpy as np
    import torch
    import torch.distributed as dist

    import oracle
    from bwd_gn3d_stats_gb300 import shard

    dist.init_process_group("gloo")
    N, C, D, H, W, G = 2, 6, 5, 3, 4, 3
    rng = np.random.default_rng(70)
    x = (1.5 + 2.0 * rng.standard_normal((N, C, D, H, W))).astype(np.float32)
    dy = rng.standard_normal((N, C, D, H, W)).astype(np.float32)
    gamma = rng.uniform(0.5, 1.5, C).astype(np.float32)
    cuts = [(0, 3), (3, 5)]  # rank 0 holds D = 0..2, rank 1 D = 3..4
    d0, d1 = cuts[rank]
    xs = np.ascontiguousarray(x[:, :, d0:d1]).reshape(-1)
    dys = np.ascontiguousarray(dy[:, :, d0:d1]).reshape(-1)
    Sk = (d1 - d0) * H * W
    n, m, q = oracle.moments(xs, N, C, Sk, G)
    mine = torch.from_numpy(np.stack([n, m, q]))
    allm = shard.all_gather_rank_order(mine)  # [2, 3, N*G], rank order
    parts = [tuple(allm[k].numpy()) for k in range(allm.shape[0])]
    cn, cm, cq = oracle.combine_moments(parts)
    rstd = oracle.rstd_of(cn, cq, 1e-5)
    _, _, s1, s2 = oracle.backward_sums(dys, xs, cm, rstd, gamma, N, C, Sk, G)
    alls = shard.all_gather_rank_order(torch.from_numpy(np.stack([s1, s2])))
    t1 = alls[0, 0] + alls[1, 0]
    t2 = alls[0, 1] + alls[1, 1]
    out.put((rank, cn.tolist(), cm.tolist(), rstd.tolist(), t1.tolist(), t2.tolist()))
    dist.destroy_process_group()


def test_sharded_statistics_exchange_gloo():
    """Two ranks, one D-slab each: after the exchange both hold the whole
    volume's counts, means, rstd and row sums (the unsharded oracle's)."""
    import numpy as np

    import oracle

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_shard_main, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    N, C, D, H, W, G = 2, 6, 5, 3, 4, 3
    rng = np.random.default_rng(70)
    x = (1.5 + 2.0 * rng.standard_normal((N, C, D, H, W))).astype(np.float32)
    dy = rng.standard_normal((N, C, D, H, W)).astype(np.float32)
    gamma = rng.uniform(0.5, 1.5, C).astype(np.float32)
    S = D * H * W
    mean, var, rstd = oracle.stats(x.reshape(-1), N, C, S, G, 1e-5)
    _, _, s1, s2 = oracle.backward_sums(dy.reshape(-1), x.reshape(-1), mean, rstd, gamma, N, C, S, G)
    for rank, cn, cm, cr, t1, t2 in got:
        assert np.all(np.array(cn) == (C // G) * S)
        assert np.allclose(cm, mean, rtol=1e-13, atol=1e-14)
        assert np.allclose(cr, rstd, rtol=1e-12)
        assert np.allclose(t1, s1, rtol=1e-12, atol=1e-12) and np.allclose(t2, s2, rtol=1e-12, atol=1e-12)
    assert got[0][1:] == got[1][1:]  # both ranks hold the same bits
