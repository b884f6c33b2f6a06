"""The N > 1 host path of bench.py on CPU: two gloo ranks on 127.0.0.1 reduce
their step times with a max and report whole-job throughput; the reference arm
does no work on ranks other than 0."""
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_total = [30.0, 45.0][rank]  # ms summed over 10 steps
    ms = bench.reduce_step_time(local_total, 10, world)
    q.put((rank, ms, bench.job_throughput(4, world, ms)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_step_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, value in out:
        assert abs(ms - 4.5) < 1e-12          # max(30, 45) / 10
        assert abs(value - 2 * 4 / 4.5e-3) < 1e-6


def test_reference_arm_is_silent_on_other_ranks():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "3", "--warmup", "3"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_shard_ranges_cover_every_context_once():
    """Weak scaling: the job of N GPUs holds N times one GPU's contexts, and the
    ranks' shares are disjoint and together cover all of them."""
    sys.path.insert(0, ROOT)
    from rank_cache_attention_flash_b300 import inputs as I

    for n_global in (1, 7, 16, 64, 128):
        for world in (1, 2, 3, 4, 8):
            seen = []
            for r in range(world):
                seen.extend(I.shard_range(n_global, world, r))
            assert sorted(seen) == list(range(n_global))
            sizes = [len(I.shard_range(n_global, world, r)) for r in range(world)]
            assert max(sizes) - min(sizes) <= 1


def test_ranks_build_disjoint_contexts():
    """Each rank's share of the long paged decode reads its own hidden-state
    streams (distinct sequences), and the union over ranks is the global job:
    rank r of 2 holds exactly global sequences [n r, n r + n)."""
    sys.path.insert(0, ROOT)
    from rank_cache_attention_flash_b300 import inputs as I

    def streams(case):
        return [q.own_stream for q in case.seqs]

    small = dict(n_seqs=4, n=48)
    world = 2
    shares = [I.long_decode(first=I.shard_range(world * 4, world, r).start, **small) for r in range(world)]
    whole = I.long_decode(n_seqs=8, n=48)
    got = streams(shares[0]) + streams(shares[1])
    assert got == streams(whole)
    assert len(set(got)) == len(got)
    # queries and adapter ids of the shares are the whole job's rows
    import torch

    assert torch.equal(torch.cat([c.dec_q for c in shares]), whole.dec_q)
    assert torch.equal(torch.cat([c.dec_adapter for c in shares]), whole.dec_adapter)
    # the weights are the same model on every rank
    for k in whole.weights:
        assert torch.equal(shares[1].weights[k], whole.weights[k])
    # every full-size workload builds one equal share per rank
    for name, units in I.SHARD_UNITS.items():
        assert sum(len(I.shard_range(world * units, world, r)) for r in range(world)) == world * units
