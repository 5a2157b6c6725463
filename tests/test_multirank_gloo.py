"""The benchmark's multi-rank plumbing on CPU: two ranks over the gloo backend (127.0.0.1).

On a multi-GPU node `bench.py` runs one independent decode replica per rank (its own seeded
sequences, no collective on the data path); the only cross-rank operations are a barrier around
the timed region and a max-reduction of the elapsed time.  These tests run exactly those
operations, and the replica seeding, in two spawned processes."""
import json
import os
import socket

import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    import bench
    import workloads as wl
    dist = bench.Dist()
    try:
        dist.barrier()
        got_max = dist.max(10.0 * rank + 0.25)                 # each rank's "elapsed time"
        w = wl.shrink(wl.WORKLOADS["decode_1m_b32_csa_hca"], seed=rank)
        res = {"max": got_max, "world": dist.world, "lengths": list(map(int, w.lengths())), "B": w.B, "H": w.H,
               "d": w.d, "k": w.k}
        dist.barrier()
    finally:
        dist.close()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump(res, f)


def test_two_gloo_ranks_time_max_and_independent_replicas(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    r = [json.load(open(tmp_path / f"rank{i}.json")) for i in range(world)]
    # the timing is the max over ranks, seen identically by every rank
    assert r[0]["max"] == r[1]["max"] == 10.25
    assert r[0]["world"] == r[1]["world"] == world
    # each rank decodes its own replica: same shapes, different seeded sequence lengths
    for key in ("B", "H", "d", "k"):
        assert r[0][key] == r[1][key]
    assert len(r[0]["lengths"]) == len(r[1]["lengths"]) == r[0]["B"]
    assert r[0]["lengths"] != r[1]["lengths"]
    assert all(524288 <= x <= 1048576 for x in r[0]["lengths"] + r[1]["lengths"])
