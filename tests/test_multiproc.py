"""The multi-rank side of the benchmark on CPU: two gloo ranks draw
independent requests, agree on the slowest rank's time and on the total row
count, with no collective on the data path (each rank's step only reads its
own inputs)."""
import json
import os
import socket

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, outdir):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    import oracle
    from speculative_decoding_pe_gb300 import workloads as wl
    dist.init_process_group("gloo", rank=rank, world_size=world)
    spec = wl.SPECS["tiny"]
    w = wl.make_workload(spec, bench.rank_seed("tiny", rank))
    o = oracle.step(w)                      # each rank: its own requests only
    ms = 1.0 + rank                         # pretend step times
    value, ms_max, rows = bench.aggregate(float(w.T), ms, world, "cpu")
    bench.barrier(world)
    res = {"rank": rank, "value": value, "ms_max": ms_max, "rows": rows,
           "tokens": w.in_tokens.tolist(), "accepted": o["accepted_len"].tolist(),
           "planted": w.planted_accept.tolist()}
    with open(os.path.join(outdir, "r%d.json" % rank), "w") as f:
        json.dump(res, f)
    dist.destroy_process_group()


def test_two_gloo_ranks(tmp_path):
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    r = [json.load(open(tmp_path / ("r%d.json" % i))) for i in range(world)]
    T = 4 * (3 + 3)                           # tiny: B=4, Kp=3, K=3
    for x in r:
        assert x["ms_max"] == 2.0             # the slowest rank's time
        assert x["rows"] == world * T         # rows of all ranks
        assert abs(x["value"] - world * T / 2e-3) < 1e-6
        assert x["accepted"] == x["planted"]
    assert r[0]["tokens"] != r[1]["tokens"]   # independent requests per rank
