"""The N>1 path of the benchmark on CPU: two ranks over the gloo backend.

The layer has no exchange step (replicas only), so what runs across ranks
is the benchmark's own bookkeeping: rendezvous, barriers, the whole-job
aggregation (bytes and tokens summed over ranks, time the maximum), and the
reference arm's rule that only rank 0 does work.
"""
import json
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, outdir: str):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist

    w, r, loc = bench.dist_setup()
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    mx = bench.allreduce_max(1.5 + r, w)
    sm = bench.allreduce_sum(1.0 + r, w)
    # rank r: 1000 bytes and 2 tokens per step over 4 steps, in (r + 1) * 10 ms
    gbs, tok_s, ms = bench.aggregate(1000, 2, 4, (r + 1) * 10.0, w)
    # the reference arm: ranks other than 0 return at once, without output
    ref_ret = bench.run_reference(None, w, r) if r != 0 else None
    bench.barrier(w)
    dist.destroy_process_group()
    with open(os.path.join(outdir, f"rank{r}.json"), "w") as f:
        json.dump({"world": w, "rank": r, "local": loc, "max": mx, "sum": sm, "gbs": gbs, "tok_s": tok_s,
                   "ms": ms, "ref": ref_ret}, f)


def test_two_rank_replica_bookkeeping(tmp_path):
    if not torch.distributed.is_available():
        pytest.skip("torch.distributed is not available")
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r, d in enumerate(res):
        assert (d["world"], d["rank"], d["local"]) == (world, r, r)
        assert d["max"] == 2.5                      # max over ranks of 1.5 + r
        assert d["sum"] == 3.0                      # sum over ranks of 1 + r
        assert d["ms"] == 20.0                      # the slower rank's time
        # 2 ranks x 4 steps x 1000 B in 20 ms; 2 x 4 x 2 tokens in 20 ms
        assert d["gbs"] == pytest.approx(8000 / 0.020 / 1e9)
        assert d["tok_s"] == pytest.approx(16 / 0.020)
    assert res[1]["ref"] is None
