"""The sharded method's data flow with real ranks (gloo, CPU processes), as the pages'
equivalence test models it: each rank owns disjoint token rows; the block all-gathers
the tokens, every rank computes its intermediate slice's partial for all of them, and
the reduce-scatter sums the partials and returns each rank its own rows (Kimi-K3 PR,
section "Change"; prhub analysis, section "关键源码片段").  The per-rank arithmetic is
the fp64 oracle's; the exchange is torch.distributed.  gloo has no reduce-scatter, so
the sum is an all-reduce of which each rank keeps its own rows; bf16 bit patterns travel
widened to int32 (gloo has no 16-bit integer type).

Each rank's rows must match the replicated layer on its own tokens, and the rejected
design (feature slices concatenated) must not."""
import os
import socket
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out_dir, T_per_rank, H, I):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import oracle
    import workloads as W
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        T = T_per_rank * world
        x_all = W.make_custom(31, 0, (T, H))                 # drawn identically on every rank
        wgu = W.make_custom(31, 1, (2 * I, H))
        wd = W.make_custom(31, 2, (H, I))
        mine = x_all[rank * T_per_rank:(rank + 1) * T_per_rank]
        # all-gather of the tokens each rank owns
        parts = [torch.empty((T_per_rank, H), dtype=torch.int32) for _ in range(world)]
        dist.all_gather(parts, torch.from_numpy(mine.astype(np.int32)))
        gathered = np.concatenate([p.numpy().astype(np.uint16) for p in parts])
        assert np.array_equal(gathered, x_all)
        # this rank's partial over its intermediate slice, for all gathered tokens (fp32)
        _, partial = oracle.shard_partial(gathered, wgu, wd, world, rank, oracle.F32)
        # reduce-scatter: the sum over ranks, this rank keeping its own token rows
        total = torch.from_numpy(partial.astype(np.float64))
        dist.all_reduce(total)
        own = total.numpy()[rank * T_per_rank:(rank + 1) * T_per_rank]
        # replicated reference: the whole layer on this rank's own tokens
        _, y_ref, _ = oracle.mlp_forward(mine, wgu, wd)
        ok = np.allclose(own, y_ref, rtol=1e-5, atol=1e-5)
        # the rejected design: every rank keeps its own tokens, computes its slice of h,
        # and the feature slices are concatenated as if they were the same tokens'
        s = I // world
        h_mine = oracle.swiglu_hidden(mine, wgu, I, rank * s, (rank + 1) * s)
        hs = [torch.empty((T_per_rank, s), dtype=torch.int32) for _ in range(world)]
        dist.all_gather(hs, torch.from_numpy(h_mine.astype(np.int32)))
        h_cat = np.concatenate([h.numpy().astype(np.uint16) for h in hs], axis=1)
        y_broken = oracle.bf16_array_to_f64(h_cat) @ oracle.bf16_array_to_f64(wd).T
        broken_ok = np.all(np.abs(y_broken - y_ref) <= 0.02 + 0.02 * np.abs(y_ref))
        with open(os.path.join(out_dir, f"r{rank}.txt"), "w") as f:
            f.write(f"{int(ok)} {int(broken_ok)}")
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,T_per_rank,H,I", [(2, 3, 16, 12), (4, 3, 16, 12), (4, 2, 24, 16)])
def test_sharded_block_with_real_ranks_matches_replicated(tmp_path, world, T_per_rank, H, I):
    port = _free_port()
    ctx = torch.multiprocessing.get_context("spawn")
    procs = [ctx.Process(target=_rank, args=(r, world, port, str(tmp_path), T_per_rank, H, I))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(180)
        assert p.exitcode == 0
    for r in range(world):
        ok, broken_ok = open(tmp_path / f"r{r}.txt").read().split()
        assert ok == "1", f"rank {r}: reduced partials differ from the replicated layer"
        assert broken_ok == "0", f"rank {r}: the feature-slice design was not caught"
