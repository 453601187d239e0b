"""The multi-GPU path of bench.py on CPU: two gloo ranks (world size 2).

Replicas only: every rank runs its own batch with no exchange in the data
path; the only collectives are the timing barrier and the max over ranks of
the step time.  This checks, with real process groups, the pieces of that
path that need no GPU: rendezvous through bench.dist_setup, distinct
replica batches, the max-over-ranks reduction every rank agrees on, and the
whole-job throughput formula."""
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    from gpt_transformer_forward_gb300 import inputs

    r, wsz, local, pg = bench.dist_setup(world)
    assert (r, wsz, local) == (rank, world, rank) and pg is not None
    w = inputs.WORKLOADS["tiny"]
    _, tok = inputs.workload_inputs(w)
    mine = bench.rank_tokens(w, tok, r)
    ms = 10.0 + 5.0 * r  # rank 1 is the slower one
    slowest = bench.max_over_ranks(ms, pg, "cpu")
    pg.barrier()
    np.save(os.path.join(out_dir, f"tok{r}.npy"), mine)
    with open(os.path.join(out_dir, f"rank{r}.txt"), "w") as f:
        f.write(f"{slowest} {bench.job_tokens_per_s(wsz, w.B * w.T, slowest)}")
    pg.destroy_process_group()


def test_two_gloo_ranks(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, start_method="spawn",
                       join=True)
    sys.path.insert(0, ROOT)
    from gpt_transformer_forward_gb300 import inputs
    w = inputs.WORKLOADS["tiny"]
    _, tok = inputs.workload_inputs(w)
    t0, t1 = np.load(tmp_path / "tok0.npy"), np.load(tmp_path / "tok1.npy")
    np.testing.assert_array_equal(t0, tok)                 # rank 0: the workload's batch
    assert t1.shape == tok.shape and not np.array_equal(t1, tok)  # rank 1: its own
    assert t1.min() >= 0 and t1.max() < w.cfg.vocab_size
    vals = [open(tmp_path / f"rank{r}.txt").read().split() for r in range(world)]
    for slowest, value in vals:  # every rank holds the max and the same job value
        assert float(slowest) == pytest.approx(15.0)
        assert float(value) == pytest.approx(world * w.B * w.T / 15e-3)
