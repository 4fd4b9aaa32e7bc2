"""The multi-rank host path on the CPU (gloo backend, world size 2).

bench.py runs one rank per GPU: every rank compresses its own gradient
replica (the path has no exchange step), the step time is the largest over
the ranks and the value is the whole job's.  These tests run that host
logic with two gloo processes: the rank environment and seeds, the max over
ranks, the whole-job value, the reference arm's exit on ranks above 0, and
the exchange that would follow compression -- each rank's hybrid output
(from the oracle) gathered in the layout the aggregation call takes, whose
rank-ordered sum equals the ranks' own decompressed values added in order."""
import os
import socket
import sys

import numpy as np
import pytest

WORLD = 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch
    import torch.distributed as dist

    import bench
    import oracle
    from gradient_compression_ef_gb300 import inputs

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (world, rank, rank)
        # the job is as slow as its slowest rank
        ms = [3.0, 5.0][rank]
        slowest = bench.max_over_ranks(torch, ms, world, "cpu")
        assert slowest == 5.0
        assert bench.whole_job_value(world, 1000, slowest) == pytest.approx(2 * 4000 / 5e-3 / 1e9)
        # every rank compresses a gradient of its own (no data-path collective)
        n, k, bits, group = 4096, 41, 8, 64
        g = inputs.student_t(inputs.rng(bench.rank_seed(rank)), n)
        e = np.zeros(n, np.float32)
        idx, codes, scales, _ = oracle.ef_topk_quant(g, e, k, bits, group, "stochastic",
                                                     5 + rank, 0)
        everyone = [torch.zeros(n) for _ in range(world)]
        dist.all_gather(everyone, torch.from_numpy(g))
        assert not np.array_equal(everyone[0].numpy(), everyone[1].numpy())
        # the exchange after compression, in the aggregation layout: rank w's
        # indices at w * K (K = k rounded up to 4), its scales at w * S
        K = -(-k // 4) * 4
        S = -(-scales.size // 4) * 4
        pi = np.zeros(K, np.int32)
        pi[:k] = idx
        ps = np.zeros(S, np.float32)
        ps[:scales.size] = scales
        gi = [torch.zeros(K, dtype=torch.int32) for _ in range(world)]
        gc_ = [torch.zeros(codes.size, dtype=torch.uint8) for _ in range(world)]
        gs = [torch.zeros(S) for _ in range(world)]
        dist.all_gather(gi, torch.from_numpy(pi))
        dist.all_gather(gc_, torch.from_numpy(codes.copy()))
        dist.all_gather(gs, torch.from_numpy(ps))
        all_idx = np.stack([t.numpy()[:k] for t in gi])
        all_codes = np.concatenate([t.numpy() for t in gc_])
        all_scales = np.concatenate([t.numpy() for t in gs])
        agg = oracle.topk_quant_aggregate(all_idx, all_codes, all_scales, world, k, bits, group, n)
        want = np.zeros(n, np.float32)
        for w in range(world):
            vals = oracle.dequant(gc_[w].numpy(), gs[w].numpy()[:scales.size], k, bits, group,
                                  "qsgd")
            for j in range(k):
                want[all_idx[w, j]] = np.float32(want[all_idx[w, j]] + vals[j])
        assert np.array_equal(agg.view(np.uint32), want.view(np.uint32))
        # the reference arm runs on rank 0 only: other ranks exit at once
        if rank != 0:
            saved = sys.argv
            sys.argv = ["bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"]
            try:
                assert bench.run_reference(bench.parse_args()) == 0
            finally:
                sys.argv = saved
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_on_gloo():
    mp = pytest.importorskip("torch.multiprocessing")
    mp.spawn(_worker, args=(WORLD, _free_port()), nprocs=WORLD, join=True)
