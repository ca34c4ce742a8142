"""Host logic of the multi-rank bench path, on CPU with the gloo backend and two ranks.

The operator shards with no exchange step: each rank reuses its own seeded copy of the
workload and the only collectives are the barrier and the max-over-ranks step time. These
tests run that logic in two processes and check that the shards differ, that nothing of the
data path is exchanged, and that the whole-job throughput divides all ranks' bytes by the
slowest rank's time."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import workloads as wl
        w = wl.config1(seed=bench.rank_seed(rank))
        acc = bench.accounting(w)
        # a fingerprint of this rank's canonical data and page table
        fp = torch.tensor([float(w.items[0].canon_k.float().sum()),
                           float(w.page_table.float().sum())], dtype=torch.float64)
        fps = [torch.zeros_like(fp) for _ in range(world)]
        dist.all_gather(fps, fp)
        # ranks report different local times; the job time is the maximum
        local_ms = 1.0 + rank
        job_ms = bench.job_time_ms(local_ms, world, "cpu")
        dist.barrier()
        value = bench.whole_job_gbs(acc["written"], world, job_ms)
        np.save(os.path.join(out_dir, f"rank{rank}.npy"),
                np.array([job_ms, value, acc["written"]] + [float(x) for f in fps for x in f]))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_rank_sharding_and_max_time(tmp_path):
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    r0 = np.load(tmp_path / "rank0.npy")
    r1 = np.load(tmp_path / "rank1.npy")
    # both ranks agree on the slowest rank's time
    assert r0[0] == r1[0] == 2.0
    # whole-job value: all ranks' bytes over the slowest rank's time
    written = r0[2]
    assert written == r1[2] > 0
    np.testing.assert_allclose(r0[1], written * world / 2e-3 / 1e9)
    np.testing.assert_allclose(r0[1], r1[1])
    # each rank built its own shard: the fingerprints differ between ranks and agree between
    # the two gathers
    fp0, fp1 = r0[3:5], r0[5:7]
    np.testing.assert_array_equal(r0[3:], r1[3:])
    assert not np.array_equal(fp0, fp1)


def test_single_rank_needs_no_process_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_time_ms(3.5, 1) == 3.5
    assert bench.whole_job_gbs(10 ** 9, 1, 1000.0) == pytest.approx(1.0)
