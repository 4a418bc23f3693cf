"""The multi-process path on the CPU (gloo, world size 2).

The store and the gather have no exchange step: each rank works on its own
seeded batch, and ranks only meet at the barrier and at the max of the step
times (weak scaling).  This runs that host logic with two gloo ranks: each rank
builds its own batch, runs it through the CPU oracle, times it, and the ranks
agree on the slowest step and on the whole-job throughput."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import time

    import torch.distributed as dist

    import bench
    import oracle
    from dequant_kvc8_store_gb300 import workloads as W

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        seed = bench.rank_seed("tiny", rank)
        w = W.tiny(seed=seed)
        t0 = time.perf_counter()
        kc, vc, ks, vs = w.k_cache.copy(), w.v_cache.copy(), w.k_scale.copy(), w.v_scale.copy()
        oracle.store(w.quant_mode, w.k_states, w.v_states, kc, vc, ks, vs, w.block_table,
                     w.cu_q_lens, w.context_kv_lens)
        ko, _ = oracle.dequant_gather(w.quant_mode, kc, vc, ks, vs, w.block_table,
                                      w.context_lengths)
        ms = (time.perf_counter() - t0) * 1e3 + 5.0 * rank  # rank 1 is the slow one
        (mx,) = bench.reduce_max([ms])
        nbytes = sum(W.algorithmic_bytes(w).values())
        out[rank] = {"seed": seed, "ms": ms, "max": mx, "first_code": int(kc.reshape(-1)[0]),
                     "digest": int(ko.astype(np.int64).sum()),
                     "value": bench.job_throughput(nbytes, world, mx), "bytes": nbytes}
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_step():
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, join=True,
                           start_method="spawn")
        res = [dict(out[r]) for r in range(world)]
    assert res[0]["seed"] != res[1]["seed"]              # each rank has its own batch
    assert res[0]["digest"] != res[1]["digest"]
    slowest = max(r["ms"] for r in res)
    assert all(abs(r["max"] - slowest) < 1e-9 for r in res)  # both see the same max
    assert res[0]["max"] >= res[1]["ms"] and res[1]["max"] >= res[0]["ms"]
    expect = world * res[0]["bytes"] / (slowest * 1e-3) / 1e9
    assert res[0]["value"] == pytest.approx(expect) and res[1]["value"] == pytest.approx(expect)


def test_single_rank_reduce_is_identity():
    import bench
    assert bench.reduce_max([1.5, 2.0]) == [1.5, 2.0]
    assert bench.job_throughput(1_000_000_000, 1, 1000.0) == pytest.approx(1.0)
