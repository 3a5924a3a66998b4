"""The multi-rank path on CPU with gloo, world size 2: each rank runs its own token batch (the
layer is token-parallel), the benchmark's timing reduction takes the maximum over ranks, and the
one cross-rank exchange of the method -- global balance statistics from summed counts and
affinity sums -- equals the statistics of the concatenated batch. The per-rank layer here is the
oracle (no GPU on this machine); the GPU layer's per-rank outputs are covered by the GPU tests."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import moe_inputs


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    import bench
    import oracle
    from fine_grained_moe_softmax_b300.layer import allreduce_routing_stats
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        sh = moe_inputs.CONFIGS["tiny_f32"].with_(T=96)
        inputs = moe_inputs.make_inputs(sh, seed=bench.rank_token_seed(sh, rank))
        cfg = oracle.OracleCfg.from_shape(sh)
        r = oracle.route(cfg, inputs["u"], inputs["centroids"])
        fw = oracle.forward_tokens(cfg, inputs, np.arange(sh.T))
        counts = torch.from_numpy(r["counts"].astype(np.int32))
        psum = torch.from_numpy(r["psum"].astype(np.float32))
        T_total = allreduce_routing_stats(counts, psum, sh.T)
        worst = bench.max_over_ranks([10.0 + rank, 3.0 - rank], world)
        np.savez(os.path.join(out_dir, f"rank{rank}.npz"), h=fw["h"], counts=counts.numpy(),
                 psum=psum.numpy(), T_total=T_total, worst=np.array(worst),
                 u=inputs["u"].numpy())
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_rank_replicas_and_global_stats(tmp_path):
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    res = [np.load(tmp_path / f"rank{r}.npz") for r in range(world)]
    import oracle
    sh = moe_inputs.CONFIGS["tiny_f32"].with_(T=96)
    # the ranks drew different token batches with the same weights
    assert not np.array_equal(res[0]["u"], res[1]["u"])
    # timing reduction: element-wise maximum on every rank
    for r in res:
        assert list(r["worst"]) == [11.0, 3.0]
        assert int(r["T_total"]) == 2 * sh.T
    # token parallelism: each rank's h equals the single-process h of the concatenated batch
    cat = moe_inputs.make_inputs(sh)
    cat["u"] = torch.cat([torch.from_numpy(r["u"]) for r in res])
    cfg2 = oracle.OracleCfg.from_shape(sh, T=2 * sh.T)
    fw = oracle.forward_tokens(cfg2, cat, np.arange(2 * sh.T))
    np.testing.assert_array_equal(np.concatenate([r["h"] for r in res]), fw["h"])
    # global statistics from the all-reduced counts / sums == statistics of the whole batch
    whole = oracle.route(cfg2, cat["u"], cat["centroids"])
    for r in res:
        np.testing.assert_array_equal(r["counts"], whole["counts"])
        np.testing.assert_allclose(r["psum"], whole["psum"], rtol=1e-6)
    st_red = oracle.balance_stats(cfg2, res[0]["counts"], res[0]["psum"].astype(np.float64))
    st_all = oracle.balance_stats(cfg2, whole["counts"], whole["psum"])
    np.testing.assert_allclose(st_red["losses"], st_all["losses"], rtol=1e-6)
