"""Token-sharded balance statistics through the CUDA layer: two processes, each with its own batch
on cuda:0, run moe_layer_forward, then MoELayer.global_balance_stats sums the selection counts and
the raw affinity sums the forward left in its workspace (moe_layer_routing) over a gloo group on
CPU copies, and recomputes f, P and the losses with the global token count (moe_balance_stats).
The result must equal the oracle's statistics of the concatenated batch. The device-level loss
is the reason such statistics cross ranks ("DeepSeekMoE 论文解读" §方法细节, L_DevBal over D
device groups). The two processes share one GPU but never wait on each other inside a kernel:
their only exchange is the host-side all-reduce between calls."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import moe_inputs

pytestmark = pytest.mark.gpu

SHAPE = moe_inputs.CONFIGS["2b_bf16"].with_(T=1000)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    if root not in sys.path:
        sys.path.insert(0, root)
    from fine_grained_moe_softmax_b300 import MoEConfig, MoELayer
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        torch.cuda.set_device(0)
        inputs = moe_inputs.make_inputs(SHAPE, seed=SHAPE.seed + 7919 * rank)
        layer = MoELayer(MoEConfig.from_shape(SHAPE), inputs["centroids"], inputs["w_gate"],
                         inputs["w_up"], inputs["w_down"], inputs["bias"])
        layer.forward(inputs["u"].to("cuda"))
        torch.cuda.synchronize()
        status = layer.device_status()
        local = {k: v.clone().cpu() for k, v in layer.routing().items()}
        f, P, losses = layer.global_balance_stats(SHAPE.T, via_host=True)
        torch.cuda.synchronize()
        np.savez(os.path.join(out_dir, f"rank{rank}.npz"), u=inputs["u"].float().numpy(),
                 idx=layer.topk_idx.cpu().numpy(), psum=local["psum"].numpy(),
                 f=f.cpu().numpy(), P=P.cpu().numpy(), losses=losses.cpu().numpy(),
                 status=np.array(status))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(600)
def test_two_ranks_global_balance_stats(tmp_path):
    import oracle
    from oracle import OracleCfg
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    res = [np.load(tmp_path / f"rank{r}.npz") for r in range(world)]
    for r in res:
        assert int(r["status"]) == 0
    assert not np.array_equal(res[0]["u"], res[1]["u"])
    # the concatenated batch on the oracle: its affinity sums, and its statistics of the GPU's own
    # selections (whose counts are the sum of the ranks' counts)
    cat = moe_inputs.make_inputs(SHAPE)
    cat["u"] = torch.cat([moe_inputs.make_tokens(SHAPE, seed=SHAPE.seed + 7919 * r)
                          for r in range(world)])
    cfg2 = OracleCfg.from_shape(SHAPE, T=world * SHAPE.T)
    ref = oracle.route(cfg2, cat["u"], cat["centroids"], cat["bias"])
    idx = np.concatenate([r["idx"] for r in res])
    counts = np.bincount(idx.ravel(), minlength=SHAPE.n_routed)
    # each rank's local sums against the oracle's sums over that rank's half
    for q, r in enumerate(res):
        half = oracle.route(OracleCfg.from_shape(SHAPE), cat["u"][q * SHAPE.T:(q + 1) * SHAPE.T],
                            cat["centroids"], cat["bias"])
        np.testing.assert_allclose(r["psum"], half["psum"], rtol=2e-4, atol=1e-5)
    st = oracle.balance_stats(cfg2, counts, ref["psum"])
    for r in res:   # every rank ends with the same global statistics
        np.testing.assert_allclose(r["f"], st["f"], rtol=1e-6)
        np.testing.assert_allclose(r["P"], st["P"], rtol=2e-4, atol=1e-7)
        np.testing.assert_allclose(r["losses"], st["losses"], rtol=2e-4)
    np.testing.assert_array_equal(res[0]["f"], res[1]["f"])
    np.testing.assert_array_equal(res[0]["losses"], res[1]["losses"])
