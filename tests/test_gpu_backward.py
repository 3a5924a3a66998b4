"""GPU parity of the layer backward (moe_layer_backward through the C ABI) against the fp64
oracle's backward, which is itself pinned by finite differences (test_oracle_backward.py).

Objective: sum_t dh_t . h_t + L_ExpBal + L_DevBal with the expert selection and counts held fixed
("DeepSeekMoE 论文解读" §方法细节). bf16 layers; every gradient tensor is compared by rel-L2."""
import numpy as np
import pytest
import torch

import moe_inputs
import oracle
from oracle import OracleCfg
from parity import NEAR_TIE, rel_l2, to_np

pytestmark = pytest.mark.gpu

TOL = 2e-2


def _shape(**kw):
    base = dict(name="bwd", T=200, d=128, n_shared=1, n_routed=16, inter=32, top_k=4,
                n_groups=4, dtype="bf16", seed=21, alpha1=0.01, alpha2=0.05)
    base.update(kw)
    return moe_inputs.MoEShape(**base)


def _run(shape, dh_scale=1.0, bias=None):
    from fine_grained_moe_softmax_b300 import MoEConfig, MoELayer
    inputs = moe_inputs.make_inputs(shape)
    if bias is not None:
        inputs["bias"] = bias
    cfg = OracleCfg.from_shape(shape)
    r = oracle.route(cfg, inputs["u"], inputs["centroids"], inputs["bias"])
    if (r["margin"] < NEAR_TIE).any():
        pytest.skip("seeded input has a near-tie token")   # routing would be ambiguous
    g = torch.Generator().manual_seed(shape.seed + 5)
    dh = (torch.randn(shape.T, shape.d, generator=g) * dh_scale).to(torch.bfloat16)
    layer = MoELayer(MoEConfig.from_shape(shape), inputs["centroids"], inputs["w_gate"],
                     inputs["w_up"], inputs["w_down"], inputs["bias"], backward=True)
    u = inputs["u"].to("cuda")
    got = layer.backward(u, dh.to("cuda"))
    torch.cuda.synchronize()
    from fine_grained_moe_softmax_b300 import moe_device_status
    assert moe_device_status(layer.ws_bwd) == 0
    want = oracle.backward(cfg, inputs, dh.to(torch.float64).numpy(), r["counts"])
    return {k: to_np(v) for k, v in got.items()}, want


def _compare(got, want, keys=("du", "d_centroids", "d_bias", "dw_gate", "dw_up", "dw_down")):
    errs = {k: rel_l2(got[k], want[k]) for k in keys}
    bad = {k: v for k, v in errs.items() if not v <= TOL}
    assert not bad, f"rel-L2 above {TOL}: {bad} (all: {errs})"
    return errs


@pytest.mark.parametrize("kw", [
    dict(),
    dict(renormalize=1),
    dict(n_shared=2, top_k=2),
    dict(n_shared=0),
    dict(skip_top=2),
    dict(drop_shared=1),
    dict(T=129, n_routed=32, top_k=6, inter=48, n_groups=8),
    dict(d=256, inter=64, T=300),
    dict(inter=16, T=77, seed=23),          # half-chunk outputs everywhere
    dict(inter=80, n_shared=3, seed=24),    # I % 32 == 16 with several shared experts
    dict(d=384, inter=192, T=150, seed=25),  # 192-column tiles (forward, dgrad, SwiGLU bwd)
    dict(d=256, inter=128, T=48, seed=26),   # <= 64 tokens: 64-row A tiles in the forward GEMMs
])
def test_backward_matches_oracle(kw):
    got, want = _run(_shape(**kw))
    _compare(got, want)


def test_backward_of_balance_losses_alone():
    """dh = 0: only L_ExpBal and L_DevBal drive the gradients (through the affinities), so the
    expert weights get none and u / centroids / bias get the router's share."""
    shape = _shape(alpha1=0.5, alpha2=0.8)
    got, want = _run(shape, dh_scale=0.0)
    for k in ("dw_gate", "dw_up", "dw_down"):
        assert np.all(got[k] == 0)
    _compare(got, want, keys=("du", "d_centroids", "d_bias"))


def test_backward_2b_shape():
    got, want = _run(moe_inputs.CONFIGS["2b_bf16"].with_(T=256))
    _compare(got, want)


def test_backward_zero_tokens():
    from fine_grained_moe_softmax_b300 import MoEConfig, MoELayer
    shape = _shape(T=16)
    inputs = moe_inputs.make_inputs(shape)
    layer = MoELayer(MoEConfig.from_shape(shape), inputs["centroids"], inputs["w_gate"],
                     inputs["w_up"], inputs["w_down"], backward=True)
    g = layer.backward(torch.empty(0, shape.d, dtype=torch.bfloat16, device="cuda"),
                       torch.empty(0, shape.d, dtype=torch.bfloat16, device="cuda"))
    torch.cuda.synchronize()
    for k in ("d_centroids", "d_bias", "dw_gate", "dw_up", "dw_down"):
        assert torch.count_nonzero(g[k]) == 0


def test_backward_full_size_sampled_du():
    """The benchmark's 16B-like shape at its full T = 16384, in the launch configuration
    `bench.py --backward` times: du on a seeded sample of tokens against the oracle.

    du_t depends on the rest of the batch only through the selection counts, which the gradient
    holds fixed, and through 1/T: the balance-loss part of the affinity gradient is
    (a1 f_j + a2 f'_g) / T with f proportional to count / T. So the oracle runs on the sample with
    the full batch's counts twice, with dh and with dh = 0. Its balance part, computed with the
    sample's T_s, is then rescaled by (T_s / T)^2."""
    from fine_grained_moe_softmax_b300 import MoEConfig, MoELayer, moe_device_status
    shape = moe_inputs.CONFIGS["16b_bf16"]
    inputs = moe_inputs.make_inputs(shape)
    T = shape.T
    g = torch.Generator().manual_seed(shape.seed + 5)
    dh = torch.randn(T, shape.d, generator=g).to(torch.bfloat16)
    layer = MoELayer(MoEConfig.from_shape(shape), inputs["centroids"], inputs["w_gate"],
                     inputs["w_up"], inputs["w_down"], inputs["bias"], backward=True)
    got = layer.backward(inputs["u"].to("cuda"), dh.to("cuda"))
    torch.cuda.synchronize()
    assert moe_device_status(layer.ws_bwd) == 0
    du_gpu = to_np(got["du"])
    del got, layer
    torch.cuda.empty_cache()

    cfg = OracleCfg.from_shape(shape)
    r = oracle.route(cfg, inputs["u"], inputs["centroids"], inputs["bias"])
    ok = np.nonzero(r["margin"] >= NEAR_TIE)[0]
    rng = np.random.default_rng(11)
    sample = np.unique(np.concatenate([ok[:2], ok[-2:], rng.choice(ok, 20, replace=False)]))
    Ts = len(sample)
    sub = dict(inputs)
    sub["u"] = inputs["u"][torch.as_tensor(sample)]
    cfg_s = OracleCfg.from_shape(shape, T=Ts)
    dh_s = dh[torch.as_tensor(sample)].to(torch.float64).numpy()
    w1 = oracle.backward(cfg_s, sub, dh_s, r["counts"])
    w0 = oracle.backward(cfg_s, sub, np.zeros_like(dh_s), r["counts"])
    du_want = w1["du"] - (1.0 - (Ts / T) ** 2) * w0["du"]
    err = rel_l2(du_gpu[sample], du_want)
    assert err <= TOL, f"rel-L2(du) on {Ts} sampled tokens = {err}"


@pytest.mark.parametrize("shape", [
    _shape(),
    _shape(n_shared=3, inter=48, T=129, renormalize=1),
    _shape(drop_shared=1, skip_top=1),
    moe_inputs.CONFIGS["2b_bf16"].with_(T=300),
], ids=["base", "3shared_renorm", "ablations", "2b"])
def test_training_pair_matches_forward_and_backward(shape):
    """moe_layer_forward_train + moe_layer_backward_saved run the same kernels on the same rows
    as moe_layer_forward and moe_layer_backward, so h, the routing outputs, the statistics and
    every gradient agree bit for bit; the saved path only skips the recompute."""
    from fine_grained_moe_softmax_b300 import MoEConfig, MoELayer, moe_device_status
    inputs = moe_inputs.make_inputs(shape)
    g = torch.Generator().manual_seed(shape.seed + 5)
    dh = torch.randn(shape.T, shape.d, generator=g).to(torch.bfloat16).to("cuda")
    layer = MoELayer(MoEConfig.from_shape(shape), inputs["centroids"], inputs["w_gate"],
                     inputs["w_up"], inputs["w_down"], inputs["bias"], backward=True)
    u = inputs["u"].to("cuda")
    h_ref = layer.forward(u).clone()
    ref = {k: getattr(layer, k).clone() for k in ("topk_idx", "topk_gate", "counts", "f", "P",
                                                   "losses")}
    g_ref = layer.backward(u, dh)
    torch.cuda.synchronize()
    h = layer.forward_train(u).clone()
    got = {k: getattr(layer, k).clone() for k in ref}
    g_saved = layer.backward_saved(u, dh)
    torch.cuda.synchronize()
    assert moe_device_status(layer.ws_bwd) == 0
    assert torch.equal(h, h_ref)
    for k in ref:
        assert torch.equal(got[k], ref[k]), k
    for k in g_ref:
        assert torch.equal(g_saved[k], g_ref[k]), k


def test_backward_saved_needs_a_training_forward():
    from fine_grained_moe_softmax_b300 import MoEConfig, MoELayer
    shape = _shape(T=32)
    inputs = moe_inputs.make_inputs(shape)
    layer = MoELayer(MoEConfig.from_shape(shape), inputs["centroids"], inputs["w_gate"],
                     inputs["w_up"], inputs["w_down"], backward=True)
    u = inputs["u"].to("cuda")
    with pytest.raises(RuntimeError):
        layer.backward_saved(u, torch.zeros_like(u))
