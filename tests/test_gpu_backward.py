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


def _run(shape, dh_scale=1.0, bias=None, tie=None):
    """GPU and oracle gradients of the same objective. A near-tie token (R9: its selection is
    decided by rounding, so the two sides may pick different experts) gets dh_t = 0: every term
    that depends on its selection is multiplied by dh_t, and the rest of its gradient (through
    the balance losses) depends only on the counts, which the oracle takes from the GPU. Those
    tokens stay in the batch and in the comparison."""
    from fine_grained_moe_softmax_b300 import MoEConfig, MoELayer
    inputs = moe_inputs.make_inputs(shape)
    if bias is not None:
        inputs["bias"] = bias
    if tie is not None:   # expert tie[1] gets expert tie[0]'s centroid: exact ties
        inputs["centroids"][tie[1]] = inputs["centroids"][tie[0]]
    cfg = OracleCfg.from_shape(shape)
    r = oracle.route(cfg, inputs["u"], inputs["centroids"], inputs["bias"])
    near = r["margin"] < NEAR_TIE
    g = torch.Generator().manual_seed(shape.seed + 5)
    dh = (torch.randn(shape.T, shape.d, generator=g) * dh_scale).to(torch.bfloat16)
    dh[torch.from_numpy(near)] = 0
    layer = MoELayer(MoEConfig.from_shape(shape), inputs["centroids"], inputs["w_gate"],
                     inputs["w_up"], inputs["w_down"], inputs["bias"], backward=True)
    u = inputs["u"].to("cuda")
    # the GPU's selection counts (the backward recomputes the same router)
    layer.forward(u)
    torch.cuda.synchronize()
    counts = to_np(layer.counts).astype(np.int64)
    idx = to_np(layer.topk_idx)
    assert np.array_equal(idx[~near], r["topk_idx"][~near])
    got = layer.backward(u, dh.to("cuda"))
    torch.cuda.synchronize()
    from fine_grained_moe_softmax_b300 import moe_device_status
    assert moe_device_status(layer.ws_bwd) == 0
    want = oracle.backward(cfg, inputs, dh.to(torch.float64).numpy(), counts)
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


def test_backward_with_near_tie_tokens():
    """Experts 3 and 7 share a centroid, so every token that ranks them among its top K'+1 has an
    exact tie: the near-tie rule zeroes those tokens' dh, they stay in the batch, and the
    gradients still match the oracle's."""
    shape = _shape(T=200, top_k=2, seed=27)
    inputs = moe_inputs.make_inputs(shape)
    inputs["centroids"][7] = inputs["centroids"][3]
    r = oracle.route(OracleCfg.from_shape(shape), inputs["u"], inputs["centroids"])
    n_near = int((r["margin"] < NEAR_TIE).sum())
    assert 5 <= n_near <= shape.T // 2
    got, want = _run(shape, tie=(3, 7))
    _compare(got, want)
