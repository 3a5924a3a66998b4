"""GPU parity of the whole layer (moe_layer_forward through the C ABI) against the fp64 oracle.

Small token counts span several 128-row tiles plus a ragged tail and are checked on every token;
the full-size workloads are checked on all routing decisions and on a seeded sample of h rows.
"""
import numpy as np
import pytest
import torch

import moe_inputs
import oracle
from oracle import OracleCfg
from parity import (NEAR_TIE, TOL, TOL_TOKEN, check_permutation, check_routing,
                    per_token_rel_l2, rel_l2, run_layer, to_np)

pytestmark = pytest.mark.gpu

C = moe_inputs.CONFIGS


def _compare_layer(shape, inputs, layer, u_dev, tokens=None):
    T = inputs["u"].shape[0]
    cfg = OracleCfg.from_shape(shape, T=T)
    ref_route = oracle.route(cfg, inputs["u"], inputs["centroids"], inputs.get("bias"))
    idx = to_np(layer.topk_idx[:T])
    gate = to_np(layer.topk_gate[:T])
    counts = to_np(layer.counts)
    ok = check_routing(cfg, ref_route, idx, gate, counts)
    # the layer's own dispatch permutation: bit for bit the oracle's counting sort of the GPU's
    # indices; its affinity sums against the oracle's
    tabs = layer.routing(T)
    check_permutation(cfg, idx, to_np(tabs["offsets"]), to_np(tabs["perm_token"]),
                      to_np(tabs["perm_slot"]))
    np.testing.assert_allclose(to_np(tabs["psum"]), ref_route["psum"], rtol=2e-4, atol=1e-5)
    # statistics: the oracle's balance statistics of the GPU's own counts and the oracle's psum
    st = oracle.balance_stats(cfg, counts, ref_route["psum"])
    np.testing.assert_allclose(to_np(layer.f), st["f"], rtol=1e-6)
    np.testing.assert_allclose(to_np(layer.P), st["P"], rtol=2e-4, atol=1e-7)
    np.testing.assert_allclose(to_np(layer.losses), st["losses"], rtol=2e-4)
    # h on the chosen tokens that are not near-ties
    toks = np.arange(T) if tokens is None else np.asarray(tokens)
    toks = toks[ok[toks]]
    fw = oracle.forward_tokens(cfg, inputs, toks)
    h = to_np(layer.h[:T])[toks]
    u = to_np(u_dev)[toks]
    tol = TOL[shape.dtype]
    err_h = rel_l2(h, fw["h"])
    err_moe = rel_l2(h - u, fw["h"] - u)
    assert err_h <= tol, f"rel-L2(h) = {err_h}"
    assert err_moe <= tol, f"rel-L2(h - u) = {err_moe}"
    tok_h = per_token_rel_l2(h, fw["h"])
    tok_moe = per_token_rel_l2(h - u, fw["h"] - u)
    worst = int(np.argmax(tok_moe))
    assert tok_h.max() <= TOL_TOKEN[shape.dtype], f"per-token rel-L2(h) = {tok_h.max()}"
    assert tok_moe.max() <= TOL_TOKEN[shape.dtype], \
        f"per-token rel-L2(h - u) = {tok_moe.max()} at token {toks[worst]}"
    assert layer.device_status() == 0
    return err_h, err_moe


@pytest.mark.parametrize("name,T", [("tiny_f32", None), ("tiny_f32", 129), ("2b_bf16", 300),
                                    ("16b_bf16", 257), ("16b_decode_bf16", None),
                                    ("145b_zipf_bf16", 130), ("2b_half_activated_bf16", 300),
                                    ("2b_gshard_top2_bf16", 300)])
def test_layer_all_tokens(name, T):
    shape = C[name]
    inputs = moe_inputs.make_inputs(shape, T=T)
    layer, u = run_layer(shape, inputs, T=inputs["u"].shape[0])
    _compare_layer(shape, inputs, layer, u)


@pytest.mark.parametrize("name", ["2b_bf16", "16b_bf16", "145b_zipf_bf16",
                                  "2b_gshard_top2_bf16"])
def test_layer_full_size_sampled(name):
    """Full token count in the launch configuration the benchmark times; every routing decision
    is compared, h on a seeded sample of tokens (including the first and last tile)."""
    shape = C[name]
    inputs = moe_inputs.make_inputs(shape)
    layer, u = run_layer(shape, inputs)
    rng = np.random.default_rng(7)
    T = shape.T
    sample = np.unique(np.concatenate([[0, 1, 127, 128, T - 1],
                                       rng.choice(T, 40, replace=False)]))
    _compare_layer(shape, inputs, layer, u, tokens=sample)


def _custom(**kw):
    base = dict(name="custom", T=200, d=128, n_shared=1, n_routed=16, inter=32, top_k=4,
                n_groups=4, dtype="bf16", seed=11)
    base.update(kw)
    return moe_inputs.MoEShape(**base)


@pytest.mark.parametrize("kw", [
    dict(),                                         # baseline small bf16
    dict(renormalize=1),                            # renormalised gates
    dict(n_shared=0),                               # no shared experts (coarse top-k special case)
    dict(n_shared=3, inter=48),                     # several shared experts, I not a multiple of 64
    dict(top_k=16, n_routed=16),                    # K' = N': dense softmax mixture
    dict(top_k=1),                                  # top-1
    dict(T=1), dict(T=127), dict(T=128), dict(T=129),
    dict(d=64, inter=16),                           # smallest supported widths
    dict(d=384, inter=192, T=300),                  # 192-column tiles in both GEMMs
    dict(d=128, inter=320, T=200),                  # 160-column gate/up tiles
    dict(d=256, inter=128, T=40),                   # <= 64 tokens: 64-row A tiles, 5 stages
    dict(n_routed=256, top_k=8, n_groups=8, T=300), # widest router
    # the placing gather in its one-CTA-per-token form (129 .. 296 tokens), 5 <= K' <= 8
    dict(n_routed=64, top_k=6, n_groups=8, d=512, inter=64, T=250),
    # router column slices with ragged ends (n_pad 224, 128, 64 over 200, 100, 40 experts), stages
    # of 2, 3 and 4 K chunks with a shorter last stage, one-tile and cluster-split tiles
    dict(n_routed=200, top_k=8, n_groups=8, d=640, T=300),
    dict(n_routed=100, top_k=5, n_groups=4, d=512, T=64),
    dict(n_routed=40, top_k=6, n_groups=5, d=1152, T=64, renormalize=1),
    dict(n_routed=40, top_k=6, n_groups=5, d=1152, T=700),
    # 75 MB of shared gate/up weights: column panels of the shared group, the last one narrower
    dict(d=2048, n_shared=9, inter=1024, T=300),
    dict(dtype="f32", renormalize=1, n_shared=2),
    dict(dtype="f32", top_k=16, n_routed=16, T=77),
    # ablations of the expert-specialisation analysis: disabled top experts / shared experts
    dict(skip_top=1), dict(skip_top=3, top_k=2, renormalize=1), dict(skip_top=6, top_k=10),
    dict(drop_shared=1), dict(drop_shared=1, n_shared=3, skip_top=2),
    dict(dtype="f32", skip_top=2, drop_shared=1),
])
def test_layer_edge_shapes(kw):
    shape = _custom(**kw)
    inputs = moe_inputs.make_inputs(shape)
    layer, u = run_layer(shape, inputs)
    _compare_layer(shape, inputs, layer, u)


def test_all_tokens_to_one_expert():
    """A large logit bias sends every token to experts 5 and 9: those two routed groups hold all
    T rows each (several row tiles), the others none. The biases keep the affinity gaps between
    ranks 1, 2 and 3 well above the near-tie threshold."""
    shape = _custom(T=300, top_k=2)
    inputs = moe_inputs.make_inputs(shape)
    bias = torch.zeros(shape.n_routed)
    bias[5] = 16.0
    bias[9] = 8.0
    inputs["bias"] = bias
    layer, u = run_layer(shape, inputs)
    counts = to_np(layer.counts)
    assert counts[5] == shape.T and counts[9] == shape.T and counts.sum() == 2 * shape.T
    _compare_layer(shape, inputs, layer, u)


def test_zero_tokens():
    shape = _custom(T=16)
    inputs = moe_inputs.make_inputs(shape)
    from fine_grained_moe_softmax_b300 import MoEConfig, MoELayer
    layer = MoELayer(MoEConfig.from_shape(shape), inputs["centroids"], inputs["w_gate"],
                     inputs["w_up"], inputs["w_down"])
    layer.counts.fill_(7)
    layer.losses.fill_(7)
    layer.forward(torch.empty(0, shape.d, dtype=torch.bfloat16, device="cuda"))
    torch.cuda.synchronize()
    assert to_np(layer.counts).sum() == 0
    assert np.all(to_np(layer.losses) == 0)
    assert layer.device_status() == 0


def test_deterministic():
    shape = C["2b_bf16"]
    inputs = moe_inputs.make_inputs(shape, T=1000)
    layer, u = run_layer(shape, inputs, T=1000)
    h1 = layer.h.clone()
    p1 = layer.P.clone()
    layer.forward(u)
    torch.cuda.synchronize()
    assert torch.equal(h1, layer.h)
    assert torch.equal(p1, layer.P)


def test_near_tie_threshold_is_rare():
    """The exclusion rule only removes a handful of tokens at the largest workload."""
    shape = C["16b_bf16"]
    cfg = OracleCfg.from_shape(shape, T=4096)
    inputs = moe_inputs.make_inputs(shape, T=4096)
    r = oracle.route(cfg, inputs["u"], inputs["centroids"])
    assert (r["margin"] < NEAR_TIE).sum() <= 8


@pytest.mark.parametrize("name,T", [("2b_bf16", 300), ("16b_decode_bf16", 64),
                                    ("145b_zipf_bf16", 1000)])
def test_graph_replay_matches_direct_calls(name, T):
    """The layer call captures into a CUDA graph; replays on new contents of the captured input
    buffer give the same bytes as direct calls: the multi-tile path with the side-stream gather,
    the one-tile decode path whose router builds the routing tables, and the 145B-like layer."""
    shape = C[name]
    inputs = moe_inputs.make_inputs(shape, T=T)
    layer, u = run_layer(shape, inputs, T=T)
    graph, kernels = layer.capture(u)
    assert kernels >= 5
    u2 = moe_inputs.make_tokens(shape, T=T, seed=99).to("cuda")
    u.copy_(u2)
    graph.replay()
    torch.cuda.synchronize()
    h_graph, idx_graph, P_graph = layer.h.clone(), layer.topk_idx.clone(), layer.P.clone()
    gate_graph, loss_graph = layer.topk_gate.clone(), layer.losses.clone()
    tabs_graph = {k: v.clone() for k, v in layer.routing(T).items()}
    assert layer.device_status() == 0
    layer.forward(u2)
    torch.cuda.synchronize()
    assert torch.equal(h_graph, layer.h)
    assert torch.equal(idx_graph, layer.topk_idx)
    assert torch.equal(gate_graph, layer.topk_gate)
    assert torch.equal(P_graph, layer.P)
    assert torch.equal(loss_graph, layer.losses)
    for k, v in layer.routing(T).items():
        assert torch.equal(tabs_graph[k], v), k
    assert layer.device_status() == 0
    # and the replayed routing is the oracle's
    cfg = OracleCfg.from_shape(shape, T=T)
    ref = oracle.route(cfg, u2.cpu(), inputs["centroids"], inputs.get("bias"))
    check_routing(cfg, ref, to_np(idx_graph[:T]), to_np(gate_graph[:T]), to_np(layer.counts))


def test_layer_four_times_benchmark_tokens():
    """The 16B-like layer at T = 65536 (4x the benchmark batch, about 5 GB of workspace): all
    routing decisions, counts and statistics, and h on a sample that includes the last tile."""
    shape = C["16b_bf16"]
    T = 65536
    inputs = moe_inputs.make_inputs(shape, T=T)
    layer, u = run_layer(shape, inputs, T=T)
    rng = np.random.default_rng(11)
    sample = np.unique(np.concatenate([[0, T - 129, T - 1], rng.choice(T, 30, replace=False)]))
    _compare_layer(shape, inputs, layer, u, tokens=sample)


def test_routing_does_not_depend_on_the_batch_it_sits_in():
    """A batch of one router tile splits the logits' K loop over a cluster of CTAs and adds the
    partial sums in rank order; a large batch computes each tile in one CTA. The logits can then
    differ in the last bits, but the routing of every token without a near-tie must be the same in
    both, and the gates agree to the router's tolerance."""
    shape = C["16b_bf16"]
    big = moe_inputs.make_tokens(shape, T=16384, seed=5)
    small = big[:64].clone()
    inputs = moe_inputs.make_inputs(shape, T=64)
    outs = {}
    for name, u in (("small", small), ("big", big)):
        inp = dict(inputs)
        inp["u"] = u
        layer, _ = run_layer(shape, inp, T=u.shape[0])
        outs[name] = (to_np(layer.topk_idx[:64]), to_np(layer.topk_gate[:64]))
        assert layer.device_status() == 0
        del layer
    cfg = OracleCfg.from_shape(shape, T=64)
    ref = oracle.route(cfg, small, inputs["centroids"])
    ok = ref["margin"] >= NEAR_TIE
    assert np.array_equal(outs["small"][0][ok], outs["big"][0][ok])
    assert np.abs(outs["small"][1][ok] - outs["big"][1][ok]).max() <= 2e-5
