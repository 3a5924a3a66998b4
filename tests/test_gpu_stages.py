"""GPU parity of each C-ABI stage against the matching oracle stage, and the device-side error
reporting of the stages (corrupt routing input is reported in the status word, never faults)."""
import numpy as np
import pytest
import torch

import moe_inputs
import oracle
from oracle import OracleCfg
from parity import TOL, check_permutation, check_routing, rel_l2, to_np

pytestmark = pytest.mark.gpu

C = moe_inputs.CONFIGS


class Stages:
    """Device buffers for running the layer stage by stage."""

    def __init__(self, shape, T=None):
        import fine_grained_moe_softmax_b300 as moe
        self.moe = moe
        self.shape = shape
        self.inputs = moe_inputs.make_inputs(shape, T=T)
        self.T = self.inputs["u"].shape[0]
        self.cfg = moe.MoEConfig.from_shape(shape, T=self.T)
        self.ocfg = OracleCfg.from_shape(shape, T=self.T)
        dt = self.cfg.torch_dtype()
        dev = "cuda"
        i32, f32 = torch.int32, torch.float32
        T, K, N, d = self.T, shape.top_k, shape.n_routed, shape.d
        self.u = self.inputs["u"].to(dev)
        self.cent = self.inputs["centroids"].to(dev)
        self.bias = None if self.inputs["bias"] is None else self.inputs["bias"].to(dev)
        self.ws = torch.empty(moe.moe_workspace_bytes(self.cfg), dtype=torch.uint8, device=dev)
        self.idx = torch.empty(T, K, dtype=i32, device=dev)
        self.gate = torch.empty(T, K, dtype=f32, device=dev)
        self.counts = torch.empty(N, dtype=i32, device=dev)
        self.psum = torch.empty(N, dtype=f32, device=dev)
        self.offsets = torch.empty(N + 1, dtype=i32, device=dev)
        self.perm_token = torch.empty(T * K, dtype=i32, device=dev)
        self.perm_slot = torch.empty(T * K, dtype=i32, device=dev)
        self.packed = torch.empty(moe.moe_packed_weight_bytes(self.cfg), dtype=torch.uint8,
                                  device=dev)
        self.y_r = torch.empty(T * K, d, dtype=dt, device=dev)
        self.y_s = torch.empty(T, d, dtype=dt, device=dev)
        self.h = torch.empty(T, d, dtype=dt, device=dev)
        self.f = torch.empty(N, dtype=f32, device=dev)
        self.P = torch.empty(N, dtype=f32, device=dev)
        self.losses = torch.empty(2, dtype=f32, device=dev)

    def route(self):
        self.moe.moe_route(self.cfg, self.u, self.cent, self.bias, self.idx, self.gate, self.counts,
                           self.psum, self.ws)

    def permute(self, idx=None, counts=None):
        self.moe.moe_permute(self.cfg, self.idx if idx is None else idx,
                             self.counts if counts is None else counts, self.offsets,
                             self.perm_token, self.perm_slot, self.ws)

    def pack(self):
        dev = "cuda"
        self.moe.moe_pack_weights(self.cfg, self.inputs["w_gate"].to(dev),
                                  self.inputs["w_up"].to(dev), self.inputs["w_down"].to(dev),
                                  self.packed)

    def ffn(self):
        self.moe.moe_expert_ffn(self.cfg, self.u, self.packed, self.offsets, self.perm_token,
                                self.y_r, self.y_s, self.ws)

    def combine(self, perm_slot=None):
        self.moe.moe_combine(self.cfg, self.u, self.y_r, self.y_s,
                             self.perm_slot if perm_slot is None else perm_slot, self.gate, self.h,
                             self.ws)

    def stats(self):
        self.moe.moe_balance_stats(self.cfg, self.counts, self.psum, self.f, self.P, self.losses)

    def status(self):
        return self.moe.moe_device_status(self.ws)


@pytest.mark.parametrize("name,T", [("tiny_f32", None), ("2b_bf16", 400), ("16b_bf16", 300),
                                    ("16b_decode_bf16", None), ("145b_zipf_bf16", 200)])
def test_stage_by_stage(name, T):
    st = Stages(C[name], T)
    sh, cfg = st.shape, st.ocfg
    # router
    st.route()
    ref = oracle.route(cfg, st.inputs["u"], st.inputs["centroids"], st.inputs["bias"])
    torch.cuda.synchronize()
    ok = check_routing(cfg, ref, to_np(st.idx), to_np(st.gate), to_np(st.counts))
    np.testing.assert_allclose(to_np(st.psum), ref["psum"], rtol=2e-4, atol=1e-5)
    assert st.status() == 0
    # permutation: bit-exact against the oracle's counting sort of the GPU's indices
    st.permute()
    torch.cuda.synchronize()
    check_permutation(cfg, to_np(st.idx), to_np(st.offsets), to_np(st.perm_token),
                      to_np(st.perm_slot))
    assert st.status() == 0
    # expert FFNs on a sample of permuted rows, and the shared sum on a sample of tokens
    st.pack()
    st.ffn()
    torch.cuda.synchronize()
    assert st.status() == 0
    rng = np.random.default_rng(3)
    off, pt = to_np(st.offsets), to_np(st.perm_token)
    rows = rng.choice(st.T * sh.top_k, min(48, st.T * sh.top_k), replace=False)
    u64 = to_np(st.u).astype(np.float64)
    want = np.stack([oracle.expert_ffn(cfg, st.inputs, sh.n_shared +
                                       int(np.searchsorted(off, r, side="right") - 1),
                                       u64[pt[r]]) for r in rows])
    tol = TOL[sh.dtype]
    assert rel_l2(to_np(st.y_r)[rows], want) <= tol
    if sh.n_shared:
        toks = rng.choice(st.T, min(24, st.T), replace=False)
        want_s = np.stack([sum(oracle.expert_ffn(cfg, st.inputs, s, u64[t])
                               for s in range(sh.n_shared)) for t in toks])
        assert rel_l2(to_np(st.y_s)[toks], want_s) <= tol
    # combine: h against the oracle's full forward on tokens without a near-tie
    st.combine()
    torch.cuda.synchronize()
    assert st.status() == 0
    toks = np.nonzero(ok)[0][:64]
    fw = oracle.forward_tokens(cfg, st.inputs, toks)
    h = to_np(st.h)[toks]
    assert rel_l2(h, fw["h"]) <= tol
    assert rel_l2(h - u64[toks], fw["h"] - u64[toks]) <= tol
    # statistics from the GPU's counts and psum
    st.stats()
    torch.cuda.synchronize()
    bs = oracle.balance_stats(cfg, to_np(st.counts), to_np(st.psum).astype(np.float64))
    np.testing.assert_allclose(to_np(st.f), bs["f"], rtol=1e-6)
    np.testing.assert_allclose(to_np(st.P), bs["P"], rtol=1e-6, atol=1e-9)
    np.testing.assert_allclose(to_np(st.losses), bs["losses"], rtol=1e-5)


def test_permute_reports_inconsistent_counts():
    st = Stages(C["2b_bf16"], 300)
    st.route()
    bad = st.counts.clone()
    bad[3] += 1
    bad[4] -= 1
    st.permute(counts=bad)
    torch.cuda.synchronize()
    assert st.status() == -6
    # the permutation still follows topk_idx exactly
    check_permutation(st.ocfg, to_np(st.idx), to_np(st.offsets), to_np(st.perm_token),
                      to_np(st.perm_slot))


def test_permute_reports_out_of_range_ids():
    st = Stages(C["2b_bf16"], 300)
    st.route()
    idx = st.idx.clone()
    idx[7, 2] = -1
    idx[250, 0] = st.shape.n_routed
    st.permute(idx=idx)
    torch.cuda.synchronize()
    assert st.status() == -6
    ps = to_np(st.perm_slot).reshape(st.T, -1)
    assert ps[7, 2] == -1 and ps[250, 0] == -1
    off = to_np(st.offsets)
    assert off[-1] == st.T * st.shape.top_k - 2
    # every valid assignment has a row, and rows hold their tokens
    pt = to_np(st.perm_token)
    valid = ps >= 0
    assert sorted(ps[valid].tolist()) == list(range(off[-1]))
    for t, k in zip(*np.nonzero(valid)):
        assert pt[ps[t, k]] == t


def test_combine_reports_bad_rows():
    st = Stages(C["2b_bf16"], 300)
    st.route()
    st.permute()
    st.pack()
    st.ffn()
    bad = st.perm_slot.clone()
    bad[5] = st.T * st.shape.top_k + 100
    bad[6] = -3
    st.combine(perm_slot=bad)
    torch.cuda.synchronize()
    assert st.status() == -6
    st.combine()   # a clean call clears the status word
    torch.cuda.synchronize()
    assert st.status() == 0


@pytest.mark.parametrize("name", ["2b_bf16", "tiny_f32"])
def test_ffn_reports_bad_token_rows(name):
    """Token indices outside [0, T) in perm_token are reported by the gather and never
    dereferenced; every other routed row comes out bit for bit as before."""
    st = Stages(C[name], 300)
    st.route()
    st.permute()
    st.pack()
    st.ffn()
    torch.cuda.synchronize()
    assert st.status() == 0
    ref = st.y_r.clone()
    st.perm_token[11] = st.T + 7
    st.perm_token[12] = -2
    st.ffn()
    torch.cuda.synchronize()
    assert st.status() == -6
    keep = torch.ones(st.y_r.shape[0], dtype=torch.bool, device=st.y_r.device)
    keep[11] = keep[12] = False
    assert torch.equal(st.y_r[keep], ref[keep])


def test_ffn_reports_bad_offsets():
    """Offsets that run past the T*K' routed rows or decrease are cut to the rows that exist and
    reported; a following call with good offsets is clean."""
    st = Stages(C["2b_bf16"], 300)
    st.route()
    st.permute()
    st.pack()
    bad = st.offsets.clone()
    bad[-1] += 500
    bad[5] = bad[6] + 3
    st.moe.moe_expert_ffn(st.cfg, st.u, st.packed, bad, st.perm_token, st.y_r, st.y_s, st.ws)
    torch.cuda.synchronize()
    assert st.status() == -6
    st.ffn()
    torch.cuda.synchronize()
    assert st.status() == 0


def test_stage_errors_raise():
    import fine_grained_moe_softmax_b300 as moe
    st = Stages(C["tiny_f32"], 64)
    small = st.ws[:1024]
    with pytest.raises(moe.MoEError) as e:
        moe.moe_route(st.cfg, st.u, st.cent, None, st.idx, st.gate, st.counts, st.psum, small)
    assert e.value.status == -3


def test_bounded_wait_times_out_and_context_survives():
    """A wait that nothing satisfies gives up, reports MOE_ERR_TIMEOUT, and the next layer call
    on the same context still runs and is correct."""
    import time

    import fine_grained_moe_softmax_b300 as moe
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    t0 = time.perf_counter()
    moe.moe_selftest_bounded_wait(ws, 50_000_000)
    assert moe.moe_device_status(ws) == -5
    assert time.perf_counter() - t0 < 1.5
    st = Stages(C["tiny_f32"], 64)
    st.route()
    torch.cuda.synchronize()
    assert st.status() == 0
    ref = oracle.route(st.ocfg, st.inputs["u"], st.inputs["centroids"])
    check_routing(st.ocfg, ref, to_np(st.idx), to_np(st.gate), to_np(st.counts))


@pytest.mark.parametrize("name,T", [("16b_decode_bf16", 64), ("2b_bf16", 1), ("2b_bf16", 100),
                                    ("2b_bf16", 128), ("145b_zipf_bf16", 77)])
def test_one_tile_layer_equals_the_stages(name, T):
    """A batch of at most 128 tokens has one router tile, and the layer call then takes its
    counts, offsets, permutation and balance statistics from the router itself instead of the
    finalize and scatter kernels. Every output must equal the stage-by-stage calls' bit for bit."""
    st = Stages(C[name], T)
    st.route()
    st.permute()
    st.pack()
    st.ffn()
    st.combine()
    st.stats()
    torch.cuda.synchronize()
    assert st.status() == 0
    layer = st.moe.MoELayer(st.cfg, st.inputs["centroids"], st.inputs["w_gate"],
                            st.inputs["w_up"], st.inputs["w_down"], st.inputs["bias"])
    h = layer.forward(st.u)
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    assert torch.equal(h, st.h)
    assert torch.equal(layer.topk_idx[:T], st.idx) and torch.equal(layer.topk_gate[:T], st.gate)
    assert torch.equal(layer.counts, st.counts)
    for got, want in ((layer.f, st.f), (layer.P, st.P), (layer.losses, st.losses)):
        assert torch.equal(got, want)


@pytest.mark.parametrize("name,T", [("2b_bf16", 300), ("16b_bf16", 1000), ("145b_zipf_bf16", 129)])
def test_split_gate_up_layer_equals_the_stages(name, T):
    """With shared experts and more than one router tile, the layer call runs the shared group's
    gate/up GEMM by itself while the gather runs on a second stream, then the
    routed groups' gate/up. Every output must equal the stage-by-stage calls (one gate/up launch
    over all groups) bit for bit, and the profile must report the split."""
    st = Stages(C[name], T)
    st.route()
    st.permute()
    st.pack()
    st.ffn()
    st.combine()
    st.stats()
    torch.cuda.synchronize()
    assert st.status() == 0
    layer = st.moe.MoELayer(st.cfg, st.inputs["centroids"], st.inputs["w_gate"],
                            st.inputs["w_up"], st.inputs["w_down"], st.inputs["bias"])
    st.moe.moe_profile_enable(True, 4)
    try:
        for _ in range(2):
            h = layer.forward(st.u)
        torch.cuda.synchronize()
        stage_ms, n = st.moe.moe_profile_read()
        gu_ms, n_gu, n_split = st.moe.moe_profile_read_gate_up()
    finally:
        st.moe.moe_profile_enable(False)
    assert layer.device_status() == 0
    assert torch.equal(h, st.h)
    assert torch.equal(layer.topk_idx[:T], st.idx) and torch.equal(layer.topk_gate[:T], st.gate)
    assert torch.equal(layer.counts, st.counts)
    for got, want in ((layer.f, st.f), (layer.P, st.P), (layer.losses, st.losses)):
        assert torch.equal(got, want)
    assert n == n_gu == 2 and n_split == 2
    assert all(v >= 0 for v in stage_ms.values())
    assert 0 < gu_ms <= stage_ms["gemm_gate_up"] + 1e-3


def test_profile_reports_unsplit_gate_up():
    """A one-tile batch (and a layer without shared experts) keeps one gate/up launch."""
    st = Stages(C["16b_decode_bf16"], 64)
    layer = st.moe.MoELayer(st.cfg, st.inputs["centroids"], st.inputs["w_gate"],
                            st.inputs["w_up"], st.inputs["w_down"], st.inputs["bias"])
    st.moe.moe_profile_enable(True, 2)
    try:
        layer.forward(st.u)
        torch.cuda.synchronize()
        stage_ms, n = st.moe.moe_profile_read()
        gu_ms, n_gu, n_split = st.moe.moe_profile_read_gate_up()
    finally:
        st.moe.moe_profile_enable(False)
    assert n == n_gu == 1 and n_split == 0
    assert 0 < gu_ms <= stage_ms["gemm_gate_up"] + 1e-3
